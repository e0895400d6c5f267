// importance.cu -- cumulative attention-importance score, four-tier classification and
// 8-bit storage of the T2 rows.
//
// "Nem Todos os Pensamentos Necessitam de HBM" (gist.science summary):
//   Metodologia 2 -- s_i(t) = s_i(t-1) + (1/|L|) sum_l (1/H) sum_h alpha_{l,h}(t)[i];
//   Metodologia 1 -- tiers T0 (HBM: protected + most important), T1 (DDR), T2 (8-bit),
//                    T3 (evicted tail);
//   Metodologia 4 -- re-tiering every Delta = 64 decode steps (the caller's schedule).
#include <algorithm>

#include "sd_common.cuh"
#include "sd_host.h"

namespace sd {
namespace {

// ------------------------------------------------------------------ score accumulate

// Dense selection (every position is a list row): thread -> 4 consecutive positions of one
// sequence (16-byte loads along T).  The rows' lse values are staged in shared memory, the
// logits of kRowBatch rows are all loaded before any is used, the rows are summed in a
// fixed order, and the fp64 running score takes one add per position.
constexpr int kAccThreads = 128;
constexpr int kRowBatch = 16;

__global__ void __launch_bounds__(kAccThreads)
    score_accumulate_dense_kernel(const float* __restrict__ logits, const float* __restrict__ lse, int rows, int T,
                                  double weight, double* __restrict__ s) {
    extern __shared__ float lse_s[];  // [rows]
    pdl_wait();
    const int b = blockIdx.y;
    const size_t q0 = (size_t)b * rows;
    for (int r = threadIdx.x; r < rows; r += kAccThreads) lse_s[r] = lse[q0 + r];
    __syncthreads();
    const int i = (blockIdx.x * kAccThreads + threadIdx.x) * 4;
    if (i >= T) return;
    const float* lrow = logits + q0 * T + i;
    float4 acc = make_float4(0.f, 0.f, 0.f, 0.f);
    for (int r0 = 0; r0 < rows; r0 += kRowBatch) {
        float4 z[kRowBatch];
#pragma unroll
        for (int u = 0; u < kRowBatch; ++u)
            z[u] = r0 + u < rows ? __ldcs(reinterpret_cast<const float4*>(lrow + (size_t)(r0 + u) * T))
                                 : make_float4(0.f, 0.f, 0.f, 0.f);
#pragma unroll
        for (int u = 0; u < kRowBatch; ++u) {
            if (r0 + u < rows) {
                const float m = lse_s[r0 + u];
                acc.x += expf(z[u].x - m);
                acc.y += expf(z[u].y - m);
                acc.z += expf(z[u].z - m);
                acc.w += expf(z[u].w - m);
            }
        }
    }
    double* srow = s + (size_t)b * T + i;
    srow[0] += weight * (double)acc.x;
    srow[1] += weight * (double)acc.y;
    srow[2] += weight * (double)acc.z;
    srow[3] += weight * (double)acc.w;
}

// Dense selection with T not a multiple of 4 (or unaligned logits): thread per position.
__global__ void __launch_bounds__(kAccThreads)
    score_accumulate_dense_scalar_kernel(const float* __restrict__ logits, const float* __restrict__ lse, int rows,
                                         int T, double weight, double* __restrict__ s) {
    extern __shared__ float lse_s[];  // [rows]
    pdl_wait();
    const int b = blockIdx.y;
    const size_t q0 = (size_t)b * rows;
    for (int r = threadIdx.x; r < rows; r += kAccThreads) lse_s[r] = lse[q0 + r];
    __syncthreads();
    const int i = blockIdx.x * kAccThreads + threadIdx.x;
    if (i >= T) return;
    float acc = 0.f;
    for (int r0 = 0; r0 < rows; r0 += kRowBatch) {
        float z[kRowBatch];
#pragma unroll
        for (int u = 0; u < kRowBatch; ++u) z[u] = r0 + u < rows ? __ldcs(logits + (q0 + r0 + u) * T + i) : 0.f;
#pragma unroll
        for (int u = 0; u < kRowBatch; ++u)
            if (r0 + u < rows) acc += expf(z[u] - lse_s[r0 + u]);
    }
    s[(size_t)b * T + i] += weight * (double)acc;
}

// Sparse selection: one thread per (b, kvh, selected row); several KV groups may select
// the same position, so the add is an fp64 atomic.
__global__ void score_accumulate_sparse_kernel(const float* __restrict__ logits,
                                               const float* __restrict__ lse,
                                               const int32_t* __restrict__ idx, int B, int V, int Hq,
                                               int Hkv, int n_idx, int block, int T, double weight,
                                               double* __restrict__ s, int32_t* err) {
    const int G = Hq / Hkv;
    const long n_rows = (long)n_idx * block;
    const long n = (long)B * Hkv * n_rows;
    for (long e = blockIdx.x * (long)blockDim.x + threadIdx.x; e < n; e += (long)gridDim.x * blockDim.x) {
        const long j = e % n_rows;
        const long bk = e / n_rows;
        const int b = (int)(bk / Hkv), kvh = (int)(bk % Hkv);
        const long sel = idx[bk * n_idx + j / block];
        if (sel == -1) continue;  // empty slot
        const long pos = sel * block + j % block;
        if (sel < 0 || pos >= T) {
            report(err, SD_DEVERR_INDEX);
            continue;
        }
        float acc = 0.f;
        for (int v = 0; v < V; ++v)
            for (int g = 0; g < G; ++g) {
                const size_t qrow = ((size_t)b * V + v) * Hq + kvh * G + g;
                acc += expf(logits[qrow * n_rows + j] - lse[qrow]);
            }
        atomicAdd(&s[(size_t)b * T + pos], weight * (double)acc);
    }
}

// ------------------------------------------------------------------ tier classify

constexpr int kTcThreads = 1024;
constexpr int kTcWarps = kTcThreads / 32;

SD_DEVINL uint32_t block_scan_incl(uint32_t v, uint32_t* wsum) {
    const int lane = threadIdx.x & 31, warp = threadIdx.x >> 5;
#pragma unroll
    for (int o = 1; o < 32; o <<= 1) {
        const uint32_t n = __shfl_up_sync(0xffffffffu, v, o);
        if (lane >= o) v += n;
    }
    if (lane == 31) wsum[warp] = v;
    __syncthreads();
    if (warp == 0) {
        uint32_t w = wsum[lane];
#pragma unroll
        for (int o = 1; o < 32; o <<= 1) {
            const uint32_t n = __shfl_up_sync(0xffffffffu, w, o);
            if (lane >= o) w += n;
        }
        wsum[lane] = w;
    }
    __syncthreads();
    const uint32_t off = warp > 0 ? wsum[warp - 1] : 0u;
    __syncthreads();
    return v + off;
}

struct TierShared {
    uint32_t hist[256];
    uint32_t wsum[32];
    uint32_t sel_digit, sel_above;
    uint32_t cnt_gt[3][kTcWarps], cnt_eq[3][kTcWarps], eq_before[3][kTcWarps];
    uint32_t counts[4];
};

// k-th largest 64-bit key among the unprotected positions of row `srow`: returns the key
// and how many entries equal to it belong to the top k (8 passes of 8-bit digits).
SD_DEVINL void select_kth_u64(const double* srow, int T, int n_sink, int n_recent, int k,
                              TierShared& sh, uint64_t& thr, int& krem) {
    const int tid = threadIdx.x, lane = tid & 31, warp = tid >> 5;
    uint64_t prefix = 0, pmask = 0;
    krem = k;
#pragma unroll 1
    for (int pass = 0; pass < 8; ++pass) {
        const int shift = 56 - 8 * pass;
        for (int b = tid; b < 256; b += kTcThreads) sh.hist[b] = 0;
        __syncthreads();
        for (int base = warp * 32; base < T; base += kTcThreads) {
            const int i = base + lane;
            const bool valid = i < T && i >= n_sink && i < T - n_recent;
            const uint64_t kk = valid ? double_key(srow[i]) : 0ull;
            const bool in = valid && (kk & pmask) == prefix;
            const uint32_t dg = (uint32_t)(kk >> shift) & 255u;
            const uint32_t peers = __match_any_sync(0xffffffffu, in ? dg : 0xffffffffu);
            if (in && lane == __ffs(peers) - 1) atomicAdd(&sh.hist[dg], (uint32_t)__popc(peers));
        }
        __syncthreads();
        // thread t < 256 owns bin 255 - t
        const uint32_t local = tid < 256 ? sh.hist[255 - tid] : 0u;
        const uint32_t incl = block_scan_incl(local, sh.wsum);
        const uint32_t excl = incl - local;
        if (tid < 256 && excl < (uint32_t)krem && (uint32_t)krem <= incl) {
            sh.sel_digit = 255u - (uint32_t)tid;
            sh.sel_above = excl;
        }
        __syncthreads();
        prefix |= (uint64_t)sh.sel_digit << shift;
        pmask |= 255ull << shift;
        krem -= (int)sh.sel_above;
        __syncthreads();
    }
    thr = prefix;
}

__global__ void __launch_bounds__(kTcThreads, 1)
    tier_classify_kernel(const double* __restrict__ s, int T, long c0, long c1, long c2, int n_sink,
                         int n_recent, uint8_t* __restrict__ tier, int32_t* __restrict__ counts) {
    __shared__ TierShared sh;
    const int tid = threadIdx.x, lane = tid & 31, warp = tid >> 5;
    const int b = blockIdx.x;
    const double* srow = s + (size_t)b * T;
    uint8_t* trow = tier + (size_t)b * T;
    // protected positions: [0, n_sink) and [T - n_recent, T)
    const int lo = min(n_sink, T), hi = max(lo, T - n_recent);
    const long n_prot = (long)lo + (T - hi);
    const long n_free = (long)hi - lo;
    const long cm[3] = {c0, c1, c2};
    uint64_t thr[3];
    int krem[3];
    int mode[3];  // 0: none of the free positions, 1: all, 2: threshold
    for (int m = 0; m < 3; ++m) {
        long km = cm[m] - n_prot;
        km = km < 0 ? 0 : (km > n_free ? n_free : km);
        if (km == 0) {
            mode[m] = 0;
        } else if (km == n_free) {
            mode[m] = 1;
        } else {
            mode[m] = 2;
            select_kth_u64(srow, T, lo, T - hi, (int)km, sh, thr[m], krem[m]);
        }
        if (mode[m] != 2) {
            thr[m] = 0;
            krem[m] = 0;
        }
    }
    if (tid < 4) sh.counts[tid] = 0;
    // ordered pass: warp w owns [w*seg, (w+1)*seg)
    const int seg = ((T + kTcWarps - 1) / kTcWarps + 31) / 32 * 32;
    const int s0 = warp * seg, s1 = min(T, s0 + seg);
    uint32_t gt[3] = {0, 0, 0}, eq[3] = {0, 0, 0};
    for (int base = s0; base < s1; base += 32) {
        const int i = base + lane;
        const bool valid = i < s1 && i >= lo && i < hi;
        const uint64_t kk = valid ? double_key(srow[i]) : 0ull;
#pragma unroll
        for (int m = 0; m < 3; ++m) {
            gt[m] += __popc(__ballot_sync(0xffffffffu, valid && kk > thr[m]));
            eq[m] += __popc(__ballot_sync(0xffffffffu, valid && kk == thr[m]));
        }
    }
    if (lane == 0)
        for (int m = 0; m < 3; ++m) {
            sh.cnt_gt[m][warp] = gt[m];
            sh.cnt_eq[m][warp] = eq[m];
        }
    __syncthreads();
    if (tid < 3) {
        uint32_t eqb = 0;
        for (int w = 0; w < kTcWarps; ++w) {
            sh.eq_before[tid][w] = eqb;
            eqb += sh.cnt_eq[tid][w];
        }
    }
    __syncthreads();
    uint32_t eq_seen[3] = {sh.eq_before[0][warp], sh.eq_before[1][warp], sh.eq_before[2][warp]};
    uint32_t local_counts[4] = {0, 0, 0, 0};
    const uint32_t lt = lanemask_lt();
    for (int base = s0; base < s1; base += 32) {
        const int i = base + lane;
        const bool in_row = i < s1;
        const bool free_pos = in_row && i >= lo && i < hi;
        const uint64_t kk = free_pos ? double_key(srow[i]) : 0ull;
        bool in_top[3];
#pragma unroll
        for (int m = 0; m < 3; ++m) {
            const bool is_eq = free_pos && kk == thr[m];
            const uint32_t eqm = __ballot_sync(0xffffffffu, is_eq);
            if (mode[m] == 0)
                in_top[m] = false;
            else if (mode[m] == 1)
                in_top[m] = true;
            else
                in_top[m] = kk > thr[m] || (is_eq && (int)(eq_seen[m] + __popc(eqm & lt)) < krem[m]);
            eq_seen[m] += __popc(eqm);
        }
        if (in_row) {
            const int t = !free_pos ? 0 : in_top[0] ? 0 : in_top[1] ? 1 : in_top[2] ? 2 : 3;
            trow[i] = (uint8_t)t;
            local_counts[t]++;
        }
    }
    for (int t = 0; t < 4; ++t) {
        uint32_t c = local_counts[t];
#pragma unroll
        for (int o = 16; o > 0; o >>= 1) c += __shfl_xor_sync(0xffffffffu, c, o);
        if (lane == 0 && c) atomicAdd(&sh.counts[t], c);
    }
    __syncthreads();
    if (tid < 4) counts[(size_t)b * 4 + tid] = (int32_t)sh.counts[tid];
}

// ------------------------------------------------------------------ int8 rows

// One warp per row (b, h, t); only rows whose tier is 2 are written.
template <typename ST, int D>
__global__ void quantize_rows_kernel(const ST* __restrict__ x, const uint8_t* __restrict__ tier,
                                     int B, int Hkv, int T, int8_t* __restrict__ codes,
                                     float* __restrict__ scales) {
    constexpr int EPL = D / 32;
    const long rows = (long)B * Hkv * T;
    const int lane = threadIdx.x & 31;
    const long warp0 = (blockIdx.x * (long)blockDim.x + threadIdx.x) >> 5;
    const long nwarps = ((long)gridDim.x * blockDim.x) >> 5;
    for (long row = warp0; row < rows; row += nwarps) {
        const int t = (int)(row % T);
        const long b = row / ((long)Hkv * T);
        if (tier[b * T + t] != 2) continue;
        float v[EPL];
        const ST* xr = x + row * D + lane * EPL;
        if constexpr (sizeof(ST) == 2) {
            const uint16_t* u = reinterpret_cast<const uint16_t*>(xr);
#pragma unroll
            for (int e = 0; e < EPL; ++e) v[e] = __uint_as_float((uint32_t)u[e] << 16);
        } else {
#pragma unroll
            for (int e = 0; e < EPL; ++e) v[e] = reinterpret_cast<const float*>(xr)[e];
        }
        float a = 0.f;
#pragma unroll
        for (int e = 0; e < EPL; ++e) a = fmaxf(a, fabsf(v[e]));
        a = warp_max(a);
        int8_t* cr = codes + row * D + lane * EPL;
        if (a == 0.f) {
#pragma unroll
            for (int e = 0; e < EPL; ++e) cr[e] = 0;
            if (lane == 0) scales[row] = 0.f;
            continue;
        }
        const float inv = __fdiv_rn(127.f, a);
#pragma unroll
        for (int e = 0; e < EPL; ++e) {
            int c = __float2int_rn(__fmul_rn(v[e], inv));
            cr[e] = (int8_t)max(-127, min(127, c));
        }
        if (lane == 0) scales[row] = __fdiv_rn(a, 127.f);
    }
}

}  // namespace
}  // namespace sd

using namespace sd;

extern "C" sd_status sd_score_accumulate(const float* logits, const float* lse, const int32_t* idx,
                                         int B, int V, int Hq, int Hkv, int n_idx, int block, int T,
                                         double weight, double* s, int32_t* err_word, void* stream) {
    clear_error();
    SD_REQUIRE(B >= 0 && V >= 1 && Hq >= 1 && Hkv >= 1 && T >= 0 && n_idx >= 0 && block >= 1,
               "sd_score_accumulate: bad sizes");
    SD_REQUIRE(Hq % Hkv == 0, "sd_score_accumulate: Hq must be a multiple of Hkv");
    if (idx == nullptr && n_idx > 0)
        SD_REQUIRE((long)n_idx * block == T, "sd_score_accumulate: dense mode needs n_idx*block == T");
    const long n_rows = (long)n_idx * block;
    if (B == 0 || n_rows == 0) return SD_OK;
    SD_REQUIRE(logits && lse && s, "sd_score_accumulate: null pointer");
    cudaStream_t st = as_stream(stream);
    const int threads = 256;
    if (idx == nullptr) {
        SD_REQUIRE(B <= 65535, "sd_score_accumulate: B must be <= 65535");
        const int rows = V * Hq;
        SD_REQUIRE(rows <= 12288, "sd_score_accumulate: V*Hq must be <= 12288");
        const size_t smem = (size_t)rows * sizeof(float);
        const bool vec = T % 4 == 0 && aligned16(logits);
        auto kern = vec ? score_accumulate_dense_kernel : score_accumulate_dense_scalar_kernel;
        const int per_cta = vec ? 4 * kAccThreads : kAccThreads;
        const dim3 grid((unsigned)((T + per_cta - 1) / per_cta), (unsigned)B);
        SD_CUDA_CHECK(launch_pdl(kern, grid, dim3(kAccThreads), smem, st, logits, lse, rows, T, weight, s),
                      "sd_score_accumulate: launch");
    } else {
        const long n = (long)B * Hkv * n_rows;
        const long blocks = std::min<long>((n + threads - 1) / threads, (long)num_sms() * 16);
        score_accumulate_sparse_kernel<<<(unsigned)blocks, threads, 0, st>>>(
            logits, lse, idx, B, V, Hq, Hkv, n_idx, block, T, weight, s, err_word);
    }
    return launch_status("sd_score_accumulate");
}

extern "C" size_t sd_tier_classify_workspace_bytes(int B, int T) {
    (void)B;
    (void)T;
    return 0;
}

extern "C" sd_status sd_tier_classify(const double* s, int B, int T, const double cum_frac[3],
                                      int n_sink, int n_recent, uint8_t* tier, int32_t* counts,
                                      void* workspace, size_t workspace_bytes, void* stream) {
    (void)workspace;
    (void)workspace_bytes;
    clear_error();
    SD_REQUIRE(B >= 0 && T >= 0 && n_sink >= 0 && n_recent >= 0, "sd_tier_classify: bad sizes");
    SD_REQUIRE(cum_frac != nullptr, "sd_tier_classify: null cum_frac");
    for (int m = 0; m < 3; ++m) {
        SD_REQUIRE(cum_frac[m] >= 0.0 && cum_frac[m] <= 1.0, "sd_tier_classify: cum_frac outside [0,1]");
        if (m > 0) SD_REQUIRE(cum_frac[m] >= cum_frac[m - 1], "sd_tier_classify: cum_frac must be nondecreasing");
    }
    if (B == 0) return SD_OK;
    SD_REQUIRE(tier && counts && (T == 0 || s), "sd_tier_classify: null pointer");
    SD_REQUIRE(B <= 65535, "sd_tier_classify: B must be <= 65535");
    long c[3];
    for (int m = 0; m < 3; ++m) c[m] = (long)floor(cum_frac[m] * (double)T);
    tier_classify_kernel<<<B, kTcThreads, 0, as_stream(stream)>>>(s, T, c[0], c[1], c[2], n_sink,
                                                                 n_recent, tier, counts);
    return launch_status("sd_tier_classify");
}

extern "C" sd_status sd_quantize_rows_int8(const void* x, sd_dtype dtype, const uint8_t* tier,
                                           int B, int Hkv, int T, int d, int8_t* codes,
                                           float* scales, void* stream) {
    clear_error();
    SD_REQUIRE(B >= 0 && Hkv >= 0 && T >= 0, "sd_quantize_rows_int8: bad sizes");
    SD_REQUIRE(valid_dtype(dtype), "sd_quantize_rows_int8: bad dtype");
    if (d != 64 && d != 128) {
        set_error("sd_quantize_rows_int8: d must be 64 or 128 (got %d)", d);
        return SD_ERR_UNSUPPORTED;
    }
    const long rows = (long)B * Hkv * T;
    if (rows == 0) return SD_OK;
    SD_REQUIRE(x && tier && codes && scales, "sd_quantize_rows_int8: null pointer");
    const int threads = 256;
    const long blocks = std::min<long>((rows * 32 + threads - 1) / threads, (long)num_sms() * 16);
    cudaStream_t st = as_stream(stream);
    if (dtype == SD_BF16) {
        if (d == 128)
            quantize_rows_kernel<bf16_t, 128><<<(unsigned)blocks, threads, 0, st>>>(
                static_cast<const bf16_t*>(x), tier, B, Hkv, T, codes, scales);
        else
            quantize_rows_kernel<bf16_t, 64><<<(unsigned)blocks, threads, 0, st>>>(
                static_cast<const bf16_t*>(x), tier, B, Hkv, T, codes, scales);
    } else {
        if (d == 128)
            quantize_rows_kernel<float, 128><<<(unsigned)blocks, threads, 0, st>>>(
                static_cast<const float*>(x), tier, B, Hkv, T, codes, scales);
        else
            quantize_rows_kernel<float, 64><<<(unsigned)blocks, threads, 0, st>>>(
                static_cast<const float*>(x), tier, B, Hkv, T, codes, scales);
    }
    return launch_status("sd_quantize_rows_int8");
}
