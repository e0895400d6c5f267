// index_score.cu -- compact indexer score (one head per KV group, no softmax) and the
// block-key pooling helper.
//
// SparDA (gist.science summary), sec. 2 "Indexador de Previsao Compacto": the indexer
// keeps one head per GQA group and scores each cached token by a dot product with no
// softmax.  Scoring reads every indexer key once, so the kernel is a pure HBM stream:
// persistent CTAs (3 per SM) walk contiguous 16 KB tiles of key rows, each tile moved by
// one 1-D bulk copy (TMA) into a 4-stage shared-memory ring completed on mbarriers, and
// the CUDA cores take the dot products straight from shared memory.  Each token row is
// read by LPR lanes with one 16-byte load each; LPR-lane shuffles finish the sum.
#include "sd_common.cuh"
#include "sd_host.h"

namespace sd {
namespace {

constexpr int kIdxThreads = 256;
constexpr int kIdxWarps = kIdxThreads / 32;
constexpr int kTileBytes = 16384;
constexpr int kStages = 4;
constexpr int kCtasPerSm = 3;
constexpr int kIdxSmem = kStages * kTileBytes + kStages * 8;

template <typename KT, int DI, int VT>
__global__ void __launch_bounds__(kIdxThreads) index_score_kernel(
    const void* __restrict__ q_idx, int q_dtype, const KT* __restrict__ k_idx, int rows, int V,
    int N, float* __restrict__ scores, int32_t* err_word) {
    using U = Unpack16<KT>;
    constexpr int ROWB = DI * (int)sizeof(KT);  // bytes per key row
    constexpr int LPR = ROWB / 16;              // lanes per row
    constexpr int EPL = U::kElems;              // elements per lane
    constexpr int RPW = 32 / LPR;               // rows per warp per step
    constexpr int TT = kTileBytes / ROWB;       // rows per tile
    static_assert(TT % (kIdxWarps * RPW) == 0, "tile must split evenly over the warps");

    extern __shared__ __align__(128) uint8_t smem[];
    uint64_t* bars = reinterpret_cast<uint64_t*>(smem + kStages * kTileBytes);

    const int tid = threadIdx.x, lane = tid & 31, warp = tid >> 5;
    const int sub = lane % LPR;
    const int rsub = lane / LPR;
    const long tiles_per_row = (N + TT - 1) / TT;
    const long total = (long)rows * tiles_per_row;

    if (tid == 0) {
        for (int s = 0; s < kStages; ++s) mbar_init(&bars[s], 1);
        fence_mbarrier_init();
    }
    __syncthreads();

    auto issue = [&](long t, int s) {
        const long r = t / tiles_per_row;
        const long t0 = (t % tiles_per_row) * TT;
        const uint32_t bytes = (uint32_t)(N - t0 < TT ? N - t0 : (long)TT) * ROWB;
        mbar_arrive_expect_tx(&bars[s], bytes);
        bulk_g2s(smem + s * kTileBytes, k_idx + (r * N + t0) * DI, bytes, &bars[s]);
    };

    if (tid == 0) {
        for (int s = 0; s < kStages; ++s) {
            const long t = blockIdx.x + (long)s * gridDim.x;
            if (t < total) issue(t, s);
        }
    }

    float q[VT][EPL];
    long cur_row = -1;
    long i = 0;
    bool timed_out = false;
    for (;; ++i) {
        const long t = blockIdx.x + i * gridDim.x;
        if (t >= total) break;
        const int s = (int)(i % kStages);
        const long r = t / tiles_per_row;
        const long t0 = (t % tiles_per_row) * TT;
        const int n = (int)(N - t0 < TT ? N - t0 : (long)TT);
        if (r != cur_row) {
            cur_row = r;
#pragma unroll
            for (int v = 0; v < VT; ++v)
#pragma unroll
                for (int e = 0; e < EPL; ++e)
                    q[v][e] = (v < V) ? load_elem(q_idx, q_dtype, (size_t)(r * V + v) * DI + sub * EPL + e)
                                      : 0.f;
        }
        const bool ok = mbar_wait(&bars[s], (uint32_t)((i / kStages) & 1));
        if (__syncthreads_or(!ok)) {
            timed_out = true;
            break;
        }
        const uint8_t* tile = smem + s * kTileBytes;
        float* out = scores + r * N + t0;
#pragma unroll
        for (int rr = warp * RPW + rsub; rr < TT; rr += kIdxWarps * RPW) {
            float x[EPL];
            U::run(lds128(tile + rr * ROWB + sub * 16), x);
            float acc[VT];
#pragma unroll
            for (int v = 0; v < VT; ++v) {
                acc[v] = 0.f;
#pragma unroll
                for (int e = 0; e < EPL; ++e) acc[v] = fmaf(x[e], q[v][e], acc[v]);
            }
#pragma unroll
            for (int o = LPR / 2; o > 0; o >>= 1)
#pragma unroll
                for (int v = 0; v < VT; ++v) acc[v] += __shfl_xor_sync(0xffffffffu, acc[v], o);
            float best = acc[0];
#pragma unroll
            for (int v = 1; v < VT; ++v)
                if (v < V) best = fmaxf(best, acc[v]);
            if (sub == 0 && rr < n) out[rr] = best;
        }
        __syncthreads();
        if (tid == 0) {
            const long tn = blockIdx.x + (i + kStages) * gridDim.x;
            if (tn < total) {
                fence_proxy_async_shared();
                issue(tn, s);
            }
        }
    }
    if (timed_out && tid == 0) {
        report(err_word, SD_DEVERR_TIMEOUT);
        // Let the copies this CTA still has in flight land (bounded) before exiting.
        for (long j = i; j < i + kStages; ++j) {
            const long t = blockIdx.x + j * gridDim.x;
            if (t >= total) break;
            mbar_wait(&bars[j % kStages], (uint32_t)((j / kStages) & 1));
        }
    }
}

template <typename KT, int DI, int VT>
sd_status launch_index_score(const void* q_idx, int q_dtype, const void* k_idx, int rows, int V,
                             int N, float* scores, int32_t* err_word, cudaStream_t st) {
    constexpr int ROWB = DI * (int)sizeof(KT);
    constexpr int TT = kTileBytes / ROWB;
    auto kern = index_score_kernel<KT, DI, VT>;
    static bool configured = false;  // attribute is per function; setting it twice is harmless
    if (!configured) {
        SD_CUDA_CHECK(cudaFuncSetAttribute(kern, cudaFuncAttributeMaxDynamicSharedMemorySize, kIdxSmem),
                      "sd_index_score: cudaFuncSetAttribute");
        configured = true;
    }
    const long total = (long)rows * ((N + TT - 1) / TT);
    const long grid = std::min<long>(total, (long)num_sms() * kCtasPerSm);
    kern<<<(unsigned)grid, kIdxThreads, kIdxSmem, st>>>(q_idx, q_dtype,
                                                        reinterpret_cast<const KT*>(k_idx), rows,
                                                        V, N, scores, err_word);
    return launch_status("sd_index_score");
}

template <typename KT>
__global__ void block_pool_kernel(const KT* __restrict__ k_idx, int dtype, int T, int dI,
                                  int block, float* __restrict__ pooled) {
    const int n = blockIdx.x, r = blockIdx.y, j = threadIdx.x;
    const int NB = T / block;
    float sum = 0.f;
    for (int t = 0; t < block; ++t)
        sum += load_elem(k_idx, dtype, ((size_t)r * T + (size_t)n * block + t) * dI + j);
    pooled[((size_t)r * NB + n) * dI + j] = __fdiv_rn(sum, (float)block);
}

}  // namespace
}  // namespace sd

using namespace sd;

extern "C" sd_status sd_index_score(const void* q_idx, sd_dtype q_dtype, const void* k_idx,
                                    sd_dtype k_dtype, int B, int Hkv, int V, int N, int d_idx,
                                    float* scores, int32_t* err_word, void* stream) {
    clear_error();
    SD_REQUIRE(B >= 0 && Hkv >= 0 && N >= 0, "sd_index_score: negative size");
    SD_REQUIRE(valid_dtype(q_dtype) && valid_dtype(k_dtype), "sd_index_score: bad dtype");
    SD_REQUIRE(V >= 1 && V <= 8, "sd_index_score: V must be in [1, 8] (got %d)", V);
    if (d_idx != 64 && d_idx != 128) {
        set_error("sd_index_score: d_idx must be 64 or 128 (got %d)", d_idx);
        return SD_ERR_UNSUPPORTED;
    }
    const long rows = (long)B * Hkv;
    if (rows == 0 || N == 0) return SD_OK;
    SD_REQUIRE(q_idx && k_idx && scores, "sd_index_score: null pointer");
    SD_REQUIRE(aligned16(k_idx) && aligned16(scores), "sd_index_score: pointers must be 16-byte aligned");
    SD_REQUIRE(rows <= (1L << 30), "sd_index_score: too many rows");
    cudaStream_t st = as_stream(stream);
    const int r = (int)rows;
    if (k_dtype == SD_BF16) {
        if (d_idx == 128)
            return V == 1 ? launch_index_score<bf16_t, 128, 1>(q_idx, q_dtype, k_idx, r, V, N, scores, err_word, st)
                          : launch_index_score<bf16_t, 128, 8>(q_idx, q_dtype, k_idx, r, V, N, scores, err_word, st);
        return V == 1 ? launch_index_score<bf16_t, 64, 1>(q_idx, q_dtype, k_idx, r, V, N, scores, err_word, st)
                      : launch_index_score<bf16_t, 64, 8>(q_idx, q_dtype, k_idx, r, V, N, scores, err_word, st);
    }
    if (d_idx == 128)
        return V == 1 ? launch_index_score<float, 128, 1>(q_idx, q_dtype, k_idx, r, V, N, scores, err_word, st)
                      : launch_index_score<float, 128, 8>(q_idx, q_dtype, k_idx, r, V, N, scores, err_word, st);
    return V == 1 ? launch_index_score<float, 64, 1>(q_idx, q_dtype, k_idx, r, V, N, scores, err_word, st)
                  : launch_index_score<float, 64, 8>(q_idx, q_dtype, k_idx, r, V, N, scores, err_word, st);
}

extern "C" sd_status sd_block_pool(const void* k_idx, sd_dtype k_dtype, int B, int Hkv, int T,
                                   int d_idx, int block, float* pooled, void* stream) {
    clear_error();
    SD_REQUIRE(B >= 0 && Hkv >= 0 && T >= 0, "sd_block_pool: negative size");
    SD_REQUIRE(valid_dtype(k_dtype), "sd_block_pool: bad dtype");
    SD_REQUIRE(block >= 1 && block <= 4096, "sd_block_pool: block must be in [1, 4096]");
    SD_REQUIRE(T % block == 0, "sd_block_pool: T (%d) must be a multiple of block (%d)", T, block);
    if (d_idx != 64 && d_idx != 128) {
        set_error("sd_block_pool: d_idx must be 64 or 128 (got %d)", d_idx);
        return SD_ERR_UNSUPPORTED;
    }
    const long rows = (long)B * Hkv;
    if (rows == 0 || T == 0) return SD_OK;
    SD_REQUIRE(k_idx && pooled, "sd_block_pool: null pointer");
    SD_REQUIRE(rows <= 65535, "sd_block_pool: B*Hkv must be <= 65535");
    dim3 grid(T / block, (unsigned)rows);
    if (k_dtype == SD_BF16)
        block_pool_kernel<bf16_t><<<grid, d_idx, 0, as_stream(stream)>>>(
            reinterpret_cast<const bf16_t*>(k_idx), k_dtype, T, d_idx, block, pooled);
    else
        block_pool_kernel<float><<<grid, d_idx, 0, as_stream(stream)>>>(
            reinterpret_cast<const float*>(k_idx), k_dtype, T, d_idx, block, pooled);
    return launch_status("sd_block_pool");
}
