// topk.cu -- exact top-k per row, ties to the lower index, ascending output.
//
// "Esparsidade de Contexto no Tempo de Inferencia" (gist.science summary), sec. 2
// "Mecanismos de Esparsidade": Oracle Top-K is the exact selection of the k highest-
// scoring tokens; SparDA (gist.science summary), sec. 2 item 1, selects top-k blocks the
// same way.  The pages are silent on ties; the lower index wins.
//
// One 1024-thread CTA per row.  Scores become order-preserving uint32 keys (kept in
// shared memory when the row fits).  A radix select with 11/11/10-bit digits finds the
// k-th largest key `thr` and how many entries equal to it are still needed (`krem`).  A
// final ordered pass gives each warp a contiguous segment of the row: per-warp counts,
// a 32-entry scan, and warp ballots emit every key > thr and the first krem keys == thr
// in ascending index order.
#include <algorithm>

#include "sd_common.cuh"
#include "sd_host.h"

namespace sd {
namespace {

constexpr int kTkThreads = 1024;
constexpr int kTkWarps = kTkThreads / 32;
constexpr int kHistBins = 2048;

// Block-wide inclusive prefix sum of one value per thread (1024 threads).
SD_DEVINL uint32_t block_inclusive_scan(uint32_t v, uint32_t* wsum) {
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

__global__ void __launch_bounds__(kTkThreads, 1)
    topk_kernel(const float* __restrict__ scores, int N, int k, int32_t* __restrict__ idx_out,
                int cache_keys) {
    extern __shared__ __align__(16) uint32_t keys_s[];
    __shared__ uint32_t hist[kHistBins];
    __shared__ uint32_t wsum[32];
    __shared__ uint32_t sel_digit, sel_above;
    __shared__ uint32_t cnt_gt[kTkWarps], cnt_eq[kTkWarps], base_out[kTkWarps], eq_before[kTkWarps];

    const int tid = threadIdx.x, lane = tid & 31, warp = tid >> 5;
    const float* srow = scores + (size_t)blockIdx.x * N;
    int32_t* orow = idx_out + (size_t)blockIdx.x * k;
    if (k == 0) return;
    if (k == N) {
        for (int i = tid; i < N; i += kTkThreads) orow[i] = i;
        return;
    }
    if (cache_keys) {
        for (int i = tid; i < N; i += kTkThreads) keys_s[i] = float_key(srow[i]);
        __syncthreads();
    }
    auto key_at = [&](int i) -> uint32_t { return cache_keys ? keys_s[i] : float_key(srow[i]); };

    // ---- radix select of the k-th largest key
    uint32_t prefix = 0, pmask = 0;
    int krem = k;
#pragma unroll 1
    for (int pass = 0; pass < 3; ++pass) {
        const int shift = pass == 0 ? 21 : (pass == 1 ? 10 : 0);
        const uint32_t nb = pass == 2 ? 1024u : 2048u;
        for (int b = tid; b < kHistBins; b += kTkThreads) hist[b] = 0;
        __syncthreads();
        for (int base = warp * 32; base < N; base += kTkThreads) {
            const int i = base + lane;
            const bool valid = i < N;
            const uint32_t kk = valid ? key_at(i) : 0u;
            const bool in = valid && (kk & pmask) == prefix;
            const uint32_t dg = (kk >> shift) & (nb - 1);
            const uint32_t peers = __match_any_sync(0xffffffffu, in ? dg : 0xffffffffu);
            if (in && lane == __ffs(peers) - 1) atomicAdd(&hist[dg], (uint32_t)__popc(peers));
        }
        __syncthreads();
        // Thread t owns the bins [nb - per*(t+1), nb - per*t): thread 0 the highest.
        const int per = (int)nb / kTkThreads;
        const int hi = (int)nb - per * tid;  // exclusive upper bin
        uint32_t local = 0;
        for (int b = hi - per; b < hi; ++b) local += hist[b];
        const uint32_t incl = block_inclusive_scan(local, wsum);
        const uint32_t excl = incl - local;
        if (excl < (uint32_t)krem && (uint32_t)krem <= incl) {
            uint32_t above = excl;
            for (int b = hi - 1; b >= hi - per; --b) {
                if (above + hist[b] >= (uint32_t)krem) {
                    sel_digit = (uint32_t)b;
                    sel_above = above;
                    break;
                }
                above += hist[b];
            }
        }
        __syncthreads();
        prefix |= sel_digit << shift;
        pmask |= (nb - 1) << shift;
        krem -= (int)sel_above;
        __syncthreads();
    }
    const uint32_t thr = prefix;

    // ---- ordered emit: warp w scans [w*seg, (w+1)*seg)
    const int seg = ((N + kTkWarps - 1) / kTkWarps + 31) / 32 * 32;
    const int s0 = warp * seg, s1 = min(N, s0 + seg);
    uint32_t gt = 0, eq = 0;
    for (int base = s0; base < s1; base += 32) {
        const int i = base + lane;
        const bool valid = i < s1;
        const uint32_t kk = valid ? key_at(i) : 0u;
        gt += __popc(__ballot_sync(0xffffffffu, valid && kk > thr));
        eq += __popc(__ballot_sync(0xffffffffu, valid && kk == thr));
    }
    if (lane == 0) {
        cnt_gt[warp] = gt;
        cnt_eq[warp] = eq;
    }
    __syncthreads();
    if (tid == 0) {
        uint32_t eqb = 0, ob = 0;
        for (int w = 0; w < kTkWarps; ++w) {
            eq_before[w] = eqb;
            const int take = max(0, min((int)cnt_eq[w], krem - (int)eqb));
            base_out[w] = ob;
            ob += cnt_gt[w] + (uint32_t)take;
            eqb += cnt_eq[w];
        }
    }
    __syncthreads();
    uint32_t eq_seen = eq_before[warp], pos = base_out[warp];
    const uint32_t lt = lanemask_lt();
    for (int base = s0; base < s1; base += 32) {
        const int i = base + lane;
        const bool valid = i < s1;
        const uint32_t kk = valid ? key_at(i) : 0u;
        const bool is_gt = valid && kk > thr;
        const bool is_eq = valid && kk == thr;
        const uint32_t eqm = __ballot_sync(0xffffffffu, is_eq);
        const bool sel = is_gt || (is_eq && (int)(eq_seen + __popc(eqm & lt)) < krem);
        const uint32_t selm = __ballot_sync(0xffffffffu, sel);
        const uint32_t at = pos + __popc(selm & lt);
        if (sel && at < (uint32_t)k) orow[at] = i;
        pos += __popc(selm);
        eq_seen += __popc(eqm);
    }
}

}  // namespace
}  // namespace sd

using namespace sd;

extern "C" size_t sd_topk_workspace_bytes(int rows, int N, int k) {
    (void)rows;
    (void)N;
    (void)k;
    return 0;
}

extern "C" sd_status sd_topk(const float* scores, int rows, int N, int k, int32_t* idx,
                             void* workspace, size_t workspace_bytes, void* stream) {
    (void)workspace;
    (void)workspace_bytes;
    clear_error();
    SD_REQUIRE(rows >= 0 && N >= 0, "sd_topk: negative size");
    SD_REQUIRE(k >= 0 && k <= N, "sd_topk: k (%d) must be in [0, N=%d]", k, N);
    if (rows == 0 || k == 0) return SD_OK;
    SD_REQUIRE(scores && idx, "sd_topk: null pointer");
    const size_t key_bytes = (size_t)N * sizeof(uint32_t);
    const size_t static_bytes = 16 * 1024;
    const int cache = key_bytes + static_bytes <= (size_t)max_smem_optin() ? 1 : 0;
    const size_t dyn = cache ? key_bytes : 0;
    if (dyn > 48 * 1024)
        SD_CUDA_CHECK(cudaFuncSetAttribute(topk_kernel, cudaFuncAttributeMaxDynamicSharedMemorySize,
                                           (int)dyn),
                      "sd_topk: cudaFuncSetAttribute");
    topk_kernel<<<rows, kTkThreads, dyn, as_stream(stream)>>>(scores, N, k, idx, cache);
    return launch_status("sd_topk");
}
