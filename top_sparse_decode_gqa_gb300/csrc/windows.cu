// windows.cu -- block scores on overlapping compression windows, and the tokens of the
// selected windows, each once.
//
// SparDA (gist.science summary), "Estrategia de Treinamento": the inference block grid is a
// compression window of 32 tokens moved by 16, and finer scores are max-pooled onto that
// grid.  Reading taken: a window's score is the maximum of the token scores it covers; the
// selected windows' tokens are their union (overlapping windows share tokens, which attention
// must see once), kept as whole segments of `stride` tokens.
#include <algorithm>

#include "sd_common.cuh"
#include "sd_host.h"

namespace sd {
namespace {

constexpr int kWinThreads = 256;
constexpr int kWinHistBins = 2048;
constexpr int kMaxSegWords = 2048;  // 65536 segments per row

int window_count(int N, int kernel, int stride) {
    if (N <= 0) return 0;
    if (N <= kernel) return 1;
    return 1 + (N - kernel + stride - 1) / stride;
}

// Grid (window groups of 256, rows): thread -> window n; the scores are read from L2 (just
// written by the indexer); the optional histogram is the one sd_topk takes (top 11 bits of
// the order key), added with warp-aggregated atomics.
__global__ void __launch_bounds__(kWinThreads)
    window_max_kernel(const float* __restrict__ scores, int N, int NW, int kernel, int stride,
                      float* __restrict__ w, uint32_t* __restrict__ key_hist) {
    pdl_wait();
    const int r = blockIdx.y;
    const int n = blockIdx.x * kWinThreads + threadIdx.x;
    const bool valid = n < NW;
    float m = -INFINITY;
    if (valid) {
        const float* srow = scores + (size_t)r * N;
        const long t0 = (long)n * stride, t1 = t0 + kernel < (long)N ? t0 + kernel : (long)N;
        if (((t0 | t1) & 3) == 0 && (reinterpret_cast<uintptr_t>(srow) & 15) == 0) {
            // 16-byte loads, eight issued before any is used (a window of 32 scores: one
            // round trip instead of one per score behind the running max)
            const float4* p4 = reinterpret_cast<const float4*>(srow + t0);
            const int n4 = (int)((t1 - t0) >> 2);
            for (int i0 = 0; i0 < n4; i0 += 8) {
                float4 x[8];
#pragma unroll
                for (int u = 0; u < 8; ++u)
                    x[u] = i0 + u < n4 ? __ldg(p4 + i0 + u) : make_float4(-INFINITY, -INFINITY, -INFINITY, -INFINITY);
#pragma unroll
                for (int u = 0; u < 8; ++u) m = fmaxf(m, fmaxf(fmaxf(x[u].x, x[u].y), fmaxf(x[u].z, x[u].w)));
            }
        } else {
            for (long t = t0; t < t1; ++t) m = fmaxf(m, __ldg(srow + t));
        }
        w[(size_t)r * NW + n] = m;
    }
    if (key_hist != nullptr) {
        const uint32_t dg = valid ? float_key(m) >> 21 : 0xffffffffu;
        const uint32_t peers = __match_any_sync(0xffffffffu, dg);
        if (valid && (threadIdx.x & 31) == __ffs(peers) - 1)
            atomicAdd(key_hist + (size_t)r * kWinHistBins + dg, (uint32_t)__popc(peers));
    }
}

// Inclusive prefix sum over the block's 256 threads.
SD_DEVINL uint32_t block_scan_256(uint32_t v, uint32_t* wsum) {
    const int lane = threadIdx.x & 31, warp = threadIdx.x >> 5;
#pragma unroll
    for (int o = 1; o < 32; o <<= 1) {
        const uint32_t x = __shfl_up_sync(0xffffffffu, v, o);
        if (lane >= o) v += x;
    }
    if (lane == 31) wsum[warp] = v;
    __syncthreads();
    uint32_t off = 0;
#pragma unroll
    for (int i = 0; i < kWinThreads / 32; ++i)
        if (i < warp) off += wsum[i];
    __syncthreads();
    return v + off;
}

// One CTA per row: a bitmap of the row's NS segments marks every segment of every selected
// window; thread t then owns bitmap words [t*W, t*W + W) and writes their set bits, in
// ascending order, at the offset a block scan gives it; the tail is padded with -1.
__global__ void __launch_bounds__(kWinThreads)
    window_union_kernel(const int32_t* __restrict__ widx, int k, int NW, int NS, int per,
                        int32_t* __restrict__ segs, int max_segs, int32_t* err) {
    __shared__ uint32_t bm[kMaxSegWords];
    __shared__ uint32_t wsum[kWinThreads / 32];
    pdl_wait();
    const int r = blockIdx.x, tid = threadIdx.x;
    const int nsw = (NS + 31) / 32;
    for (int i = tid; i < nsw; i += kWinThreads) bm[i] = 0u;
    __syncthreads();
    for (int j = tid; j < k; j += kWinThreads) {
        const int n = widx[(size_t)r * k + j];
        if (n < 0 || n >= NW) {
            report(err, SD_DEVERR_INDEX);
            continue;
        }
        for (int q = 0; q < per; ++q) {
            const int g = n + q;
            if (g < NS) atomicOr(&bm[g >> 5], 1u << (g & 31));
        }
    }
    __syncthreads();
    const int W = (nsw + kWinThreads - 1) / kWinThreads;
    const int w0 = tid * W, w1 = w0 + W < nsw ? w0 + W : nsw;
    uint32_t cnt = 0;
    for (int i = w0; i < w1; ++i) cnt += __popc(bm[i]);
    const uint32_t incl = block_scan_256(cnt, wsum);
    uint32_t at = incl - cnt;
    int32_t* orow = segs + (size_t)r * max_segs;
    for (int i = w0; i < w1; ++i) {
        uint32_t bits = bm[i];
        while (bits != 0u) {
            const int b = __ffs(bits) - 1;
            bits &= bits - 1u;
            if (at < (uint32_t)max_segs) orow[at] = i * 32 + b;
            ++at;
        }
    }
    if (tid == kWinThreads - 1) wsum[0] = incl;  // the row's total (the last thread's inclusive sum)
    __syncthreads();
    for (int i = (int)wsum[0] + tid; i < max_segs; i += kWinThreads) orow[i] = -1;
}

}  // namespace
}  // namespace sd

using namespace sd;

extern "C" int sd_window_count(int N, int kernel, int stride) {
    if (N < 0 || kernel < 1 || stride < 1) return 0;
    return window_count(N, kernel, stride);
}

extern "C" sd_status sd_window_max(const float* scores, int rows, int N, int kernel, int stride, float* wscores,
                                   uint32_t* key_hist, void* stream) {
    clear_error();
    SD_REQUIRE(rows >= 0 && N >= 0, "sd_window_max: negative size");
    SD_REQUIRE(stride >= 1 && kernel >= stride && kernel <= 1024,
               "sd_window_max: need 1 <= stride <= kernel <= 1024 (kernel %d, stride %d)", kernel, stride);
    SD_REQUIRE(rows <= 65535, "sd_window_max: rows must be <= 65535");
    const int NW = window_count(N, kernel, stride);
    if (rows == 0 || NW == 0) return SD_OK;
    SD_REQUIRE(scores && wscores, "sd_window_max: null pointer");
    const dim3 grid((unsigned)((NW + kWinThreads - 1) / kWinThreads), (unsigned)rows);
    SD_CUDA_CHECK(launch_pdl(window_max_kernel, grid, dim3(kWinThreads), 0, as_stream(stream), scores, N, NW, kernel,
                             stride, wscores, key_hist),
                  "sd_window_max: launch");
    return launch_status("sd_window_max");
}

extern "C" sd_status sd_window_union(const int32_t* widx, int rows, int k, int N, int kernel, int stride,
                                     int32_t* segs, int max_segs, int32_t* err_word, void* stream) {
    clear_error();
    SD_REQUIRE(rows >= 0 && k >= 0 && N >= 0, "sd_window_union: negative size");
    SD_REQUIRE(stride >= 1 && kernel >= stride && kernel % stride == 0,
               "sd_window_union: kernel (%d) must be a multiple of stride (%d)", kernel, stride);
    SD_REQUIRE(N % stride == 0, "sd_window_union: N (%d) must be a multiple of stride (%d)", N, stride);
    SD_REQUIRE(N / stride <= kMaxSegWords * 32, "sd_window_union: at most %d segments per row", kMaxSegWords * 32);
    SD_REQUIRE((long)max_segs >= (long)k * (kernel / stride),
               "sd_window_union: max_segs (%d) must be >= k * kernel/stride (%d)", max_segs, k * (kernel / stride));
    if (rows == 0 || max_segs == 0) return SD_OK;
    SD_REQUIRE(segs && (k == 0 || widx), "sd_window_union: null pointer");
    SD_CUDA_CHECK(launch_pdl(window_union_kernel, dim3((unsigned)rows), dim3(kWinThreads), 0, as_stream(stream), widx,
                             k, window_count(N, kernel, stride), N / stride, kernel / stride, segs, max_segs, err_word),
                  "sd_window_union: launch");
    return launch_status("sd_window_union");
}
