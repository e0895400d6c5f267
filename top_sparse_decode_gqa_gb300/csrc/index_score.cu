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
#include <cuda_fp16.h>

#include "sd_common.cuh"
#include "sd_host.h"

namespace sd {
namespace {

constexpr int kIdxWarps = 12;
constexpr int kIdxThreads = kIdxWarps * 32;
constexpr int kWarpTileBytes = 4096;  // one bulk copy: 16 rows of 256 B (8 of 512 B, 32 of 128 B)
constexpr int kWarpStages = 4;
constexpr int kIdxSmem = kIdxWarps * kWarpStages * (kWarpTileBytes + 8);

// Reduce-scatter of kR partial sums across the L lanes that share them (lane bits below L):
// after it, each lane holds the complete sum of one of the kR values, namely acc[0], and
// the index of that value is returned.  Halving steps exchange half of the remaining
// values with the partner lane; once one value is left, the remaining steps just add.
template <int L, int kR>
SD_DEVINL int reduce_scatter(float (&acc)[kR], int lane) {
    int base = 0;
    int count = kR;
#pragma unroll
    for (int o = L / 2; o > 0; o >>= 1) {
        if (count > 1) {
            const int half = count / 2;
            const bool hi = (lane & o) != 0;
#pragma unroll
            for (int j = 0; j < half; ++j) {
                const float send = hi ? acc[j] : acc[j + half];
                const float keep = hi ? acc[j + half] : acc[j];
                acc[j] = keep + __shfl_xor_sync(0xffffffffu, send, o);
            }
            if (hi) base += half;
            count = half;
        } else {
            acc[0] += __shfl_xor_sync(0xffffffffu, acc[0], o);
        }
    }
    return base;
}

// Persistent CTAs of kIdxWarps independent warps.  Each warp owns a contiguous range of
// 4 KB key tiles and runs its own kWarpStages-deep pipeline: lane 0 issues one bulk copy
// per tile into the warp's ring, all lanes wait on that stage's mbarrier, score the tile
// and hand the stage back to lane 0 with a warp barrier -- no CTA-wide synchronization.
// Lane layout within a tile: lane = g * LPR + c; c picks the 16-byte chunk of a row, g
// one of the GROUPS row groups; the lane accumulates 8 rows (g, g + GROUPS, ...) for its
// chunk and a reduce-scatter over the LPR lanes leaves each lane one complete row sum.
template <typename KT, int DI, int VT>
__global__ void __launch_bounds__(kIdxThreads, 1) index_score_kernel(
    const void* __restrict__ q_idx, int q_dtype, const KT* __restrict__ k_idx, int rows, int V,
    int N, float* __restrict__ scores, uint32_t* __restrict__ key_hist, int32_t* err_word, int per_query) {
    using U = Unpack16<KT>;
    constexpr int ROWB = DI * (int)sizeof(KT);  // bytes per key row: 128, 256 or 512
    constexpr int LPR = ROWB / 16;              // lanes sharing a row
    constexpr int EPL = U::kElems;              // elements per lane
    constexpr int TR = kWarpTileBytes / ROWB;   // rows per tile
    constexpr int GROUPS = 32 / LPR;            // row groups per warp
    constexpr int RPL = TR / GROUPS;            // rows per lane
    static_assert(RPL == 8, "each lane accumulates 8 rows");

    extern __shared__ __align__(128) uint8_t smem[];
    const int lane = threadIdx.x & 31, warp = threadIdx.x >> 5;
    uint8_t* ring = smem + warp * kWarpStages * kWarpTileBytes;
    uint64_t* bars =
        reinterpret_cast<uint64_t*>(smem + kIdxWarps * kWarpStages * kWarpTileBytes) + warp * kWarpStages;
    const int c = lane % LPR, g = lane / LPR;

    // Tiles are dealt round-robin over all warps of the grid (tile = gw + i * nw), so the
    // tiles in flight at any moment are neighbours in memory (DRAM page locality).
    const uint32_t tpr = (uint32_t)((N + TR - 1) / TR);
    const uint32_t total = (uint32_t)rows * tpr;
    const uint32_t gw = blockIdx.x * kIdxWarps + warp;
    const uint32_t nw = gridDim.x * kIdxWarps;
    const uint32_t ntiles = gw < total ? (total - gw + nw - 1) / nw : 0u;

    pdl_launch_dependents();
    if (lane == 0) {
        for (int s = 0; s < kWarpStages; ++s) mbar_init(&bars[s], 1);
        fence_mbarrier_init();
    }
    __syncwarp();

    const uint64_t stream_policy = l2_evict_first_policy();  // keys are read once
    auto issue = [&](uint32_t j, int s) {  // lane 0: tile j of this warp into stage s
        const uint32_t t = gw + j * nw;
        const uint32_t ir = t / tpr, it0 = (t - ir * tpr) * TR;
        const uint32_t n = min((uint32_t)TR, (uint32_t)N - it0);
        mbar_arrive_expect_tx(&bars[s], n * ROWB);
        bulk_g2s_hint(ring + s * kWarpTileBytes, k_idx + ((size_t)ir * N + it0) * DI, n * ROWB, &bars[s],
                      stream_policy);
    };
    if (lane == 0)
        for (uint32_t s = 0; s < min((uint32_t)kWarpStages, ntiles); ++s) issue(s, (int)s);

    float q[VT][EPL];
    uint32_t q_row = 0xffffffffu;
    uint32_t i = 0;
    bool timed_out = false;
    for (; i < ntiles; ++i) {
        const int s = (int)(i % kWarpStages);
        const uint32_t t = gw + i * nw;
        const uint32_t cr = t / tpr, ct0 = (t - cr * tpr) * TR;
        if (cr != q_row) {
            q_row = cr;
#pragma unroll
            for (int v = 0; v < VT; ++v)
#pragma unroll
                for (int e = 0; e < EPL; ++e)
                    q[v][e] = (v < V) ? load_elem(q_idx, q_dtype, ((size_t)cr * V + v) * DI + c * EPL + e) : 0.f;
        }
        const bool ok = mbar_wait(&bars[s], (i / kWarpStages) & 1u);
        if (__any_sync(0xffffffffu, !ok)) {
            timed_out = true;
            break;
        }
        const uint8_t* tile = ring + s * kWarpTileBytes;
        float acc[VT][RPL];
#pragma unroll
        for (int j = 0; j < RPL; ++j) {
            float x[EPL];
            U::run(lds128(tile + (g + GROUPS * j) * ROWB + c * 16), x);
#pragma unroll
            for (int v = 0; v < VT; ++v) {
                float a = 0.f;
#pragma unroll
                for (int e = 0; e < EPL; ++e) a = fmaf(x[e], q[v][e], a);
                acc[v][j] = a;
            }
        }
        int ridx = 0;
#pragma unroll
        for (int v = 0; v < VT; ++v) ridx = reduce_scatter<LPR>(acc[v], lane);
        // lanes holding a duplicate of the same row (bits below LPR/8) do not store
        const int row = g + GROUPS * ridx;
        const uint32_t n = min((uint32_t)TR, (uint32_t)N - ct0);
        const bool store = (lane & (LPR / 8 - 1)) == 0 && (uint32_t)row < n;
        auto put = [&](uint32_t srow, float x) {  // score row srow: store, histogram
            if (store) scores[(size_t)srow * N + ct0 + row] = x;
            if (key_hist != nullptr) {
                const uint32_t dg = float_key(x) >> 21;
                const uint32_t peers = __match_any_sync(0xffffffffu, store ? dg : 0xffffffffu);
                if (store && lane == __ffs(peers) - 1)
                    atomicAdd(&key_hist[(size_t)srow * 2048 + dg], (uint32_t)__popc(peers));
            }
        };
        if (per_query) {
#pragma unroll
            for (int v = 0; v < VT; ++v)
                if (v < V) put(cr * (uint32_t)V + (uint32_t)v, acc[v][0]);
        } else {
            float best = acc[0][0];
#pragma unroll
            for (int v = 1; v < VT; ++v)
                if (v < V) best = fmaxf(best, acc[v][0]);
            put(cr, best);
        }
        __syncwarp();
        if (lane == 0 && i + kWarpStages < ntiles) {
            fence_proxy_async_shared();
            issue(i + kWarpStages, s);
        }
    }
    if (timed_out && lane == 0) {
        report(err_word, SD_DEVERR_TIMEOUT);
        // Let the copies this warp still has in flight land (bounded) before exiting.
        for (uint32_t j = i; j < ntiles && j < i + kWarpStages; ++j)
            mbar_wait(&bars[j % kWarpStages], (j / kWarpStages) & 1u);
    }
}

template <typename KT, int DI, int VT>
sd_status launch_index_score(const void* q_idx, int q_dtype, const void* k_idx, int rows, int V,
                             int N, float* scores, uint32_t* key_hist, int32_t* err_word, int per_query,
                             cudaStream_t st) {
    auto kern = index_score_kernel<KT, DI, VT>;
    SD_CUDA_CHECK(cudaFuncSetAttribute(kern, cudaFuncAttributeMaxDynamicSharedMemorySize, kIdxSmem),
                  "sd_index_score: cudaFuncSetAttribute");
    constexpr int TR = kWarpTileBytes / (DI * (int)sizeof(KT));
    const long tiles = (long)rows * ((N + TR - 1) / TR);
    const long grid = std::min<long>((tiles + kIdxWarps - 1) / kIdxWarps, (long)num_sms());
    kern<<<(unsigned)grid, kIdxThreads, kIdxSmem, st>>>(q_idx, q_dtype, reinterpret_cast<const KT*>(k_idx),
                                                       rows, V, N, scores, key_hist, err_word, per_query);
    return launch_status("sd_index_score");
}

template <typename KT, typename OT>
__global__ void block_pool_kernel(const KT* __restrict__ k_idx, int dtype, int T, int dI,
                                  int block, OT* __restrict__ pooled) {
    const int n = blockIdx.x, r = blockIdx.y, j = threadIdx.x;
    const int NB = T / block;
    float sum = 0.f;
    for (int t = 0; t < block; ++t)
        sum += load_elem(k_idx, dtype, ((size_t)r * T + (size_t)n * block + t) * dI + j);
    const float mean = __fdiv_rn(sum, (float)block);
    if constexpr (sizeof(OT) == 2)
        pooled[((size_t)r * NB + n) * dI + j] = __float2half_rn(mean);
    else
        pooled[((size_t)r * NB + n) * dI + j] = mean;
}

}  // namespace
}  // namespace sd

using namespace sd;

namespace {

sd_status index_score_common(const char* who, const void* q_idx, sd_dtype q_dtype, const void* k_idx,
                             sd_dtype k_dtype, int B, int Hkv, int V, int N, int d_idx, float* scores,
                             uint32_t* key_hist, int32_t* err_word, int per_query, void* stream) {
    clear_error();
    SD_REQUIRE(B >= 0 && Hkv >= 0 && N >= 0, "%s: negative size", who);
    const bool f16 = q_dtype == SD_F16 && k_dtype == SD_F16;
    SD_REQUIRE(f16 || (valid_dtype(q_dtype) && valid_dtype(k_dtype)),
               "%s: q and k must be F32 or BF16 each, or both F16", who);
    const bool tc = f16 || (k_dtype == SD_BF16 && q_dtype == SD_BF16);
    const int vmax = per_query && tc ? 16 : 8;
    SD_REQUIRE(V >= 1 && V <= vmax, "%s: V must be in [1, %d] (got %d)", who, vmax, V);
    if (d_idx != 64 && d_idx != 128) {
        set_error("%s: d_idx must be 64 or 128 (got %d)", who, d_idx);
        return SD_ERR_UNSUPPORTED;
    }
    const long rows = (long)B * Hkv;
    if (rows == 0 || N == 0) return SD_OK;
    SD_REQUIRE(q_idx && k_idx && scores, "%s: null pointer", who);
    SD_REQUIRE(aligned16(k_idx) && aligned16(scores), "%s: pointers must be 16-byte aligned", who);
    SD_REQUIRE(rows <= (1L << 30) && rows * (per_query ? V : 1) * (long)N < (1L << 36), "%s: too many rows", who);
    cudaStream_t st = as_stream(stream);
    const int r = (int)rows;
    // bf16 keys and queries: the contraction runs on the tensor cores (exact for the
    // integer-valued indexer: products exact, fp32 sums of integers below 2^24 exact)
    if (tc) {
        SD_REQUIRE(aligned16(q_idx), "%s: q must be 16-byte aligned", who);
        SD_REQUIRE((long)rows * N * (per_query ? V : 1) < (1L << 31) && (long)rows * V < (1L << 31),
                   "%s: too many rows", who);
        return index_score_tc_launch(q_idx, k_idx, r, V, N, d_idx, scores, key_hist, err_word, per_query, f16, st);
    }
    const int pq = per_query;
    if (k_dtype == SD_BF16) {
        if (d_idx == 128)
            return V == 1 ? launch_index_score<bf16_t, 128, 1>(q_idx, q_dtype, k_idx, r, V, N, scores, key_hist, err_word, pq, st)
                          : launch_index_score<bf16_t, 128, 8>(q_idx, q_dtype, k_idx, r, V, N, scores, key_hist, err_word, pq, st);
        return V == 1 ? launch_index_score<bf16_t, 64, 1>(q_idx, q_dtype, k_idx, r, V, N, scores, key_hist, err_word, pq, st)
                      : launch_index_score<bf16_t, 64, 8>(q_idx, q_dtype, k_idx, r, V, N, scores, key_hist, err_word, pq, st);
    }
    if (d_idx == 128)
        return V == 1 ? launch_index_score<float, 128, 1>(q_idx, q_dtype, k_idx, r, V, N, scores, key_hist, err_word, pq, st)
                      : launch_index_score<float, 128, 8>(q_idx, q_dtype, k_idx, r, V, N, scores, key_hist, err_word, pq, st);
    return V == 1 ? launch_index_score<float, 64, 1>(q_idx, q_dtype, k_idx, r, V, N, scores, key_hist, err_word, pq, st)
                  : launch_index_score<float, 64, 8>(q_idx, q_dtype, k_idx, r, V, N, scores, key_hist, err_word, pq, st);
}

}  // namespace

extern "C" sd_status sd_index_score(const void* q_idx, sd_dtype q_dtype, const void* k_idx,
                                    sd_dtype k_dtype, int B, int Hkv, int V, int N, int d_idx,
                                    float* scores, uint32_t* key_hist, int32_t* err_word,
                                    void* stream) {
    return index_score_common("sd_index_score", q_idx, q_dtype, k_idx, k_dtype, B, Hkv, V, N, d_idx, scores,
                              key_hist, err_word, 0, stream);
}

extern "C" sd_status sd_index_score_heads(const void* q, sd_dtype q_dtype, const void* k, sd_dtype k_dtype, int B,
                                          int Hkv, int V, int N, int d, float* scores, uint32_t* key_hist,
                                          int32_t* err_word, void* stream) {
    return index_score_common("sd_index_score_heads", q, q_dtype, k, k_dtype, B, Hkv, V, N, d, scores, key_hist,
                              err_word, 1, stream);
}

extern "C" sd_status sd_block_pool(const void* k_idx, sd_dtype k_dtype, int B, int Hkv, int T,
                                   int d_idx, int block, void* pooled, sd_dtype pooled_dtype, void* stream) {
    clear_error();
    SD_REQUIRE(B >= 0 && Hkv >= 0 && T >= 0, "sd_block_pool: negative size");
    SD_REQUIRE(valid_dtype(k_dtype), "sd_block_pool: bad dtype");
    SD_REQUIRE(pooled_dtype == SD_F32 || pooled_dtype == SD_F16, "sd_block_pool: pooled_dtype must be F32 or F16");
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
    cudaStream_t st = as_stream(stream);
    const bool half_out = pooled_dtype == SD_F16;
    if (k_dtype == SD_BF16) {
        auto k = reinterpret_cast<const bf16_t*>(k_idx);
        if (half_out)
            block_pool_kernel<bf16_t, __half><<<grid, d_idx, 0, st>>>(k, k_dtype, T, d_idx, block, static_cast<__half*>(pooled));
        else
            block_pool_kernel<bf16_t, float><<<grid, d_idx, 0, st>>>(k, k_dtype, T, d_idx, block, static_cast<float*>(pooled));
    } else {
        auto k = reinterpret_cast<const float*>(k_idx);
        if (half_out)
            block_pool_kernel<float, __half><<<grid, d_idx, 0, st>>>(k, k_dtype, T, d_idx, block, static_cast<__half*>(pooled));
        else
            block_pool_kernel<float, float><<<grid, d_idx, 0, st>>>(k, k_dtype, T, d_idx, block, static_cast<float*>(pooled));
    }
    return launch_status("sd_block_pool");
}
