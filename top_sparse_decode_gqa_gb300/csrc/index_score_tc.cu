// index_score_tc.cu -- the compact indexer on the 5th-generation tensor cores (tcgen05).
//
// SparDA (gist.science summary), sec. 2 "Indexador de Previsao Compacto": one indexer
// head per KV group scores every cached token with a dot product, no softmax.  With V
// verify queries sharing the selection the scores of a tile of 128 tokens are a small
// dense contraction, S[128 x V] = K_tile[128 x d] . Q[V x d]^T, followed by a max over V.
//
// Warp roles in a persistent CTA (one per SM), over 128-token tiles dealt round-robin,
// with E epilogue warpgroups (E = 1, or more when every query column is a score row of its
// own and the epilogue has V times the stores and histogram updates per tile):
//   warp 4E     TMA producer: per tile one mbarrier-completed stage of the 4-stage ring
//               holding the key tile (d/64 boxes of 128 rows x 64 bf16, 128-byte swizzle)
//               and the 16 query rows starting at the tile's first query (same layout);
//   warp 4E+1   MMA issuer: allocates 32E TMEM columns (2E 16-column fp32 accumulators),
//               issues d/16 tcgen05.mma (M = 128 tokens, N = 16 query rows, K = 16) per
//               tile, then commits to the stage's "empty" barrier and the accumulator's
//               "full" barrier;
//   warps 0..4E-1  epilogue, warpgroup e taking tiles i = e mod E: tcgen05.ld of the
//               warp's 32 TMEM lanes (= 32 tokens x 16 columns), which frees the
//               accumulator, then the max over the V real query columns (or, per query,
//               every column to its own score row), coalesced score store and optional
//               fused histogram of the score's top 11 order-key bits.
// Query rows past V (the next group's queries, or zero fill past the end) only produce
// accumulator columns that are never read.  Tokens past N in a tile are never stored.
// Every wait is bounded; a wait that runs out raises an abort flag that the other roles
// see at their next bounded wait, so the CTA drains its copies, frees TMEM and returns.
#include <cudaTypedefs.h>

#include "sd_host.h"
#include "tc_common.cuh"

namespace sd {
namespace {

constexpr int kTileM = 128;   // tokens per tile
constexpr int kQN = 16;       // query rows per MMA (N)
constexpr int kTcStages = 4;
constexpr int kAtomA = kTileM * 128;  // one 64-element K slice of the key tile: 16 KB
constexpr int kAtomB = kQN * 128;     // one 64-element K slice of the query tile: 2 KB

// Epilogue warpgroups: the shared score (max over V) needs one; per-query scores have V
// stores and histogram updates per token.
int tc_epilogue_groups(int V, int per_query) { return !per_query || V == 1 ? 1 : V == 2 ? 2 : 4; }

constexpr int kTcMaxAcc = 8;  // accumulators NB = 2E for up to E = 4 epilogue warpgroups

template <int DI>
struct TcLayout {
    static constexpr int kAtoms = DI / 64;
    static constexpr int kStageA = kAtoms * kAtomA;
    static constexpr int kStageB = kAtoms * kAtomB;
    static constexpr int kStage = kStageA + kStageB;
    static constexpr int oBars = kTcStages * kStage;              // 1024-aligned stages first
    static constexpr int kBars = 2 * kTcStages + 2 * kTcMaxAcc;    // full, empty, tfull[NB], tempty[NB]
    static constexpr int oMisc = oBars + kBars * 8;                // tmem slot, abort flag, consumed
    static constexpr int kBytes = oMisc + 16 + 1024;               // + alignment slack
};

template <int DI, int E>
__global__ void __launch_bounds__(32 * (4 * E + 2), 1) index_score_tc_kernel(
    const __grid_constant__ CUtensorMap kmap, const __grid_constant__ CUtensorMap qmap, int rows,
    int V, int N, float* __restrict__ scores, uint32_t* __restrict__ key_hist, int32_t* err_word, int per_query,
    uint32_t idesc) {
    using L = TcLayout<DI>;
    constexpr int NB = 2 * E;                   // accumulators (16 TMEM columns each)
    static_assert(NB <= kTcMaxAcc, "the barrier block holds tfull and tempty for kTcMaxAcc accumulators");
    constexpr uint32_t kTmemCols = 32u * E;     // a power of two >= 32
    constexpr int kProducer = 4 * E, kIssuer = 4 * E + 1;
    extern __shared__ uint8_t smem_raw[];
    // the 128-byte swizzle layout needs 1024-byte aligned tiles
    const uint32_t raw_addr = smem_addr(smem_raw);
    uint8_t* smem = smem_raw + ((1024u - (raw_addr & 1023u)) & 1023u);
    uint64_t* full = reinterpret_cast<uint64_t*>(smem + L::oBars);
    uint64_t* empty = full + kTcStages;
    uint64_t* tfull = empty + kTcStages;
    uint64_t* tempty = tfull + NB;
    uint32_t* tmem_slot = reinterpret_cast<uint32_t*>(smem + L::oMisc);
    volatile int* abort_flag = reinterpret_cast<volatile int*>(smem + L::oMisc + 4);
    volatile uint32_t* consumed = reinterpret_cast<volatile uint32_t*>(smem + L::oMisc + 8);

    const int tid = threadIdx.x, warp = tid >> 5, lane = tid & 31;
    // tiles dealt round-robin over the CTAs (tile = blockIdx.x + i * gridDim.x): the tiles
    // in flight at any moment are neighbours in memory
    const uint32_t tpr = (uint32_t)((N + kTileM - 1) / kTileM);
    const uint32_t total = (uint32_t)rows * tpr;
    const uint32_t ntiles = blockIdx.x < total ? (total - blockIdx.x + gridDim.x - 1) / gridDim.x : 0u;
    auto tile_pos = [&](uint32_t i, uint32_t& r, uint32_t& t0) {
        const uint32_t t = blockIdx.x + i * gridDim.x;
        r = t / tpr;
        t0 = (t - r * tpr) * kTileM;
    };

    if (tid == 0) {
        for (int s = 0; s < kTcStages; ++s) {
            mbar_init(&full[s], 1);
            mbar_init(&empty[s], 1);
        }
        for (int b = 0; b < NB; ++b) {
            mbar_init(&tfull[b], 1);
            mbar_init(&tempty[b], 4);  // one arrive per epilogue warp
        }
        *abort_flag = 0;
        *consumed = 0;
        fence_mbarrier_init();
    }
    if (warp == kIssuer) tmem_alloc(tmem_slot, kTmemCols);
    tc_fence_before_sync();
    __syncthreads();
    tc_fence_after_sync();
    const uint32_t tmem_base = *tmem_slot;
    pdl_launch_dependents();

    uint32_t issued = 0;
    if (warp == kProducer) {
        if (lane == 0) {
            // keys are read once: evict them first, so the scores written meanwhile stay in L2
            const uint64_t stream_policy = l2_evict_first_policy();
            for (uint32_t i = 0; i < ntiles; ++i) {
                const int s = (int)(i % kTcStages);
                uint32_t r, t0;
                tile_pos(i, r, t0);
                if (!mbar_wait(&empty[s], ((i / kTcStages) & 1u) ^ 1u) || *abort_flag) {
                    *abort_flag = 1;
                    break;
                }
                uint8_t* st = smem + s * L::kStage;
                mbar_arrive_expect_tx(&full[s], L::kStage);
                const int krow = (int)((uint64_t)r * N + t0);
#pragma unroll
                for (int a = 0; a < L::kAtoms; ++a) {
                    tma_load_2d_hint(st + a * kAtomA, &kmap, a * 64, krow, &full[s], stream_policy);
                    tma_load_2d(st + L::kStageA + a * kAtomB, &qmap, a * 64, (int)(r * V), &full[s]);
                }
                ++issued;
            }
        }
    } else if (warp == kIssuer) {
        if (lane == 0) {
            for (uint32_t i = 0; i < ntiles; ++i) {
                const int s = (int)(i % kTcStages);
                const int buf = (int)(i % NB);
                if (!mbar_wait(&full[s], (i / kTcStages) & 1u) ||
                    !mbar_wait(&tempty[buf], ((i / NB) & 1u) ^ 1u) || *abort_flag) {
                    *abort_flag = 1;
                    break;
                }
                tc_fence_after_sync();
                const uint32_t a0 = smem_addr(smem + s * L::kStage);
                const uint32_t b0 = a0 + L::kStageA;
#pragma unroll
                for (int k = 0; k < DI / 16; ++k) {
                    const uint32_t koff = (uint32_t)((k & 3) * 32);
                    const uint64_t ad = umma_desc_k_sw128(a0 + (k >> 2) * kAtomA + koff);
                    const uint64_t bd = umma_desc_k_sw128(b0 + (k >> 2) * kAtomB + koff);
                    umma_bf16(tmem_base + (uint32_t)buf * kQN, ad, bd, idesc, k > 0 ? 1u : 0u);
                }
                umma_commit(&empty[s]);
                umma_commit(&tfull[buf]);
                *consumed = i + 1;
            }
        }
    } else {
        // epilogue: warp w reads TMEM lanes [32q, 32q + 32), q = w mod 4 = tokens t0 + 32q + lane
        const int quarter = warp & 3;
        for (uint32_t i = (uint32_t)(warp >> 2); i < ntiles; i += E) {
            const int buf = (int)(i % NB);
            uint32_t r, t0;
            tile_pos(i, r, t0);
            const bool ok = mbar_wait(&tfull[buf], (i / NB) & 1u);
            if (__any_sync(0xffffffffu, !ok || *abort_flag)) {
                *abort_flag = 1;
                break;
            }
            tc_fence_after_sync();
            float v[16];
            tmem_ld16(tmem_base + ((uint32_t)(quarter * 32) << 16) + (uint32_t)buf * kQN, v);
            // the values are in registers: hand the accumulator back to the MMA issuer
            tc_fence_before_sync();
            __syncwarp();
            if (lane == 0) mbar_arrive(&tempty[buf]);
            const uint32_t tok = t0 + (uint32_t)(quarter * 32 + lane);
            const bool store = tok < (uint32_t)N;
            auto put = [&](uint32_t srow, float x) {  // score row srow: store, histogram
                if (store) scores[(size_t)srow * N + tok] = x;
                if (key_hist != nullptr) {
                    const uint32_t dg = float_key(x) >> 21;
                    const uint32_t peers = __match_any_sync(0xffffffffu, store ? dg : 0xffffffffu);
                    if (store && lane == __ffs(peers) - 1)
                        atomicAdd(&key_hist[(size_t)srow * 2048 + dg], (uint32_t)__popc(peers));
                }
            };
            if (per_query) {
#pragma unroll
                for (int j = 0; j < 16; ++j)
                    if (j < V) put(r * (uint32_t)V + (uint32_t)j, v[j]);
            } else {
                float best = v[0];
#pragma unroll
                for (int j = 1; j < 16; ++j)
                    if (j < V) best = fmaxf(best, v[j]);
                put(r, best);
            }
        }
    }
    __syncthreads();
    if (tid == 0 && *abort_flag) {
        report(err_word, SD_DEVERR_TIMEOUT);
        // let the stages the producer filled but no MMA consumed land before exiting
        for (uint32_t j = *consumed; j < issued; ++j) mbar_wait(&full[j % kTcStages], (j / kTcStages) & 1u);
    }
    __syncthreads();
    if (warp == kIssuer) {
        tc_fence_after_sync();
        tmem_dealloc(tmem_base, kTmemCols);
    }
}

}  // namespace

static PFN_cuTensorMapEncodeTiled_v12000 encode_fn() {
    static PFN_cuTensorMapEncodeTiled_v12000 fn = nullptr;
    if (fn == nullptr) {
        void* p = nullptr;
        cudaDriverEntryPointQueryResult q{};
        if (cudaGetDriverEntryPointByVersion("cuTensorMapEncodeTiled", &p, 12000, cudaEnableDefault, &q) ==
                cudaSuccess &&
            q == cudaDriverEntryPointSuccess)
            fn = reinterpret_cast<PFN_cuTensorMapEncodeTiled_v12000>(p);
    }
    return fn;
}

// 2-D tensor map of 16-bit elements (bf16 or fp16) over [nrows, d] (row-major), box = 64
// columns x box_rows rows, 128-byte swizzle, zero fill outside the tensor.
bool make_tensor_map_2d(CUtensorMap* m, const void* base, uint64_t nrows, int d, int box_rows, bool f16) {
    auto fn = encode_fn();
    if (fn == nullptr) return false;
    cuuint64_t dims[2] = {(cuuint64_t)d, (cuuint64_t)nrows};
    cuuint64_t strides[1] = {(cuuint64_t)d * 2};
    cuuint32_t box[2] = {64, (cuuint32_t)box_rows};
    cuuint32_t estr[2] = {1, 1};
    CUresult r = fn(m, f16 ? CU_TENSOR_MAP_DATA_TYPE_FLOAT16 : CU_TENSOR_MAP_DATA_TYPE_BFLOAT16, 2,
                    const_cast<void*>(base), dims, strides, box, estr,
                    CU_TENSOR_MAP_INTERLEAVE_NONE, CU_TENSOR_MAP_SWIZZLE_128B, CU_TENSOR_MAP_L2_PROMOTION_L2_256B,
                    CU_TENSOR_MAP_FLOAT_OOB_FILL_NONE);
    return r == CUDA_SUCCESS;
}

// bf16 (or fp16) keys and queries of the same type on the tensor cores; d_idx in {64, 128},
// V <= 16.  per_query: every query row gets its own score row (rows*V of them) instead of
// the max over V.
sd_status index_score_tc_launch(const void* q_idx, const void* k_idx, int rows, int V, int N, int d_idx,
                                float* scores, uint32_t* key_hist, int32_t* err_word, int per_query, bool f16, cudaStream_t st) {
    CUtensorMap kmap, qmap;
    if (!make_tensor_map_2d(&kmap, k_idx, (uint64_t)rows * N, d_idx, kTileM, f16) ||
        !make_tensor_map_2d(&qmap, q_idx, (uint64_t)rows * V, d_idx, kQN, f16)) {
        set_error("sd_index_score: cuTensorMapEncodeTiled failed");
        return SD_ERR_CUDA;
    }
    const uint32_t tpr = (uint32_t)((N + kTileM - 1) / kTileM);
    const long tiles = (long)rows * tpr;
    const unsigned grid = (unsigned)std::min<long>(tiles, (long)num_sms());
    const int E = tc_epilogue_groups(V, per_query);
    const bool d128 = d_idx == 128;
    auto kern = d128 ? (E == 1 ? index_score_tc_kernel<128, 1> : E == 2 ? index_score_tc_kernel<128, 2>
                                                                        : index_score_tc_kernel<128, 4>)
                     : (E == 1 ? index_score_tc_kernel<64, 1> : E == 2 ? index_score_tc_kernel<64, 2>
                                                                       : index_score_tc_kernel<64, 4>);
    const int bytes = d128 ? TcLayout<128>::kBytes : TcLayout<64>::kBytes;
    SD_CUDA_CHECK(cudaFuncSetAttribute(kern, cudaFuncAttributeMaxDynamicSharedMemorySize, bytes),
                  "sd_index_score: cudaFuncSetAttribute");
    const uint32_t idesc = f16 ? umma_idesc_f16_f32(kTileM, kQN) : umma_idesc_bf16_f32(kTileM, kQN);
    kern<<<grid, 32 * (4 * E + 2), bytes, st>>>(kmap, qmap, rows, V, N, scores, key_hist, err_word, per_query, idesc);
    return launch_status("sd_index_score (tensor cores)");
}

}  // namespace sd
