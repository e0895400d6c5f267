// dense_attend.cu -- sd_gather_attend's path for attention over a cache resident in HBM
// read as whole tiles: every one of the T rows of each KV group (the per-layer step of
// importance scoring, which keeps every logit), or the rows of selected blocks of 16 or more
// rows (block-sparse selection; compression windows as 16-token segments); bf16, d = 128, at
// most 16 query rows per group.
//
// "Nem Todos os Pensamentos Necessitam de HBM" (gist.science summary), Metodologia 2: the
// importance of a position accumulates the attention weight every query head gives it, so
// each layer attends densely and keeps its logits.  "Esparsidade de Contexto no Tempo de
// Inferencia" (gist.science summary), sec. 2: exact softmax attention.  Adaptive DHiSparse
// (news page), "Metodologia": the query rows of a group share each fetched row.
//
// The rows of a group are contiguous, so they move as whole tiles: CTA (split, kvh, b)
// streams its contiguous range of the group's rows (or of its list of selected rows, whose
// 16-row sub-tiles are contiguous in the cache and are resolved once into shared memory)
// through a two-stage ring of 64-row
// stages (tiled TMA, 128-byte swizzle; warp 4 issues the copies), and consumer warps 0-3
// take the 32-row halves of the stages (stage n to warps 2(n % 2) and 2(n % 2) + 1) with the
// transposed mma.sync tile of step_tiles.cuh, each keeping its own online softmax over all
// query rows.  The four warps' states merge into the CTA's (m, l, O): with one split that is
// the output; with several it is the split's partial in sd_gather_attend's workspace, which
// its merge kernel combines.  Every mbarrier wait is bounded; a wait that runs out sets
// SD_DEVERR_TIMEOUT, and the CTA lets its copies in flight land before it exits.
#include <algorithm>
#include <cmath>

#include "sd_host.h"
#include "step_tiles.cuh"
#include "tc_common.cuh"

namespace sd {
namespace {

constexpr int kDaCons = 4;                  // consumer warps 0-3
constexpr int kDaProd = kDaCons;            // producer warp 4
constexpr int kDaThreads = 32 * (kDaCons + 1);
constexpr int kDaSlot = 32768;              // a ring stage: 64 K rows and 64 V rows
constexpr int kDaRows = 64;                 // rows per stage
constexpr int kDaRing = 2;                  // stages (stage n in slot n % 2, taken by pair n % 2)
constexpr int kDaQ = kDaRing * kDaSlot;     // query rows: 16 x 256 bytes
constexpr int kDaBars = kDaQ + 16 * 256;    // full[2], empty[2], q
constexpr int kDaMisc = kDaBars + 64;       // the abort flag
constexpr int kDaMaxSub = 1024;             // 16-row sub-tiles a split of a block-sparse call covers
constexpr int kDaYs = kDaMisc + 16;         // their first rows in the cache, or -1: [kDaMaxSub] int32
constexpr int kDaBytes = kDaYs + kDaMaxSub * 4 + 1024;  // slack for the 1024-byte alignment of the ring
// after the loop, in the ring: the warps' O rows [4][16][128] floats, then their (m, l) [4][16]
constexpr int kDaPartML = kDaCons * 16 * 128 * 4;
static_assert(kDaPartML + kDaCons * 16 * 8 <= kDaRing * kDaSlot, "the warps' states fit in the ring");

struct DaParams {
    const uint8_t* q;  // [B, V, Hq, 128] bf16
    float* out;        // [B, V, Hq, 128]
    float* lse;        // [B, V, Hq]
    float* logits;     // [B, V, Hq, T] or null
    int32_t* err;
    float* ws_o;       // with splits > 1: [B*Hkv][splits][RP][128], then m and l [..][RP]
    float* ws_m;
    float* ws_l;
    const int32_t* idx;  // block-sparse: [B*Hkv][n_idx] selected blocks, else null (dense)
    int n_idx, block;
    int n_rows;          // rows of a group's list: n_idx * block (T when dense)
    int total_rows;      // rows of the cache tensor (B*Hkv*T): a coordinate past them loads zeros
    int V, Hq, Hkv, G, R, T, rps, splits, RP;
    float scale_log2;
    unsigned long long wait_ns;
};

// Writes a logit (base 2 in, natural log out) of query row qc and key `key` of the 32-row
// half at row t0 of the group; keys outside the valid mask never reach it.
struct DaLogits {
    float* base;  // logits of (b, v = 0, head kvh*G), or null
    int G, R, Hq, T, t0;
    SD_DEVINL void operator()(int qc, int key, float x) const {
        if (base == nullptr || qc >= R) return;
        const int v = qc / G, gi = qc - v * G;
        base[((size_t)v * Hq + gi) * T + t0 + key] = x * 0.69314718055994530942f;
    }
};

// CTAs per SM: three with one query tile (128 registers a thread), two with two
template <int NQ>
__global__ void __launch_bounds__(kDaThreads, NQ == 1 ? 3 : 2)
    dense_attend_kernel(const __grid_constant__ CUtensorMap kvk, const __grid_constant__ CUtensorMap kvv,
                        const DaParams p) {
    extern __shared__ uint8_t smem_raw[];
    const uint32_t raw = smem_addr(smem_raw);
    uint8_t* sm = smem_raw + ((1024u - (raw & 1023u)) & 1023u);
    const int split = (int)blockIdx.x, kvh = (int)blockIdx.y, b = (int)blockIdx.z;
    const int g = b * p.Hkv + kvh;
    const int tid = threadIdx.x, warp = tid >> 5, lane = tid & 31;
    uint64_t* full = reinterpret_cast<uint64_t*>(sm + kDaBars);
    uint64_t* empty = full + kDaRing;
    uint64_t* qbar = empty + kDaRing;
    volatile int* abort_flag = reinterpret_cast<volatile int*>(sm + kDaMisc);
    const uint32_t ring = smem_addr(sm);
    const uint64_t lim = p.wait_ns;

    if (tid == 0) {
        for (int s = 0; s < kDaRing; ++s) {
            mbar_init(&full[s], 1);   // the producer's arrival with the stage's bytes
            mbar_init(&empty[s], 2);  // the two consumer warps of the stage
        }
        mbar_init(qbar, 1);
        *abort_flag = 0;
        fence_mbarrier_init();
    }
    __syncthreads();
    pdl_wait();  // q and the cache may be the preceding kernels' results

    const int t0 = split * p.rps, n_rows = max(0, min(p.n_rows, t0 + p.rps) - t0);
    const int n_st = (n_rows + kDaRows - 1) / kDaRows;
    // block-sparse: the split's 16-row sub-tiles (one block holds whole sub-tiles) resolved to
    // their first cache row, or -1 for an empty slot (-1) or a bad index (reported)
    const int32_t* ys = reinterpret_cast<const int32_t*>(sm + kDaYs);
    const int n_sub = (n_rows + 15) / 16;
    if (p.idx != nullptr) {
        int32_t* yw = reinterpret_cast<int32_t*>(sm + kDaYs);
        for (int i = tid; i < n_sub; i += kDaThreads) {
            const int j0 = t0 + 16 * i;
            const long sel = p.idx[(size_t)g * p.n_idx + j0 / p.block];
            const long pos = sel * p.block + j0 % p.block;
            int32_t y = -1;
            if (sel == -1) {
                // empty slot
            } else if (sel < 0 || pos >= p.T) {
                report(p.err, SD_DEVERR_INDEX);
            } else {
                y = (int32_t)((long)g * p.T + pos);
            }
            yw[i] = y;
        }
        __syncthreads();
    }
    int n_issued = 0;  // stages the producer filled (its lane 0)
    AttAccT<NQ> acc;
    if (warp == kDaProd) {
        if (lane == 0) {
            // the query rows v*G + gi: each verify query's G heads are contiguous
            const uint32_t gb = (uint32_t)p.G * 256u;
            mbar_arrive_expect_tx(qbar, (uint32_t)p.V * gb);
            for (int v = 0; v < p.V; ++v)
                bulk_g2s(sm + kDaQ + v * gb, p.q + (((size_t)b * p.V + v) * p.Hq + (size_t)kvh * p.G) * 256, gb, qbar);
            const uint64_t pol = l2_evict_first_policy();  // the rows are read once
            for (int n = 0; n < n_st; ++n) {
                const int s = n % kDaRing;
                if (n >= kDaRing && !ds_wait(&empty[s], (uint32_t)((n / kDaRing - 1) & 1), abort_flag, lim)) {
                    *abort_flag = 1;
                    break;
                }
                uint8_t* st = sm + s * kDaSlot;
                mbar_arrive_expect_tx(&full[s], kDaSlot);
                if (p.idx == nullptr) {
                    // rows past the group's end load the next group's rows (or the tensor's
                    // fill) and are masked out
                    const int row = g * p.T + t0 + n * kDaRows;
#pragma unroll
                    for (int h = 0; h < 2; ++h) {
                        uint8_t* dk = st + h * 16384;
                        tma_load_2d_hint(dk, &kvk, 0, row + 32 * h, &full[s], pol);
                        tma_load_2d_hint(dk + 4096, &kvk, 64, row + 32 * h, &full[s], pol);
                        tma_load_2d_hint(dk + 8192, &kvv, 0, row + 32 * h, &full[s], pol);
                        tma_load_2d_hint(dk + 12288, &kvv, 64, row + 32 * h, &full[s], pol);
                    }
                } else {
                    // four 16-row boxes per stage, each where its sub-tile's rows are; a
                    // sub-tile without rows loads past the tensor (zeros) and is masked out.
                    // Two 16-row boxes 2 KB apart land as one 32-row box would (swizzle atoms
                    // of 8 rows, every box 1024-byte aligned).
#pragma unroll
                    for (int q = 0; q < 4; ++q) {
                        const int i = 4 * n + q;
                        const int y0 = i < n_sub ? ys[i] : -1;
                        const int y = y0 >= 0 ? y0 : p.total_rows;
                        uint8_t* dk = st + (q >> 1) * 16384 + (q & 1) * 2048;
                        tma_load_2d_hint(dk, &kvk, 0, y, &full[s], pol);
                        tma_load_2d_hint(dk + 4096, &kvk, 64, y, &full[s], pol);
                        tma_load_2d_hint(dk + 8192, &kvv, 0, y, &full[s], pol);
                        tma_load_2d_hint(dk + 12288, &kvv, 64, y, &full[s], pol);
                    }
                }
                n_issued = n + 1;
            }
        }
    } else {
        // zero the padding query rows R .. 8*NQ - 1, then wait for the copied ones
        for (int i = tid; i < (8 * NQ - p.R) * 16; i += 32 * kDaCons)
            reinterpret_cast<uint4*>(sm + kDaQ + p.R * 256)[i] = make_uint4(0u, 0u, 0u, 0u);
        warp_wait(qbar, 0u, abort_flag, lim);
        asm volatile("bar.sync 1, %0;" ::"n"(32 * kDaCons) : "memory");
        att_init_t(acc);
        uint32_t qf[8][NQ][2];
        load_q_frags_t<NQ>(smem_addr(sm + kDaQ), lane, qf);
        const int h = warp & 1;
        DaLogits lg{nullptr, p.G, p.R, p.Hq, p.T, 0};
        if (p.logits != nullptr) lg.base = p.logits + ((size_t)b * p.V * p.Hq + (size_t)kvh * p.G) * p.T;
        for (int n = (warp >> 1); n < n_st; n += 2) {
            if (*abort_flag) break;
            const int s = n % kDaRing;
            if (!warp_wait(&full[s], (uint32_t)((n / kDaRing) & 1), abort_flag, lim)) break;
            const int jb = n * kDaRows + 32 * h;  // this half's first row in the CTA's range
            const int nv = max(0, min(32, n_rows - jb));
            uint32_t valid = nv >= 32 ? 0xffffffffu : ((1u << nv) - 1u);
            if (p.idx != nullptr) {  // the half's two sub-tiles
                const int i0 = 4 * n + 2 * h;
                valid &= ((i0 < n_sub && ys[i0] >= 0) ? 0x0000ffffu : 0u) |
                         ((i0 + 1 < n_sub && ys[i0 + 1] >= 0) ? 0xffff0000u : 0u);
            }
            const uint32_t kb = ring + s * kDaSlot + h * 16384;
            lg.t0 = t0 + jb;
            if (valid != 0u) attend_stage_t<NQ>(kb, kb + 8192, lane, qf, valid, p.scale_log2, acc, lg);
            __syncwarp();
            if (lane == 0) mbar_arrive(&empty[s]);
        }
    }
    __syncthreads();
    if (tid == 32 * kDaProd && *abort_flag) {
        // let every stage issued but not consumed land before the ring is reused
        for (int n = max(0, n_issued - kDaRing); n < n_issued; ++n)
            mbar_wait(&full[n % kDaRing], (uint32_t)((n / kDaRing) & 1), lim);
        mbar_wait(qbar, 0u, lim);
    }
    pdl_launch_dependents();
    __syncthreads();

    // the four warps' states into the CTA's (m, l, O), one (query row, 4 columns) item per thread
    float* wo = reinterpret_cast<float*>(sm);                  // [4][16][128]
    float2* wml = reinterpret_cast<float2*>(sm + kDaPartML);  // [4][16]
    if (warp < kDaCons) {  // O^T fragments: column 16md + g8 (+8) of query row 8nq + 2t4 + e
        const int g8 = lane >> 2, t4 = lane & 3;
#pragma unroll
        for (int nq = 0; nq < NQ; ++nq)
#pragma unroll
            for (int e = 0; e < 2; ++e) {
                const int row = 8 * nq + 2 * t4 + e;
                if (row >= p.R) continue;
#pragma unroll
                for (int md = 0; md < 8; ++md) {
                    wo[(warp * 16 + row) * 128 + 16 * md + g8] = acc.o[md][nq][e];
                    wo[(warp * 16 + row) * 128 + 16 * md + g8 + 8] = acc.o[md][nq][2 + e];
                }
                if (g8 == 0) wml[warp * 16 + row] = make_float2(acc.m[nq][e], acc.l[nq][e]);
            }
    }
    __syncthreads();
    for (int i = tid; i < p.R * 32; i += kDaThreads) {
        const int row = i >> 5, c4 = i & 31;
        float2 ml[kDaCons];
        float4 o[kDaCons];
#pragma unroll
        for (int w = 0; w < kDaCons; ++w) {
            ml[w] = wml[w * 16 + row];
            o[w] = reinterpret_cast<const float4*>(wo + (w * 16 + row) * 128)[c4];
        }
        float M = -INFINITY;
#pragma unroll
        for (int w = 0; w < kDaCons; ++w) M = fmaxf(M, ml[w].x);
        float L = 0.f;
        float4 O = make_float4(0.f, 0.f, 0.f, 0.f);
#pragma unroll
        for (int w = 0; w < kDaCons; ++w) {
            const float f = ml[w].x == -INFINITY ? 0.f : exp2f(ml[w].x - M);
            L = fmaf(ml[w].y, f, L);
            O.x = fmaf(o[w].x, f, O.x);
            O.y = fmaf(o[w].y, f, O.y);
            O.z = fmaf(o[w].z, f, O.z);
            O.w = fmaf(o[w].w, f, O.w);
        }
        if (p.splits == 1) {
            const int v = row / p.G, gi = row % p.G;
            const size_t qrow = ((size_t)b * p.V + v) * p.Hq + (size_t)kvh * p.G + gi;
            const float inv = L > 0.f ? 1.f / L : 0.f;
            reinterpret_cast<float4*>(p.out + qrow * 128)[c4] = make_float4(O.x * inv, O.y * inv, O.z * inv, O.w * inv);
            if (c4 == 0) p.lse[qrow] = L > 0.f ? (M + log2f(L)) * 0.69314718055994530942f : -INFINITY;
        } else {
            const size_t prow = ((size_t)g * p.splits + split) * p.RP + row;
            reinterpret_cast<float4*>(p.ws_o + prow * 128)[c4] = O;
            if (c4 == 0) {
                p.ws_m[prow] = M;
                p.ws_l[prow] = L;
            }
        }
    }
    if (tid == 0 && *abort_flag) report(p.err, SD_DEVERR_TIMEOUT);
}

}  // namespace

int dense_tma_ctas_per_sm(const sd_attend_args* a) { return (a->Hq / a->Hkv) * a->V <= 8 ? 3 : 2; }

int dense_tma_max_split_rows() { return kDaMaxSub * 16; }

bool dense_tma_eligible(const sd_attend_args* a) {
    const int R = (a->Hq / a->Hkv) * a->V;
    const bool common = a->slot_map == nullptr && a->ring_w == 0 && !a->per_head && a->tier == nullptr &&
                        a->k_stage == nullptr && a->row_loop == 0 && a->dtype == SD_BF16 && a->d == 128 && R >= 1 &&
                        R <= 16 && a->T > 0 && (long)a->B * a->Hkv * a->T < (1L << 31);
    if (!common) return false;
    if (a->idx == nullptr) return (long)a->n_idx * a->block == a->T;
    // block-sparse: whole 16-row sub-tiles per block, whole blocks per cache, and no logits
    // (the row loop defines those of empty slots)
    return a->logits == nullptr && a->n_idx > 0 && a->block % 16 == 0 && a->T % a->block == 0;
}

sd_status dense_tma_launch(const sd_attend_args* a, int max_splits, int RP, float* ws_o, float* ws_m, float* ws_l,
                           int* splits_used, cudaStream_t st) {
    const char* who = "sd_gather_attend";
    const int NG = a->B * a->Hkv;
    const bool sparse = a->idx != nullptr;
    const int n_rows = sparse ? a->n_idx * a->block : a->T;  // a group's list rows
    // contiguous ranges of whole 64-row stages, no more splits than the workspace holds and,
    // unless the caller asked for a count, one wave of CTAs; a block-sparse range at most
    // kDaMaxSub sub-tiles (the plan's splits are at most that long, so they still fit)
    int S0 = std::max(1, max_splits);
    if (a->splits <= 0 && NG > 0) S0 = std::min(S0, std::max(1, dense_tma_ctas_per_sm(a) * num_sms() / NG));
    int rps = (n_rows + S0 - 1) / S0;
    rps = (rps + kDaRows - 1) / kDaRows * kDaRows;
    if (sparse) rps = std::min(rps, kDaMaxSub * 16);
    const int S = (n_rows + rps - 1) / rps;
    if (S > std::max(1, max_splits)) {
        set_error("%s: %d splits exceed the workspace's %d", who, S, max_splits);
        return SD_ERR_INVALID_ARG;
    }
    *splits_used = S;
    const int box_rows = sparse ? 16 : 32;
    CUtensorMap kvk, kvv;
    if (!make_tensor_map_2d(&kvk, a->k_cache, (uint64_t)NG * a->T, 128, box_rows, false) ||
        !make_tensor_map_2d(&kvv, a->v_cache, (uint64_t)NG * a->T, 128, box_rows, false)) {
        set_error("%s: cuTensorMapEncodeTiled failed", who);
        return SD_ERR_CUDA;
    }
    DaParams p{};
    p.q = static_cast<const uint8_t*>(a->q);
    p.out = a->out;
    p.lse = a->lse;
    p.logits = a->logits;
    p.err = a->err_word;
    p.ws_o = ws_o;
    p.ws_m = ws_m;
    p.ws_l = ws_l;
    p.idx = a->idx;
    p.n_idx = a->n_idx;
    p.block = a->block;
    p.n_rows = n_rows;
    p.total_rows = NG * a->T;
    p.V = a->V;
    p.Hq = a->Hq;
    p.Hkv = a->Hkv;
    p.G = a->Hq / a->Hkv;
    p.R = p.G * a->V;
    p.T = a->T;
    p.rps = rps;
    p.splits = S;
    p.RP = RP;
    p.scale_log2 = a->scale * 1.44269504088896340736f;
    p.wait_ns = (unsigned long long)kWaitDeadlineNs;
    auto kern = p.R <= 8 ? dense_attend_kernel<1> : dense_attend_kernel<2>;
    SD_CUDA_CHECK(cudaFuncSetAttribute(kern, cudaFuncAttributeMaxDynamicSharedMemorySize, kDaBytes),
                  "sd_gather_attend: cudaFuncSetAttribute");
    SD_CUDA_CHECK(launch_pdl(kern, dim3((unsigned)S, (unsigned)a->Hkv, (unsigned)a->B), dim3(kDaThreads), kDaBytes, st,
                             kvk, kvv, p),
                  "sd_gather_attend: launch");
    return launch_status(who);
}

}  // namespace sd
