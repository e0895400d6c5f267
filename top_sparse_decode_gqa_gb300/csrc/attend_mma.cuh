// attend_mma.cuh -- the per-warp exact-attention loop on the warp-level tensor cores
// (mma.sync m16n8k16, bf16 in, fp32 accumulate), shared by sd_gather_attend and the
// fused select + attend kernel.
//
// "Esparsidade de Contexto no Tempo de Inferencia" (gist.science summary), sec. 2: sparse
// decode attention over an irregular per-token selection; Adaptive DHiSparse (news page),
// "Metodologia": every query row of a group shares each fetched row.
//
// A CTA of NW warps owns a list of `nrows` K/V rows.  The list is cut into 16-row
// sub-chunks dealt round-robin to the warps; each warp runs its own NS-deep cp.async
// pipeline (8 lanes move one 128-byte line of a row, 4 rows per instruction) and
// its own online softmax in base 2 over all RP query rows: S[16q x 8k] tiles from Q and K
// through ldmatrix, P split into bf16 hi + lo parts so the PV product keeps ~16
// significant bits, V fragments through ldmatrix.trans.  mma_combine_warps then merges
// the NW warps' (m, l, O) in shared memory.
#pragma once

#include <stdint.h>

#include "sd_common.cuh"

namespace sd {

constexpr int kMmaWarps = 4;          // warps of a CTA that run the attention loop (default)
constexpr int kSub = 16;              // rows per warp sub-chunk
constexpr int kWStages = 2;           // sub-chunks in flight per warp (default)
constexpr int32_t kNoRow = INT32_MIN;  // source code of a skipped row (contributes nothing)
constexpr int32_t kRingBase = 1 << 30;  // codes >= this: slot code - kRingBase of the draft ring
constexpr int32_t kI8Base = 1 << 29;    // codes in [kI8Base, kRingBase): int8 row code - kI8Base
constexpr float kLn2f = 0.69314718055994530942f;

template <int D, int NW = kMmaWarps, int NS = kWStages>
struct MmaRows {
    static constexpr int kRowB = D * 2 + 16;         // padded bf16 row: conflict-free ldmatrix
    static constexpr int kStage = 2 * kSub * kRowB;  // K rows then V rows
    static constexpr int kWarpBytes = NS * kStage;
    static constexpr int kStagesBytes = NW * kWarpBytes;
};

// cp.async.wait_group with a run-time count below NS (the instruction takes an immediate).
template <int NS>
SD_DEVINL void cp_async_wait_dyn(int n) {
    if constexpr (NS > 3) {
        if (n >= 3) { cp_async_wait<3>(); return; }
    }
    if constexpr (NS > 2) {
        if (n == 2) { cp_async_wait<2>(); return; }
    }
    if (n >= 1) cp_async_wait<1>();
    else cp_async_wait<0>();
}

// Where a row's bytes are: code >= kRingBase is slot code - kRingBase of the draft ring
// (k_ring + slot * row bytes, offset to this (b, kvh)); with int8 rows (SmemScales), code in
// [kI8Base, kRingBase) is int8 row code - kI8Base (k_i8 + row * d); other code >= 0 is row `code` of the
// device pool (k_pool + code * row bytes, likewise offset); code < 0 is host row -1 - code
// of the mapped host cache (k_host likewise offset); kNoRow is skipped.
struct RowSource {
    const uint8_t* k_pool;
    const uint8_t* v_pool;
    const uint8_t* k_host;
    const uint8_t* v_host;
    const uint8_t* k_ring = nullptr;
    const uint8_t* v_ring = nullptr;
    const int8_t* k_i8 = nullptr;  // int8 rows (codes), offset to this (b, kvh) like the pool
    const int8_t* v_i8 = nullptr;
    const float* k_scl = nullptr;  // their per-row scales, likewise offset
    const float* v_scl = nullptr;
};

// Whether the list holds int8 rows (the loop then widens their codes to bf16 in shared
// memory and keeps every row's scale in its slot's pad: 1 for rows at full precision).
struct NoScales {
    static constexpr bool kInt8 = false;
};
struct Int8Rows {
    static constexpr bool kInt8 = true;
};

// Visibility of list row j to query row r when every row is visible to every query.
struct AllVisible {
    SD_DEVINL bool operator()(int, int) const { return true; }
};

template <int D, int RP>
struct WarpAcc {
    static constexpr int MT = RP / 16;  // 16-row M tiles of query rows
    static constexpr int NT = D / 8;    // 8-column n-tiles of PV
    float m[MT][2], l[MT][2];
    float o[MT][NT][4];
    SD_DEVINL void init() {
#pragma unroll
        for (int mt = 0; mt < MT; ++mt) {
            m[mt][0] = m[mt][1] = -INFINITY;
            l[mt][0] = l[mt][1] = 0.f;
#pragma unroll
            for (int nt = 0; nt < NT; ++nt)
#pragma unroll
                for (int e = 0; e < 4; ++e) o[mt][nt][e] = 0.f;
        }
    }
};

// One warp's share of the CTA's rows.  `stages` is this warp's kWarpBytes of shared
// memory, `q_base` the shared address of the RP query rows (kRowB apart, pre-loaded, rows
// beyond the real ones zero).  row_code(j) returns the source of list row j (kNoRow for a
// skipped row; called only for j < nrows).  logit(r, j, x) receives every (query row,
// list row) score in base-2 units (x * ln 2 is the natural logit) of valid rows, -inf where
// vis(r, j) hides the row from the query row (the causal mask of the draft ring).
// nq = the real query rows (<= RP): an upper half tile (rows 8..15 of an M tile) holding
// none of them skips its softmax, and its P fragments are zero.
// Scl: NoScales, or Int8Rows with int8 rows: a row's codes are copied into the upper half of
// its bf16 slot and widened in place before use, and its scale into the slot's 16-byte pad
// (the pad of full-precision rows holds 1); the K scale multiplies the row's logits and the
// V scale its softmax weights in the PV product.
template <int D, int RP, int NW = kMmaWarps, int NS = kWStages, class RowCode, class Logit, class Vis = AllVisible,
          class Scl = NoScales>
SD_DEVINL void mma_attend_warp(WarpAcc<D, RP>& acc, uint8_t* stages, uint32_t q_base, int warp, int nrows, int nq,
                               const RowSource& rs, float scale_log2, RowCode row_code, Logit logit,
                               Vis vis = Vis(), Scl scl = Scl()) {
    static_assert(!Scl::kInt8 || D == 128, "int8 rows: d = 128 (one 128-byte line per row)");
    static_assert(NS >= 2 && NS <= 4, "2 to 4 stages per warp");
    using L = MmaRows<D, NW, NS>;
    constexpr int MT = RP / 16, KS = D / 16, NT = D / 8;
    constexpr int PPR = D * 2 / 16;  // 16-byte pieces per row
    const int lane = threadIdx.x & 31;
    const int g = lane >> 2, t4 = lane & 3;
    auto code_of = [&](int j) -> int32_t { return j < nrows ? row_code(j) : kNoRow; };
    const int nsub = (nrows + kSub - 1) / kSub;
    const int my_n = warp < nsub ? (nsub - warp + NW - 1) / NW : 0;

    // Lanes 8q..8q+7 move one 128-byte line of a row per instruction (4 rows at a time), so
    // every request is a whole line, in HBM and over the host link alike.
    auto issue = [&](int ci, int st) {
        const int c = warp + NW * ci;
        uint8_t* kst = stages + st * L::kStage;
        const int sub = lane >> 3, piece = lane & 7;
        int32_t code[kSub / 4];
#pragma unroll
        for (int q = 0; q < kSub / 4; ++q) code[q] = code_of(c * kSub + q * 4 + sub);
#pragma unroll
        for (int which = 0; which < 2; ++which)
#pragma unroll
            for (int q = 0; q < kSub / 4; ++q) {
                uint8_t* dst = kst + which * kSub * L::kRowB + (q * 4 + sub) * L::kRowB + piece * 16;
                if constexpr (Scl::kInt8) {
                    float* pad = reinterpret_cast<float*>(dst - piece * 16 + 2 * D);
                    if (code[q] >= kI8Base && code[q] < kRingBase) {  // one 128-byte line of codes
                        const int8_t* srow = (which ? rs.v_i8 : rs.k_i8) + (size_t)(code[q] - kI8Base) * D;
                        cp_async16(dst + D, srow + piece * 16);
                        if (piece == 0) cp_async4(pad, (which ? rs.v_scl : rs.k_scl) + (code[q] - kI8Base));
                        continue;
                    }
                    if (piece == 0) *pad = 1.f;
                }
                if (code[q] == kNoRow) {
#pragma unroll
                    for (int h = 0; h < PPR / 8; ++h) *reinterpret_cast<uint4*>(dst + h * 128) = make_uint4(0u, 0u, 0u, 0u);
                } else {
                    const uint8_t* srow = code[q] >= kRingBase
                        ? (which ? rs.v_ring : rs.k_ring) + (size_t)(code[q] - kRingBase) * (D * 2)
                        : code[q] >= 0
                        ? (which ? rs.v_pool : rs.k_pool) + (size_t)code[q] * (D * 2)
                        : (which ? rs.v_host : rs.k_host) + (size_t)(-1 - (long)code[q]) * (D * 2);
                    srow += piece * 16;
#pragma unroll
                    for (int h = 0; h < PPR / 8; ++h) cp_async16(dst + h * 128, srow + h * 128);
                }
            }
        cp_async_commit();
    };

    int issued = 0;
    for (; issued < min(NS, my_n); ++issued) issue(issued, issued);
    for (int ci = 0; ci < my_n; ++ci) {
        const int st = ci % NS;
        cp_async_wait_dyn<NS>(issued - ci - 1);  // chunk ci has landed; later ones may still fly
        __syncwarp();
        const uint32_t k_base = smem_addr(stages + st * L::kStage);
        const uint32_t v_base = k_base + kSub * L::kRowB;
        const int c = warp + NW * ci;
        // with int8 rows: the chunk's row codes, one per lane (lanes 16..31 none)
        int32_t my_code = kNoRow;
        if constexpr (Scl::kInt8) my_code = lane < kSub ? code_of(c * kSub + lane) : kNoRow;
        if constexpr (Scl::kInt8) {
            // widen the chunk's int8 rows in place: lane l reads codes 4l .. 4l + 3 of the K and
            // the V row (upper half of their slots), and after the whole warp has read, writes
            // their bf16 values at elements 4l .. 4l + 3 (small integers are exact in bf16)
            uint32_t i8 = __ballot_sync(0xffffffffu, my_code >= kI8Base && my_code < kRingBase);
            while (i8 != 0u) {
                const int r = __ffs(i8) - 1;
                i8 &= i8 - 1u;
                uint8_t* krow = stages + st * L::kStage + r * L::kRowB;
                uint8_t* vrow = krow + kSub * L::kRowB;
                const uint32_t wk = *reinterpret_cast<const uint32_t*>(krow + D + 4 * lane);
                const uint32_t wv = *reinterpret_cast<const uint32_t*>(vrow + D + 4 * lane);
                __syncwarp();
                *reinterpret_cast<uint2*>(krow + 8 * lane) =
                    make_uint2(pack_bf16x2((float)(int8_t)(wk & 0xffu), (float)(int8_t)((wk >> 8) & 0xffu)),
                               pack_bf16x2((float)(int8_t)((wk >> 16) & 0xffu), (float)(int8_t)(wk >> 24)));
                *reinterpret_cast<uint2*>(vrow + 8 * lane) =
                    make_uint2(pack_bf16x2((float)(int8_t)(wv & 0xffu), (float)(int8_t)((wv >> 8) & 0xffu)),
                               pack_bf16x2((float)(int8_t)((wv >> 16) & 0xffu), (float)(int8_t)(wv >> 24)));
            }
            __syncwarp();
        }

        // ---- S = Q K^T for this warp's 16 rows: [MT][2 n-tiles][4].  Even and odd k-steps
        // accumulate separately (4 independent MMA chains per M tile), then add.
        float sacc[MT][2][4], sodd[MT][2][4];
#pragma unroll
        for (int mt = 0; mt < MT; ++mt)
#pragma unroll
            for (int nt = 0; nt < 2; ++nt)
#pragma unroll
                for (int e = 0; e < 4; ++e) sacc[mt][nt][e] = sodd[mt][nt][e] = 0.f;
#pragma unroll
        for (int ks = 0; ks < KS; ks += 2) {
            uint32_t bk0[4], bk1[4];  // n-tile 0 / 1: (b0, b1) of k-step ks, then of ks + 1
            ldsm_x4(k_base + (0 * 8 + (lane & 7)) * L::kRowB + (ks * 16 + (lane >> 3) * 8) * 2, bk0[0], bk0[1], bk0[2], bk0[3]);
            ldsm_x4(k_base + (1 * 8 + (lane & 7)) * L::kRowB + (ks * 16 + (lane >> 3) * 8) * 2, bk1[0], bk1[1], bk1[2], bk1[3]);
#pragma unroll
            for (int mt = 0; mt < MT; ++mt) {
                uint32_t a[2][4];
#pragma unroll
                for (int kk = 0; kk < 2; ++kk)
                    ldsm_x4(q_base + (mt * 16 + (lane & 15)) * L::kRowB + ((ks + kk) * 16 + (lane >> 4) * 8) * 2,
                            a[kk][0], a[kk][1], a[kk][2], a[kk][3]);
                mma_bf16_16816(sacc[mt][0], a[0][0], a[0][1], a[0][2], a[0][3], bk0[0], bk0[1]);
                mma_bf16_16816(sacc[mt][1], a[0][0], a[0][1], a[0][2], a[0][3], bk1[0], bk1[1]);
                mma_bf16_16816(sodd[mt][0], a[1][0], a[1][1], a[1][2], a[1][3], bk0[2], bk0[3]);
                mma_bf16_16816(sodd[mt][1], a[1][0], a[1][1], a[1][2], a[1][3], bk1[2], bk1[3]);
            }
        }
#pragma unroll
        for (int mt = 0; mt < MT; ++mt)
#pragma unroll
            for (int nt = 0; nt < 2; ++nt)
#pragma unroll
                for (int e = 0; e < 4; ++e) sacc[mt][nt][e] += sodd[mt][nt][e];

        // ---- online softmax (base 2); this lane holds rows 8*nt + 2*t4 + e of query rows g, g + 8
        bool kval[2][2];
#pragma unroll
        for (int nt = 0; nt < 2; ++nt)
#pragma unroll
            for (int e = 0; e < 2; ++e) {
                if constexpr (Scl::kInt8)
                    kval[nt][e] = __shfl_sync(0xffffffffu, my_code, nt * 8 + 2 * t4 + e) != kNoRow;
                else
                    kval[nt][e] = code_of(c * kSub + nt * 8 + 2 * t4 + e) != kNoRow;
            }
        uint32_t ph[MT][4], pl[MT][4];  // P as A fragments (hi, lo)
#pragma unroll
        for (int mt = 0; mt < MT; ++mt) {
            const int nhf = mt * 16 + 8 < nq ? 2 : 1;  // warp-uniform
#pragma unroll
            for (int hf = 0; hf < 2; ++hf) {
                if (hf >= nhf) {  // rows mt*16 + 8.. are padding: P = 0 there
                    sacc[mt][0][2] = sacc[mt][0][3] = sacc[mt][1][2] = sacc[mt][1][3] = 0.f;
                    break;
                }
                const int r = mt * 16 + g + 8 * hf;
                float x[2][2];
                float tmax = -INFINITY;
#pragma unroll
                for (int nt = 0; nt < 2; ++nt)
#pragma unroll
                    for (int e = 0; e < 2; ++e) {
                        const int jk = c * kSub + nt * 8 + 2 * t4 + e;
                        const bool on = kval[nt][e] && vis(r, jk);
                        float xs = sacc[mt][nt][2 * hf + e] * scale_log2;
                        if constexpr (Scl::kInt8)
                            xs *= *reinterpret_cast<const float*>(stages + st * L::kStage +
                                                                  (nt * 8 + 2 * t4 + e) * L::kRowB + 2 * D);
                        x[nt][e] = on ? xs : -INFINITY;
                        tmax = fmaxf(tmax, x[nt][e]);
                    }
                tmax = fmaxf(tmax, __shfl_xor_sync(0xffffffffu, tmax, 1));
                tmax = fmaxf(tmax, __shfl_xor_sync(0xffffffffu, tmax, 2));
                const float mo = acc.m[mt][hf];
                const float mn = fmaxf(mo, tmax);
                const float alpha = (mn == -INFINITY || mn == mo) ? 1.f : fast_exp2(mo - mn);
                float rsum = 0.f;
#pragma unroll
                for (int nt = 0; nt < 2; ++nt)
#pragma unroll
                    for (int e = 0; e < 2; ++e) {
                        const float pv = (x[nt][e] == -INFINITY) ? 0.f : fast_exp2(x[nt][e] - mn);
                        sacc[mt][nt][2 * hf + e] = pv;
                        if constexpr (Scl::kInt8)
                            sacc[mt][nt][2 * hf + e] =
                                pv * *reinterpret_cast<const float*>(stages + st * L::kStage + kSub * L::kRowB +
                                                                     (nt * 8 + 2 * t4 + e) * L::kRowB + 2 * D);
                        rsum += pv;
                    }
                rsum += __shfl_xor_sync(0xffffffffu, rsum, 1);
                rsum += __shfl_xor_sync(0xffffffffu, rsum, 2);
                acc.l[mt][hf] = acc.l[mt][hf] * alpha + rsum;
                acc.m[mt][hf] = mn;
                if (__any_sync(0xffffffffu, alpha != 1.f)) {  // only when a row's maximum moved
#pragma unroll
                    for (int nt = 0; nt < NT; ++nt) {
                        acc.o[mt][nt][2 * hf] *= alpha;
                        acc.o[mt][nt][2 * hf + 1] *= alpha;
                    }
                }
#pragma unroll
                for (int nt = 0; nt < 2; ++nt)
#pragma unroll
                    for (int e = 0; e < 2; ++e) {
                        const int j = c * kSub + nt * 8 + 2 * t4 + e;
                        if (j < nrows) logit(r, j, x[nt][e]);
                    }
            }
            // A fragments: a0 = (g, rows 2t..), a1 = (g+8, 2t..), a2 = (g, 2t+8..), a3 = (g+8, 2t+8..)
            split_bf16x2(sacc[mt][0][0], sacc[mt][0][1], ph[mt][0], pl[mt][0]);
            split_bf16x2(sacc[mt][0][2], sacc[mt][0][3], ph[mt][1], pl[mt][1]);
            split_bf16x2(sacc[mt][1][0], sacc[mt][1][1], ph[mt][2], pl[mt][2]);
            split_bf16x2(sacc[mt][1][2], sacc[mt][1][3], ph[mt][3], pl[mt][3]);
        }

        // ---- O += P V: V fragments by ldmatrix.trans, 4 n-tiles per round: the hi parts of
        // the 4 accumulators, then the lo parts (4 MMAs between dependent ones)
#pragma unroll
        for (int nt = 0; nt < NT; nt += 4) {
            uint32_t v[8];
            ldsm_x4_t(v_base + (lane & 15) * L::kRowB + (nt * 8 + (lane >> 4) * 8) * 2, v[0], v[1], v[2], v[3]);
            ldsm_x4_t(v_base + (lane & 15) * L::kRowB + ((nt + 2) * 8 + (lane >> 4) * 8) * 2, v[4], v[5], v[6], v[7]);
#pragma unroll
            for (int mt = 0; mt < MT; ++mt) {
#pragma unroll
                for (int u = 0; u < 4; ++u)
                    mma_bf16_16816(acc.o[mt][nt + u], ph[mt][0], ph[mt][1], ph[mt][2], ph[mt][3], v[2 * u], v[2 * u + 1]);
#pragma unroll
                for (int u = 0; u < 4; ++u)
                    mma_bf16_16816(acc.o[mt][nt + u], pl[mt][0], pl[mt][1], pl[mt][2], pl[mt][3], v[2 * u], v[2 * u + 1]);
            }
        }
        __syncwarp();
        if (ci + NS < my_n) {
            issue(ci + NS, st);
            ++issued;
        }
    }
}

// Combines the NW warps' (m, l, O) of a CTA; called by all NW*32 threads after every
// warp's loop.  Scratch: mlw [2*NW*RP] floats, rowv [(2+NW)*RP] floats, ow [NW][RP][D]
// floats (the warps' stage area may be reused: the call starts with a barrier).  Leaves, for
// the nq real query rows r < nq (the padding rows are not combined), rowM = rowv[0, RP) (the
// CTA's row maxima), rowL = rowv[RP, 2RP) (sums of l rescaled to them) and ow[w][r] = warp
// w's O row r rescaled to rowM[r]; the CTA's unnormalised O row is the sum over w.
template <int D, int RP, int NW = kMmaWarps>
SD_DEVINL void mma_combine_warps(const WarpAcc<D, RP>& acc, float* mlw, float* rowv, float* ow, int nq) {
    constexpr int MT = RP / 16, NT = D / 8;
    const int tid = threadIdx.x, lane = tid & 31, warp = tid >> 5;
    const int g = lane >> 2, t4 = lane & 3;
    if (t4 == 0) {
#pragma unroll
        for (int mt = 0; mt < MT; ++mt)
#pragma unroll
            for (int hf = 0; hf < 2; ++hf) {
                const int r = mt * 16 + g + 8 * hf;
                mlw[warp * RP + r] = acc.m[mt][hf];
                mlw[NW * RP + warp * RP + r] = acc.l[mt][hf];
            }
    }
    __syncthreads();  // every warp is done with its stages: they may hold the warps' O now
    float* rowM = rowv;
    float* rowL = rowv + RP;
    float* fac = rowv + 2 * RP;  // [NW][RP]
    if (tid < RP && tid < nq) {
        const int r = tid;
        float M = mlw[r];
#pragma unroll
        for (int w = 1; w < NW; ++w) M = fmaxf(M, mlw[w * RP + r]);
        float Ls = 0.f;
#pragma unroll
        for (int w = 0; w < NW; ++w) {
            const float mw = mlw[w * RP + r];
            const float f = (mw == -INFINITY) ? 0.f : exp2f(mw - M);
            fac[w * RP + r] = f;
            Ls = fmaf(mlw[NW * RP + w * RP + r], f, Ls);
        }
        rowM[r] = M;
        rowL[r] = Ls;
    }
    __syncthreads();
#pragma unroll
    for (int mt = 0; mt < MT; ++mt)
#pragma unroll
        for (int hf = 0; hf < 2; ++hf) {
            const int r = mt * 16 + g + 8 * hf;
            if (r >= nq) continue;
            const float f = fac[warp * RP + r];
#pragma unroll
            for (int nt = 0; nt < NT; ++nt) {
                const float2 o2 = make_float2(acc.o[mt][nt][2 * hf] * f, acc.o[mt][nt][2 * hf + 1] * f);
                *reinterpret_cast<float2*>(ow + ((size_t)warp * RP + r) * D + nt * 8 + 2 * t4) = o2;
            }
        }
    __syncthreads();
}

// The CTA's unnormalised O columns [col, col + 4) of row r: the sum of the NW warps' parts.
template <int D, int RP, int NW = kMmaWarps>
SD_DEVINL float4 mma_cta_row4(const float* ow, int r, int col) {
    float4 o = *reinterpret_cast<const float4*>(ow + (size_t)r * D + col);
#pragma unroll
    for (int w = 1; w < NW; ++w) {
        const float4 x = *reinterpret_cast<const float4*>(ow + ((size_t)w * RP + r) * D + col);
        o.x += x.x;
        o.y += x.y;
        o.z += x.z;
        o.w += x.w;
    }
    return o;
}

}  // namespace sd
