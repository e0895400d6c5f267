// step_tiles.cuh -- the per-warp tensor-core tiles of a decode step: indexer scores of 64
// keys, and exact online-softmax attention over 32 K/V rows, for the query rows of one GQA
// group (mma.sync m16n8k16, operands in shared memory in the 128-byte-swizzled layout that
// tiled TMA writes).
//
// SparDA (gist.science summary), sec. 2 "Indexador de Previsao Compacto": the indexer score
// of a token (or block) is a dot product with no softmax, the max over the query rows of a
// verify batch.  "Esparsidade de Contexto no Tempo de Inferencia" (gist.science summary),
// sec. 2: exact attention over the selected rows only.
#pragma once

#include <cmath>

#include "sd_common.cuh"

namespace sd {

// ------------------------------------------------------------------ waits

// A bounded mbarrier wait that also gives up as soon as another role raised the abort flag.
// Between checks of the deadline and the flag the thread sleeps in the barrier (up to 20 us,
// woken when the phase completes), so waiting warps leave the issue slots to working ones.
SD_DEVINL bool ds_wait(uint64_t* bar, uint32_t parity, const volatile int* abort_flag, uint64_t limit) {
    if (mbar_try_wait(bar, parity)) return true;
    const uint64_t t0 = globaltimer_ns();
    for (;;) {
        if (mbar_try_wait_sleep(bar, parity, 20000u)) return true;
        if (*abort_flag) return false;
        if (globaltimer_ns() - t0 > limit) return false;
    }
}

// Lane 0 waits (bounded) and the warp follows its result; on success every lane then observes
// the completed phase itself (acquire), which cannot have moved on: the next phase needs this
// warp first.
SD_DEVINL bool warp_wait(uint64_t* bar, uint32_t parity, volatile int* abort_flag, uint64_t limit) {
    bool ok = true;
    if ((threadIdx.x & 31) == 0) ok = ds_wait(bar, parity, abort_flag, limit);
    ok = __shfl_sync(0xffffffffu, ok ? 1 : 0, 0) != 0;
    if (ok) (void)mbar_try_wait(bar, parity);
    else *abort_flag = 1;
    return ok;
}

// ------------------------------------------------------------------ tiles

// Byte offset of 16-byte chunk c (0..15 over a 128-element bf16 row) of row r in a stage
// tile of `rows` rows stored as two 64-column halves with the 128-byte swizzle.
SD_DEVINL uint32_t swz(int rows, int r, int c) {
    return (uint32_t)((c >> 3) * rows * 128 + r * 128 + (((c & 7) ^ (r & 7)) << 4));
}

// ------------------------------------------------------------------ scoring

// Scores of 64 indexer keys (a swizzled 64-row tile at kb) against the V <= 8 query rows at qb
// (256 bytes apart; the max over V is the key's score), one warp, mma.sync m16n8k16: written
// to the warp's 64-float buffer.  Products of integer-valued keys and queries are exact, and
// so are their fp32 sums.
template <bool F16>
SD_DEVINL void score_tile(uint32_t kb, uint32_t qb, int lane, int V, float* sbuf) {
    float acc[4][4];
#pragma unroll
    for (int mt = 0; mt < 4; ++mt)
#pragma unroll
        for (int e = 0; e < 4; ++e) acc[mt][e] = 0.f;
#pragma unroll
    for (int ks = 0; ks < 8; ks += 2) {
        // B = q^T: matrices (query rows 0-7) x (dims 16ks + 0..7, +8..15, 16(ks+1) + 0..7, +8..15)
        uint32_t b[4];
        ldsm_x4(qb + (lane & 7) * 256 + (ks * 16 + (lane >> 3) * 8) * 2, b[0], b[1], b[2], b[3]);
#pragma unroll
        for (int kk = 0; kk < 2; ++kk)
#pragma unroll
            for (int mt = 0; mt < 4; ++mt) {
                const int row = 16 * mt + (lane & 15);
                const int chunk = 2 * (ks + kk) + (lane >> 4);
                uint32_t a0, a1, a2, a3;
                ldsm_x4(kb + swz(64, row, chunk), a0, a1, a2, a3);
                if constexpr (F16)
                    mma_f16_16816(acc[mt], a0, a1, a2, a3, b[2 * kk], b[2 * kk + 1]);
                else
                    mma_bf16_16816(acc[mt], a0, a1, a2, a3, b[2 * kk], b[2 * kk + 1]);
            }
    }
    const int g8 = lane >> 2, t4 = lane & 3;
#pragma unroll
    for (int mt = 0; mt < 4; ++mt) {
        float v0 = -INFINITY, v1 = -INFINITY;  // keys g8 and g8 + 8 of this M tile
        if (2 * t4 < V) {
            v0 = acc[mt][0];
            v1 = acc[mt][2];
        }
        if (2 * t4 + 1 < V) {
            v0 = fmaxf(v0, acc[mt][1]);
            v1 = fmaxf(v1, acc[mt][3]);
        }
        v0 = fmaxf(v0, __shfl_xor_sync(0xffffffffu, v0, 1));
        v0 = fmaxf(v0, __shfl_xor_sync(0xffffffffu, v0, 2));
        v1 = fmaxf(v1, __shfl_xor_sync(0xffffffffu, v1, 1));
        v1 = fmaxf(v1, __shfl_xor_sync(0xffffffffu, v1, 2));
        if (t4 == 0) {
            sbuf[16 * mt + g8] = v0;
            sbuf[16 * mt + g8 + 8] = v1;
        }
    }
}

// ------------------------------------------------------------------ attention

// One warp's running state over the rows it has attended: the unnormalised output of the 16
// (padded) query rows, their running max and denominator.
struct AttAcc {
    float o[16][4];    // the 128 output columns: n-tiles of 8, C fragments
    float m[2], l[2];  // query rows g8 and g8 + 8 (base-2 units)
};

// Query A fragments of the 16 (padded) query rows for the 8 k-steps of d = 128; rows >= R zero.
SD_DEVINL void load_q_frags(uint32_t qb, int lane, int R, uint32_t (&qf)[8][4]) {
    const int g8 = lane >> 2;
#pragma unroll
    for (int ks = 0; ks < 8; ++ks) {
        ldsm_x4(qb + (lane & 15) * 256 + (2 * ks + (lane >> 4)) * 16, qf[ks][0], qf[ks][1], qf[ks][2], qf[ks][3]);
        if (g8 >= R) qf[ks][0] = qf[ks][2] = 0u;
        if (g8 + 8 >= R) qf[ks][1] = qf[ks][3] = 0u;
    }
}

// 32 K rows at kb and the 32 V rows at vb (swizzled 32-row tiles) for all query rows, one
// warp: S = Q K^T (16 x 32), the online softmax (base 2) over the rows whose bit is set in
// `valid`, then O += P V over all 128 columns.
SD_DEVINL void attend_stage(uint32_t kb, uint32_t vb, int lane, const uint32_t (&qf)[8][4], bool two_halves,
                            uint32_t valid, float scale_log2, AttAcc& acc) {
    float s[4][4];
#pragma unroll
    for (int n = 0; n < 4; ++n)
#pragma unroll
        for (int e = 0; e < 4; ++e) s[n][e] = 0.f;
#pragma unroll
    for (int ks = 0; ks < 8; ++ks)
#pragma unroll
        for (int pp = 0; pp < 2; ++pp) {
            // matrices: keys 16pp + 0..7 (dims 16ks + 0..7, +8..15), keys 16pp + 8..15 (same)
            const int key = 16 * pp + (lane & 7) + ((lane >> 4) << 3);
            const int chunk = 2 * ks + ((lane >> 3) & 1);
            uint32_t r0, r1, r2, r3;
            ldsm_x4(kb + swz(32, key, chunk), r0, r1, r2, r3);
            mma_bf16_16816(s[2 * pp], qf[ks][0], qf[ks][1], qf[ks][2], qf[ks][3], r0, r1);
            mma_bf16_16816(s[2 * pp + 1], qf[ks][0], qf[ks][1], qf[ks][2], qf[ks][3], r2, r3);
        }
    const int t4 = lane & 3;
#pragma unroll
    for (int hf = 0; hf < 2; ++hf) {
        if (hf == 1 && !two_halves) {  // query rows 8..15 are padding: P = 0 there
#pragma unroll
            for (int n = 0; n < 4; ++n) s[n][2] = s[n][3] = 0.f;
            break;
        }
        float tmax = -INFINITY;
#pragma unroll
        for (int n = 0; n < 4; ++n)
#pragma unroll
            for (int e = 0; e < 2; ++e) {
                const int j = 8 * n + 2 * t4 + e;
                const float x = ((valid >> j) & 1u) ? s[n][2 * hf + e] * scale_log2 : -INFINITY;
                s[n][2 * hf + e] = x;
                tmax = fmaxf(tmax, x);
            }
        tmax = fmaxf(tmax, __shfl_xor_sync(0xffffffffu, tmax, 1));
        tmax = fmaxf(tmax, __shfl_xor_sync(0xffffffffu, tmax, 2));
        const float mo = acc.m[hf];
        const float mn = fmaxf(mo, tmax);
        const float alpha = (mn == -INFINITY || mn == mo) ? 1.f : fast_exp2(mo - mn);
        float rsum = 0.f;
#pragma unroll
        for (int n = 0; n < 4; ++n)
#pragma unroll
            for (int e = 0; e < 2; ++e) {
                const float x = s[n][2 * hf + e];
                const float pv = (x == -INFINITY) ? 0.f : fast_exp2(x - mn);
                s[n][2 * hf + e] = pv;
                rsum += pv;
            }
        rsum += __shfl_xor_sync(0xffffffffu, rsum, 1);
        rsum += __shfl_xor_sync(0xffffffffu, rsum, 2);
        acc.l[hf] = acc.l[hf] * alpha + rsum;
        acc.m[hf] = mn;
        if (alpha != 1.f) {
#pragma unroll
            for (int nt = 0; nt < 16; ++nt) {
                acc.o[nt][2 * hf] *= alpha;
                acc.o[nt][2 * hf + 1] *= alpha;
            }
        }
    }
    // P as A fragments (bf16 hi + lo, ~16 significant bits), k-step kk = keys 16kk .. 16kk + 15
#pragma unroll
    for (int kk = 0; kk < 2; ++kk) {
        uint32_t ph[4], pl[4];
        split_bf16x2(s[2 * kk][0], s[2 * kk][1], ph[0], pl[0]);
        split_bf16x2(s[2 * kk][2], s[2 * kk][3], ph[1], pl[1]);
        split_bf16x2(s[2 * kk + 1][0], s[2 * kk + 1][1], ph[2], pl[2]);
        split_bf16x2(s[2 * kk + 1][2], s[2 * kk + 1][3], ph[3], pl[3]);
#pragma unroll
        for (int c2 = 0; c2 < 8; ++c2) {
            // V rows 16kk + 0..15, columns 16 c2 .. 16 c2 + 15, transposed into B fragments
            const int key = 16 * kk + (lane & 15);
            const int chunk = 2 * c2 + (lane >> 4);
            uint32_t v0, v1, v2, v3;
            ldsm_x4_t(vb + swz(32, key, chunk), v0, v1, v2, v3);
            mma_bf16_16816(acc.o[2 * c2], ph[0], ph[1], ph[2], ph[3], v0, v1);
            mma_bf16_16816(acc.o[2 * c2 + 1], ph[0], ph[1], ph[2], ph[3], v2, v3);
            mma_bf16_16816(acc.o[2 * c2], pl[0], pl[1], pl[2], pl[3], v0, v1);
            mma_bf16_16816(acc.o[2 * c2 + 1], pl[0], pl[1], pl[2], pl[3], v2, v3);
        }
    }
}

// ------------------------------------------------------------------ attention, transposed

// The same exact online-softmax attention with the roles of the operands swapped, for few
// query rows: S^T = K Q^T puts the 32 keys on the M side (two 16-row tiles) and the query rows
// on the N side (NQ tiles of 8), and O^T = V^T P^T puts the 128 output columns on the M side,
// so the tensor cores do 16 + 32 (hi and lo parts of P) mma.sync per 32 rows and 8 query rows,
// half of what the 16-row query tile of attend_stage takes.  P^T leaves the S^T accumulators
// (keys by row) and enters the B operand (keys by column) through movmatrix transposes.
template <int NQ>
struct AttAccT {
    float o[8][NQ][4];     // O^T: column tiles of 16 x query tiles of 8, C fragments
    float m[NQ][2], l[NQ][2];  // query rows 8nq + 2(lane % 4) + e (base-2 units)
};

// B fragments of the query rows (rows 8nq .. 8nq + 7 at qb, 256 bytes apart) for the 8 k-steps
// of d = 128: qf[ks][nq][0..1].  Rows >= R must hold zeros in shared memory.
template <int NQ>
SD_DEVINL void load_q_frags_t(uint32_t qb, int lane, uint32_t (&qf)[8][NQ][2]) {
#pragma unroll
    for (int nq = 0; nq < NQ; ++nq)
#pragma unroll
        for (int ks = 0; ks < 8; ks += 2) {
            uint32_t b0, b1, b2, b3;
            ldsm_x4(qb + (8 * nq + (lane & 7)) * 256 + (ks * 16 + (lane >> 3) * 8) * 2, b0, b1, b2, b3);
            qf[ks][nq][0] = b0;
            qf[ks][nq][1] = b1;
            qf[ks + 1][nq][0] = b2;
            qf[ks + 1][nq][1] = b3;
        }
}

template <int NQ>
SD_DEVINL void att_init_t(AttAccT<NQ>& acc) {
#pragma unroll
    for (int md = 0; md < 8; ++md)
#pragma unroll
        for (int nq = 0; nq < NQ; ++nq)
#pragma unroll
            for (int e = 0; e < 4; ++e) acc.o[md][nq][e] = 0.f;
#pragma unroll
    for (int nq = 0; nq < NQ; ++nq) {
        acc.m[nq][0] = acc.m[nq][1] = -INFINITY;
        acc.l[nq][0] = acc.l[nq][1] = 0.f;
    }
}

// A logit sink that keeps nothing.
struct NoLogits {
    SD_DEVINL void operator()(int, int, float) const {}
};

// 32 K rows at kb and the 32 V rows at vb (swizzled 32-row tiles) for the query rows of
// qf, one warp; keys whose bit is clear in `valid` take no part.  logit(query row, key,
// scaled logit in base 2) receives every valid key's logit of every query row of the tile.
template <int NQ, class Logit = NoLogits>
SD_DEVINL void attend_stage_t(uint32_t kb, uint32_t vb, int lane, const uint32_t (&qf)[8][NQ][2], uint32_t valid,
                              float scale_log2, AttAccT<NQ>& acc, const Logit& logit = Logit()) {
    const int g8 = lane >> 2, t4 = lane & 3;
    float s[2][NQ][4];
#pragma unroll
    for (int mt = 0; mt < 2; ++mt)
#pragma unroll
        for (int nq = 0; nq < NQ; ++nq)
#pragma unroll
            for (int e = 0; e < 4; ++e) s[mt][nq][e] = 0.f;
    // S^T = K Q^T: keys 16mt + 0..15 by dims 16ks + 0..15
#pragma unroll
    for (int ks = 0; ks < 8; ++ks)
#pragma unroll
        for (int mt = 0; mt < 2; ++mt) {
            uint32_t a0, a1, a2, a3;
            ldsm_x4(kb + swz(32, 16 * mt + (lane & 15), 2 * ks + (lane >> 4)), a0, a1, a2, a3);
#pragma unroll
            for (int nq = 0; nq < NQ; ++nq) mma_bf16_16816(s[mt][nq], a0, a1, a2, a3, qf[ks][nq][0], qf[ks][nq][1]);
        }
    // online softmax per query column: this lane holds keys 16mt + g8 (+8) of query 8nq + 2t4 + e
    uint32_t ph[2][NQ][2], pl[2][NQ][2];  // P^T halves packed by key rows: [kk][nq][e-pair]
#pragma unroll
    for (int nq = 0; nq < NQ; ++nq) {
#pragma unroll
        for (int e = 0; e < 2; ++e) {
            float tmax = -INFINITY;
#pragma unroll
            for (int mt = 0; mt < 2; ++mt)
#pragma unroll
                for (int h = 0; h < 2; ++h) {
                    const int key = 16 * mt + g8 + 8 * h;
                    const bool on = (valid >> key) & 1u;
                    const float x = on ? s[mt][nq][2 * h + e] * scale_log2 : -INFINITY;
                    if (on) logit(8 * nq + 2 * t4 + e, key, x);
                    s[mt][nq][2 * h + e] = x;
                    tmax = fmaxf(tmax, x);
                }
            tmax = fmaxf(tmax, __shfl_xor_sync(0xffffffffu, tmax, 4));
            tmax = fmaxf(tmax, __shfl_xor_sync(0xffffffffu, tmax, 8));
            tmax = fmaxf(tmax, __shfl_xor_sync(0xffffffffu, tmax, 16));
            const float mo = acc.m[nq][e];
            const float mn = fmaxf(mo, tmax);
            const float alpha = (mn == -INFINITY || mn == mo) ? 1.f : fast_exp2(mo - mn);
            float rsum = 0.f;
#pragma unroll
            for (int mt = 0; mt < 2; ++mt)
#pragma unroll
                for (int h = 0; h < 2; ++h) {
                    const float x = s[mt][nq][2 * h + e];
                    const float pv = (x == -INFINITY) ? 0.f : fast_exp2(x - mn);
                    s[mt][nq][2 * h + e] = pv;
                    rsum += pv;
                }
            rsum += __shfl_xor_sync(0xffffffffu, rsum, 4);
            rsum += __shfl_xor_sync(0xffffffffu, rsum, 8);
            rsum += __shfl_xor_sync(0xffffffffu, rsum, 16);
            acc.l[nq][e] = acc.l[nq][e] * alpha + rsum;
            acc.m[nq][e] = mn;
            if (alpha != 1.f) {
#pragma unroll
                for (int md = 0; md < 8; ++md) {
                    acc.o[md][nq][e] *= alpha;
                    acc.o[md][nq][2 + e] *= alpha;
                }
            }
        }
        // P^T as B fragments: the 8x8 block of keys 16kk + 8h + 0..7 by these 8 query
        // columns, split into bf16 hi + lo parts and transposed (keys by column)
#pragma unroll
        for (int kk = 0; kk < 2; ++kk)
#pragma unroll
            for (int h = 0; h < 2; ++h) {
                uint32_t hi, lo;
                split_bf16x2(s[kk][nq][2 * h], s[kk][nq][2 * h + 1], hi, lo);
                ph[kk][nq][h] = movmatrix_t(hi);
                pl[kk][nq][h] = movmatrix_t(lo);
            }
    }
    // O^T += V^T P^T: output columns 16md + 0..15 by keys 16kk + 0..15
#pragma unroll
    for (int kk = 0; kk < 2; ++kk)
#pragma unroll
        for (int md = 0; md < 8; ++md) {
            uint32_t a0, a1, a2, a3;
            ldsm_x4_t(vb + swz(32, 16 * kk + (lane & 7) + ((lane >> 4) << 3), 2 * md + ((lane >> 3) & 1)), a0, a1, a2,
                      a3);
#pragma unroll
            for (int nq = 0; nq < NQ; ++nq) {
                mma_bf16_16816(acc.o[md][nq], a0, a1, a2, a3, ph[kk][nq][0], ph[kk][nq][1]);
                mma_bf16_16816(acc.o[md][nq], a0, a1, a2, a3, pl[kk][nq][0], pl[kk][nq][1]);
            }
        }
}

}  // namespace sd
