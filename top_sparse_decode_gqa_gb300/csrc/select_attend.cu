// select_attend.cu -- exact top-k selection fused with the gather-attend: one thread-block
// cluster of P CTAs per (b, kvh).
//
// "Esparsidade de Contexto no Tempo de Inferencia" (gist.science summary), sec. 2: Oracle
// Top-K (the exact k highest-scoring tokens) feeding a sparse decode kernel over the
// irregular selection; sec. 3C: memory traffic O(k*d).  SparDA (gist.science summary),
// sec. 2 item 1: top-k blocks.  Adaptive DHiSparse (news page), "Metodologia": the query
// rows of a group share each fetched row.  The pages are silent on ties; the lower index
// wins, as in sd_topk.
//
// Computes exactly what sd_topk followed by sd_gather_attend computes, in one launch and
// without leaving the SMs between the two steps.  CTA c of a cluster owns the contiguous
// part [c*part, (c+1)*part) of the row's N scores.  Exchanges between the CTAs go through
// distributed shared memory (DSMEM) as pushes (remote adds and stores) followed by one
// cluster barrier, never as remote reads:
//   1. the row's top digit d0 (11 bits of the order key) comes from the indexer's
//      histogram; one pass over the part marks every score above d0's bin in a bitmap
//      (float compares against the bin's bounds) and keeps the bin's scores as candidates;
//      each CTA histograms their next digit and pushes 64 coarse sums of it to every CTA
//      (barrier B1);
//   2. every CTA picks the same coarse group, then reads that group's 32 fine bins from
//      the cluster and picks the same digit d1; candidates above it join the bitmap, and
//      those in the final 21-bit bin are pushed with their positions to every CTA,
//      together with the part's count of scores above that bin (barrier B2);
//   3. locally, every CTA finds the threshold key among the final-bin entries, every
//      part's counts above / equal to it, its own ties (lowest indices first) and its
//      offset in the row's ascending output, and writes its selected indices there;
//   4. the CTA attends over its own selected rows with the warp-MMA loop of
//      attend_mma.cuh (all G*V query rows of the group per fetched row);
//   5. the partial (m, l, O) of each query row is pushed to the CTA that owns the row
//      (barrier B4), which merges the P partials.
// When the candidates or the final bin overflow their buffers (heavy ties), every CTA
// resolves the threshold over the whole row from global memory instead (same result).
#include <cooperative_groups.h>

#include <algorithm>
#include <map>
#include <mutex>
#include <tuple>

#include "attend_mma.cuh"
#include "sd_common.cuh"
#include "sd_host.h"

namespace cg = cooperative_groups;

// Most of this kernel's code runs once per launch, so its time goes to fetching instructions
// into a cold cache.  Helpers called more than once, and paths that normally do not run, are
// kept out of line: repeated calls then hit a warm cache and the common path stays compact.
#define SD_DEVNOINL __device__ __noinline__

namespace sd {
namespace {

constexpr int kSaThreads = kMmaWarps * 32;
constexpr int kSaWarps = kMmaWarps;
constexpr int kSaHist = 2048;      // bins of the 11-bit digits
constexpr int kSaMaxCluster = 8;   // portable cluster size
constexpr int kSaWin = 512;        // selected rows whose sources are resolved at a time
constexpr int kSaPartAlign = 128;  // part sizes are multiples of this many scores

struct SelAttParams {
    const float* scores;  // [rows, N]
    uint32_t* key_hist;   // [rows, 2048] or null
    int32_t* idx;         // [rows, k]
    int N, k, part, staged;
    const void* q;
    const uint8_t* kc;
    const uint8_t* vc;
    const uint8_t* kh;
    const uint8_t* vh;
    const int32_t* slot_map;
    int B, V, Hq, Hkv, G, R, T, pool_rows, block;
    float scale_log2;
    float* out;
    float* lse;
    float* logits;
    int32_t* err;
    int inbox_own;  // 1: the merge inbox has its own shared memory after the layout's end
    int attend;     // 0: selection only (idx written; q, K/V and the outputs untouched)
    int slot_per_head;  // 1: slot_map is [B, Hkv, T]
};

// Shared-memory layout (byte offsets), in order:
//   Q    the RP query rows (bf16, padded rows)
//   U    the warps' K/V stages; before them, the part's scores when they are staged
//   H    hist0 (top digit; after B1 the row's final-bin entries pushed by the cluster),
//        hist1 (this part's digit 1), hist2 (the cluster's coarse digit-1 sums, then digit 2
//        of the final bin); the merge inbox when it has no memory of its own (after B3)
//   S    sel and tie bitmaps of the part
//   C    phase A: the candidates' keys and indices; phase B: row sources, warp and
//        row statistics
//   Lst  this CTA's final-bin candidates, then its selected entries in ascending order
//   Misc SaMisc
struct SaLayout {
    int oQ, oU, oH, oHist0, oHist1, oHist2, oSel, oTie, oCandK, oCandI, oSrc, oML, oRow, oLst, oMisc, bytes;
};

constexpr int kSaCand = 1024;  // candidates a CTA keeps
constexpr int kSaList = 512;   // selected entries a CTA keeps in shared memory
constexpr int kSaFb = 1024;    // final-bin entries of a row (keys + positions in hist0's 8 KB)
constexpr int kSaHBytes = (2 * kSaHist + kSaHist / 2) * 4;
constexpr int kSaCoarse = 64;  // coarse groups of the digit-1 histogram exchanged by pushes
constexpr int kSaTwoPerSm = 233472 / 2 - 1024;  // dynamic shared memory of one of two CTAs per SM

__host__ __device__ constexpr int sa_align(int x, int a) { return (x + a - 1) / a * a; }

__host__ __device__ inline SaLayout sa_layout(int D, int RP, int part, int staged) {
    SaLayout L{};
    const int row_b = D * 2 + 16;
    const int stages = kMmaWarps * kWStages * 2 * kSub * row_b;
    L.oQ = 0;
    L.oU = sa_align(RP * row_b, 128);
    L.oH = L.oU + sa_align(staged && part * 4 > stages ? part * 4 : stages, 128);
    L.oHist0 = L.oH;
    L.oHist1 = L.oHist0 + kSaHist * 4;
    L.oHist2 = L.oHist1 + kSaHist * 4;
    L.oSel = L.oH + kSaHBytes;
    L.oTie = L.oSel + part / 8;
    L.oCandK = L.oTie + part / 8;
    L.oCandI = L.oCandK + kSaCand * 4;
    L.oSrc = L.oCandK;
    L.oML = L.oSrc + kSaWin * 4;
    L.oRow = L.oML + 2 * kMmaWarps * RP * 4;
    L.oLst = L.oCandI + kSaCand * 4;
    L.oMisc = L.oLst + kSaList * 4;
    L.bytes = L.oMisc + 256;
    return L;
}

// Merge inbox inside H: for each of this CTA's query rows (r = lr * P + rank) and each
// source CTA s, O[lr][s][D], then m[lr][s], l[lr][s].
__host__ __device__ inline int sa_inbox_bytes(int D, int R, int P) {
    const int slots = (R + P - 1) / P * P;
    return slots * (D + 2) * 4;
}

// Values the CTAs of a cluster exchange (ovf, cnt_gt and cnt_eq are written by the other
// CTAs) and the CTA's own scratch.
struct SaMisc {
    uint32_t ovf;                     // some CTA's candidate list overflowed
    uint32_t dsure[kSaMaxCluster];    // per CTA of the cluster: entries above the final bin
    uint32_t fb_n;                    // final-bin entries pushed into this CTA so far
    uint32_t fb_off[kSaMaxCluster];   // where this CTA's entries go in each CTA's buffer
    uint32_t cgt[kSaMaxCluster], ceq[kSaMaxCluster];  // per part: above / equal to the threshold
    uint32_t nfb;                     // this CTA's final-bin entries
    uint32_t ncand;                   // candidates of this part (may exceed kSaCand)
    uint32_t nabove;                  // entries of this part marked in sel so far
    uint32_t wgt[kSaWarps], weq[kSaWarps];
    uint32_t wsum[kSaWarps];
    uint32_t sel_digit, sel_above, tot;
    uint64_t bar;
};
static_assert(sizeof(SaMisc) <= 256, "misc area");

// Inclusive prefix sum over the CTA's 128 threads (one value each).
SD_DEVINL uint32_t cta_inclusive_scan(uint32_t v, uint32_t* wsum) {
    const int lane = threadIdx.x & 31, warp = threadIdx.x >> 5;
#pragma unroll
    for (int o = 1; o < 32; o <<= 1) {
        const uint32_t n = __shfl_up_sync(0xffffffffu, v, o);
        if (lane >= o) v += n;
    }
    if (lane == 31) wsum[warp] = v;
    __syncthreads();
    uint32_t off = 0;
#pragma unroll
    for (int w = 0; w < kSaWarps; ++w)
        if (w < warp) off += wsum[w];
    __syncthreads();
    return v + off;
}

SD_DEVINL uint32_t warp_inclusive_scan(uint32_t v) {
    const int lane = threadIdx.x & 31;
#pragma unroll
    for (int o = 1; o < 32; o <<= 1) {
        const uint32_t n = __shfl_up_sync(0xffffffffu, v, o);
        if (lane >= o) v += n;
    }
    return v;
}

// Block-wide exclusive prefix sums of two values per thread at once (the total of each
// comes from the warp sums): two barriers.
SD_DEVNOINL void cta_exclusive_scan2(uint32_t a, uint32_t b, SaMisc* ms, uint32_t& ea, uint32_t& eb, uint32_t& ta,
                                     uint32_t& tb) {
    const int lane = threadIdx.x & 31, warp = threadIdx.x >> 5;
    uint32_t ia = a, ib = b;
#pragma unroll
    for (int o = 1; o < 32; o <<= 1) {
        const uint32_t na = __shfl_up_sync(0xffffffffu, ia, o), nb = __shfl_up_sync(0xffffffffu, ib, o);
        if (lane >= o) {
            ia += na;
            ib += nb;
        }
    }
    if (lane == 31) {
        ms->wsum[warp] = ia;
        ms->wgt[warp] = ib;
    }
    __syncthreads();
    uint32_t oa = 0, ob = 0, sa = 0, sb = 0;
#pragma unroll
    for (int w = 0; w < kSaWarps; ++w) {
        const uint32_t xa = ms->wsum[w], xb = ms->wgt[w];
        oa += w < warp ? xa : 0u;
        ob += w < warp ? xb : 0u;
        sa += xa;
        sb += xb;
    }
    __syncthreads();  // the warp sums are rewritten by the next scan
    ea = ia - a + oa;
    eb = ib - b + ob;
    ta = sa;
    tb = sb;
}


// Given the histogram of one digit (128 * PER bins, higher bins = larger keys) of the
// entries still in the running, the digit holding the krem-th largest and how many entries
// lie in higher bins.  Thread t holds its bins [PER*(127-t), PER*(128-t)) in registers (v,
// four bins per word), so thread order is descending bin order; the bins are read as 16-byte
// words, a few lanes to a shared-memory bank.  If no bin crosses (a histogram that does not
// match the scores) the answer is digit 0, 0 above.
template <int PER>
SD_DEVINL void cta_select_digit_regs(const uint4 (&v)[PER / 4], uint32_t krem, SaMisc* ms, uint32_t& digit,
                                     uint32_t& above) {
    static_assert(kSaThreads == 128 && PER % 4 == 0, "digit select layout");
    const int tid = threadIdx.x;
    if (tid == 0) {
        ms->sel_digit = 0;
        ms->sel_above = 0;
    }
    uint32_t local = 0;
#pragma unroll
    for (int q = 0; q < PER / 4; ++q) local += v[q].x + v[q].y + v[q].z + v[q].w;
    const uint32_t incl = cta_inclusive_scan(local, ms->wsum);
    const uint32_t excl = incl - local;
    if (excl < krem && krem <= incl) {
        const uint32_t lo = (uint32_t)(PER * (kSaThreads - 1 - tid));
        uint32_t acc = excl;
        bool found = false;
#pragma unroll
        for (int i = PER - 1; i >= 0; --i) {
            const uint4 w = v[i / 4];
            const uint32_t h = (i & 3) == 0 ? w.x : (i & 3) == 1 ? w.y : (i & 3) == 2 ? w.z : w.w;
            if (!found && acc + h >= krem) {
                ms->sel_digit = lo + (uint32_t)i;
                ms->sel_above = acc;
                found = true;
            }
            acc += h;
        }
    }
    __syncthreads();
    digit = ms->sel_digit;
    above = ms->sel_above;
    __syncthreads();
}

// The same over a histogram in shared memory (16-byte aligned) of nb = 2048 or 1024 bins.
SD_DEVNOINL void cta_select_digit(const uint32_t* hist, int nb, uint32_t krem, SaMisc* ms, uint32_t& digit,
                                uint32_t& above) {
    const int t = kSaThreads - 1 - (int)threadIdx.x;
    if (nb == kSaHist) {
        const uint4* h4 = reinterpret_cast<const uint4*>(hist) + 4 * t;
        const uint4 v[4] = {h4[0], h4[1], h4[2], h4[3]};
        cta_select_digit_regs<16>(v, krem, ms, digit, above);
    } else {
        const uint4* h4 = reinterpret_cast<const uint4*>(hist) + 2 * t;
        const uint4 v[2] = {h4[0], h4[1]};
        cta_select_digit_regs<8>(v, krem, ms, digit, above);
    }
}

// dst[i] = sum over the cluster's P CTAs of their copy of src[i], i < n (n a multiple of 4).
SD_DEVNOINL void cluster_sum_hist(cg::cluster_group& cl, const uint32_t* src, uint32_t* dst, int n, int P) {
    for (int i = threadIdx.x; i < n / 4; i += kSaThreads) {
        uint4 x[kSaMaxCluster];
#pragma unroll
        for (int c = 0; c < kSaMaxCluster; ++c)
            if (c < P) x[c] = reinterpret_cast<const uint4*>(cl.map_shared_rank(const_cast<uint32_t*>(src), c))[i];
        uint4 s = make_uint4(0u, 0u, 0u, 0u);
#pragma unroll
        for (int c = 0; c < kSaMaxCluster; ++c)
            if (c < P) {
                s.x += x[c].x;
                s.y += x[c].y;
                s.z += x[c].z;
                s.w += x[c].w;
            }
        reinterpret_cast<uint4*>(dst)[i] = s;
    }
}

// The float whose order key is k (the inverse of float_key); k = 0x7FFFFFFF, the key no
// float maps to (-0 takes the key of +0), gives the largest float below it, -denorm_min.
SD_DEVINL float key_float(uint32_t k) {
    if (k == 0x7FFFFFFFu) return __uint_as_float(0x80000001u);
    return __uint_as_float((k & 0x80000000u) ? (k & 0x7FFFFFFFu) : ~k);
}

// One pass over the part [p0, p1): sel word w = the entries of 32-score group w above the
// d0 bin, tie word w cleared.  The entries in the bin (the candidates) are listed with their
// order keys and positions in the part (in no particular order; only the first kSaCand are
// kept) and their next digit (bits 20..10) is counted into hist1; *ncand ends as the part's
// candidate count and *nabove as its entries above the bin.  Staged scores: each lane builds
// the bits of two words in registers, reading entry (j + lane) mod 32 of each at step j so
// the warp's reads fall in 32 distinct banks; the listing takes one warp prefix sum and one
// atomic per warp.  Scores read from global memory: each warp votes on 32-score groups
// (coalesced), U groups per round.
template <bool STAGED, bool FCMP>
SD_DEVNOINL void sa_scan(const uint32_t* keys_s, const float* srow, int p0, int p1, int nw, uint32_t d0, float f_lo,
                       float f_hi, uint32_t k_hi, uint32_t* sel, uint32_t* tie, uint32_t* cand_k, uint32_t* cand_i,
                       uint32_t* hist1, uint32_t* ncand, uint32_t* nabove) {
    const int lane = threadIdx.x & 31, warp = threadIdx.x >> 5;
    auto classify = [&](float f, bool& above, bool& in) {
        if constexpr (FCMP) {
            above = f > f_hi;
            in = f >= f_lo && f <= f_hi;
        } else {
            const uint32_t kk = float_key(f);
            above = kk > k_hi;
            in = (kk >> 21) == d0;
        }
    };
    if constexpr (STAGED) {
        const int np = p1 - p0;
        // lane words wa = wb + lane and wb + kSaThreads + lane (warp-uniform bounds: shuffles below)
        for (int wb = warp * 32; wb < nw; wb += 2 * kSaThreads) {
            const int wa = wb + lane, wz = wa + kSaThreads;
            const int na = wa < nw ? min(32, np - wa * 32) : 0, nz = wz < nw ? min(32, np - wz * 32) : 0;
            const uint32_t* ra = keys_s + (na > 0 ? wa : 0) * 32;
            const uint32_t* rz = keys_s + (nz > 0 ? wz : 0) * 32;
            // above the bin (s) and at or above its low end (g); in the bin = g and not s
            uint32_t sa = 0u, ga = 0u, sz = 0u, gz = 0u;
            uint32_t bit = 1u << lane;  // the bit of entry (j + lane) mod 32 at step j
#pragma unroll 8
            for (int j = 0; j < 32; ++j) {
                const int e = (j + lane) & 31;
                const float fa = __uint_as_float(ra[e]), fz = __uint_as_float(rz[e]);
                if constexpr (FCMP) {
                    sa |= fa > f_hi ? bit : 0u;
                    ga |= fa >= f_lo ? bit : 0u;
                    sz |= fz > f_hi ? bit : 0u;
                    gz |= fz >= f_lo ? bit : 0u;
                } else {
                    const uint32_t ka = float_key(fa), kz = float_key(fz);
                    sa |= ka > k_hi ? bit : 0u;
                    ga |= (ka >> 21) >= d0 ? bit : 0u;
                    sz |= kz > k_hi ? bit : 0u;
                    gz |= (kz >> 21) >= d0 ? bit : 0u;
                }
                bit = __funnelshift_l(bit, bit, 1);
            }
            const uint32_t ma = na >= 32 ? 0xffffffffu : (1u << na) - 1u;
            const uint32_t mz = nz >= 32 ? 0xffffffffu : (1u << nz) - 1u;
            sa &= ma;
            sz &= mz;
            uint32_t ca = ga & ~sa & ma, cz = gz & ~sz & mz;
            if (na > 0) {
                sel[wa] = sa;
                tie[wa] = 0u;
            }
            if (nz > 0) {
                sel[wz] = sz;
                tie[wz] = 0u;
            }
            const uint32_t nab = __reduce_add_sync(0xffffffffu, (uint32_t)(__popc(sa) + __popc(sz)));
            if (lane == 0 && nab != 0u) atomicAdd(nabove, nab);
            const uint32_t c = (uint32_t)(__popc(ca) + __popc(cz));
            uint32_t incl = c;
#pragma unroll
            for (int o = 1; o < 32; o <<= 1) {
                const uint32_t n = __shfl_up_sync(0xffffffffu, incl, o);
                if (lane >= o) incl += n;
            }
            uint32_t at = 0u;
            if (lane == 31 && incl != 0u) at = atomicAdd(ncand, incl);
            at = __shfl_sync(0xffffffffu, at, 31) + incl - c;
#pragma unroll
            for (int h = 0; h < 2; ++h) {
                uint32_t cb = h == 0 ? ca : cz;
                const uint32_t* row = h == 0 ? ra : rz;
                const int w = h == 0 ? wa : wz;
                while (cb != 0u) {
                    const int e = __ffs(cb) - 1;
                    cb &= cb - 1u;
                    const uint32_t key = float_key(__uint_as_float(row[e]));
                    atomicAdd(&hist1[(key >> 10) & (kSaHist - 1)], 1u);
                    if (at < (uint32_t)kSaCand) {
                        cand_k[at] = key;
                        cand_i[at] = (uint32_t)(w * 32 + e);
                    }
                    ++at;
                }
            }
        }
    } else {
        constexpr int U = 8;
        const uint32_t lt = lanemask_lt();
        for (int g0 = warp; g0 < nw; g0 += U * kSaWarps) {
            float f[U];
            uint32_t sure[U], cm[U];
#pragma unroll
            for (int u = 0; u < U; ++u) {
                const int i = p0 + (g0 + u * kSaWarps) * 32 + lane;
                f[u] = i < p1 ? __ldcg(srow + i) : 0.f;
            }
#pragma unroll
            for (int u = 0; u < U; ++u) {
                const bool valid = p0 + (g0 + u * kSaWarps) * 32 + lane < p1;  // also false past nw
                bool above, in;
                classify(f[u], above, in);
                sure[u] = __ballot_sync(0xffffffffu, valid && above);
                cm[u] = __ballot_sync(0xffffffffu, valid && in);
            }
            uint32_t my_s = 0, nc = 0, na = 0;  // lane u keeps group u's word
#pragma unroll
            for (int u = 0; u < U; ++u) {
                my_s = lane == u ? sure[u] : my_s;
                nc += __popc(cm[u]);
                na += __popc(sure[u]);
            }
            if (lane == 0 && na != 0u) atomicAdd(nabove, na);
            const int gw = g0 + lane * kSaWarps;
            if (lane < U && gw < nw) {
                sel[gw] = my_s;
                tie[gw] = 0u;
            }
            if (nc != 0u) {
                uint32_t at = 0u;
                if (lane == 0) at = atomicAdd(ncand, nc);
                at = __shfl_sync(0xffffffffu, at, 0);
#pragma unroll
                for (int u = 0; u < U; ++u) {
                    if ((cm[u] >> lane) & 1u) {
                        const uint32_t key = float_key(f[u]);
                        const uint32_t slot = at + __popc(cm[u] & lt);
                        atomicAdd(&hist1[(key >> 10) & (kSaHist - 1)], 1u);
                        if (slot < (uint32_t)kSaCand) {
                            cand_k[slot] = key;
                            cand_i[slot] = (uint32_t)((g0 + u * kSaWarps) * 32 + lane);
                        }
                    }
                    at += __popc(cm[u]);
                }
            }
        }
    }
}

// Heavy ties (a candidate list or the final bin overflowed): the threshold key over the
// whole row from global memory, starting from the top digit d0 with krem0 entries still
// needed, and every part's counts above / equal to it (ms->cgt, ms->ceq).  No exchange with
// the other CTAs.  Returns the threshold; *krem_out = entries equal to it still needed.
SD_DEVNOINL uint32_t sa_fallback_threshold(const float* srow, int N, int part, int P, uint32_t d0, uint32_t krem0,
                                           uint32_t* hist, SaMisc* ms, uint32_t& krem_out) {
    const int tid = threadIdx.x, lane = tid & 31, warp = tid >> 5;
    uint32_t prefix = d0 << 21, pmask = 0x7FFu << 21, krem = krem0;
#pragma unroll 1
    for (int pass = 1; pass < 3; ++pass) {
        const int shift = pass == 1 ? 10 : 0;
        const uint32_t nb = pass == 1 ? 2048u : 1024u;
        for (int i = tid; i < kSaHist; i += kSaThreads) hist[i] = 0u;
        __syncthreads();
        for (int base0 = warp * 32; base0 < N; base0 += kSaThreads) {
            const int i = base0 + lane;
            const bool valid = i < N;
            const uint32_t kk = valid ? float_key(__ldcg(srow + i)) : 0u;
            const bool in = valid && (kk & pmask) == prefix;
            const uint32_t dg = (kk >> shift) & (nb - 1);
            const uint32_t peers = __match_any_sync(0xffffffffu, in ? dg : 0xffffffffu);
            if (in && lane == __ffs(peers) - 1) atomicAdd(&hist[dg], (uint32_t)__popc(peers));
        }
        __syncthreads();
        uint32_t dg, ab;
        cta_select_digit(hist, (int)nb, krem, ms, dg, ab);
        prefix |= (dg & (nb - 1)) << shift;
        pmask |= (nb - 1) << shift;
        krem -= ab;
    }
    const uint32_t thr = prefix;
    if (tid < kSaMaxCluster) ms->cgt[tid] = ms->ceq[tid] = 0u;
    __syncthreads();
    for (int base0 = warp * 32; base0 < N; base0 += kSaThreads) {  // groups never straddle parts
        const int i = base0 + lane;
        const bool valid = i < N;
        const uint32_t kk = valid ? float_key(__ldcg(srow + i)) : 0u;
        const uint32_t gt = __popc(__ballot_sync(0xffffffffu, valid && kk > thr));
        const uint32_t eq = __popc(__ballot_sync(0xffffffffu, valid && kk == thr));
        if (lane == 0 && (gt | eq)) {
            const int r = min(base0 / part, P - 1);
            atomicAdd(&ms->cgt[r], gt);
            atomicAdd(&ms->ceq[r], eq);
        }
    }
    __syncthreads();
    krem_out = krem;
    return thr;
}

// Ordered emit over the keys of the part [p0, p1) (staged in keys_s, or read from global
// memory when keys_s is null): every key above thr and the first `take` keys equal to it, in
// ascending index order, to out[0, n_mine) and the first kSaList of them to lst as well.
// Warp w scans the contiguous segment [p0 + w*seg, p0 + (w+1)*seg).
SD_DEVNOINL void sa_emit_ordered(const uint32_t* keys_s, const float* srow, int p0, int p1, uint32_t thr,
                                 uint32_t take, uint32_t n_mine, SaMisc* ms, int32_t* out, int32_t* lst) {
    const int tid = threadIdx.x, lane = tid & 31, warp = tid >> 5;
    auto key_at = [&](int i) -> uint32_t {
        return float_key(keys_s != nullptr ? __uint_as_float(keys_s[i - p0]) : __ldcg(srow + i));
    };
    const int np = p1 - p0;
    const int seg = ((np + kSaWarps - 1) / kSaWarps + 31) / 32 * 32;
    const int s0 = p0 + warp * seg, s1 = min(p1, s0 + seg);
    {
        uint32_t gt = 0, eq = 0;
        for (int i0 = s0; i0 < s1; i0 += 32) {
            const int i = i0 + lane;
            const bool valid = i < s1;
            const uint32_t kk = valid ? key_at(i) : 0u;
            gt += __popc(__ballot_sync(0xffffffffu, valid && kk > thr));
            eq += __popc(__ballot_sync(0xffffffffu, valid && kk == thr));
        }
        if (lane == 0) {
            ms->wgt[warp] = gt;
            ms->weq[warp] = eq;
        }
    }
    __syncthreads();
    uint32_t eq_seen = 0, pos = 0;
    for (int w = 0; w < warp; ++w) {
        const uint32_t tw = take > eq_seen ? min(ms->weq[w], take - eq_seen) : 0u;
        pos += ms->wgt[w] + tw;
        eq_seen += ms->weq[w];
    }
    const uint32_t lt = lanemask_lt();
    for (int i0 = s0; i0 < s1; i0 += 32) {
        const int i = i0 + lane;
        const bool valid = i < s1;
        const uint32_t kk = valid ? key_at(i) : 0u;
        const bool is_gt = valid && kk > thr;
        const bool is_eq = valid && kk == thr;
        const uint32_t eqm = __ballot_sync(0xffffffffu, is_eq);
        const bool pick = is_gt || (is_eq && eq_seen + __popc(eqm & lt) < take);
        const uint32_t pm = __ballot_sync(0xffffffffu, pick);
        const uint32_t at = pos + __popc(pm & lt);
        if (pick && at < n_mine) {
            out[at] = i;
            if (at < (uint32_t)kSaList) lst[at] = i;
        }
        pos += __popc(pm);
        eq_seen += __popc(eqm);
    }
}

template <int D, int RP>
__global__ void __launch_bounds__(kSaThreads) select_attend_kernel(const SelAttParams p) {
    using Rows = MmaRows<D>;
    constexpr int PPR = D * 2 / 16;
    extern __shared__ __align__(128) uint8_t sm[];
    cg::cluster_group cl = cg::this_cluster();
    const int P = (int)cl.num_blocks();
    const int rank = (int)cl.block_rank();
    const SaLayout L = sa_layout(D, RP, p.part, p.staged);
    uint32_t* keys_s = reinterpret_cast<uint32_t*>(sm + L.oU);
    uint32_t* hist0 = reinterpret_cast<uint32_t*>(sm + L.oHist0);
    uint32_t* hist1 = reinterpret_cast<uint32_t*>(sm + L.oHist1);
    uint32_t* hist2 = reinterpret_cast<uint32_t*>(sm + L.oHist2);
    uint32_t* coarse = hist2;  // [P][kSaCoarse] coarse digit-1 sums pushed by the cluster, until B2
    uint32_t* sel = reinterpret_cast<uint32_t*>(sm + L.oSel);
    uint32_t* tie = reinterpret_cast<uint32_t*>(sm + L.oTie);
    uint32_t* cand_k = reinterpret_cast<uint32_t*>(sm + L.oCandK);
    uint32_t* cand_i = reinterpret_cast<uint32_t*>(sm + L.oCandI);
    int32_t* lst = reinterpret_cast<int32_t*>(sm + L.oLst);
    SaMisc* ms = reinterpret_cast<SaMisc*>(sm + L.oMisc);

    const int tid = threadIdx.x, lane = tid & 31, warp = tid >> 5;
    const int kvh = blockIdx.y, b = blockIdx.z;
    const int bk = b * p.Hkv + kvh;
    const int N = p.N, k = p.k;
    const int p0 = min(N, rank * p.part), p1 = min(N, p0 + p.part), np = p1 - p0;
    const int nw = (np + 31) / 32;  // bitmap words of the part
    const float* srow = p.scores + (size_t)bk * N;
    int32_t* orow = p.idx + (size_t)bk * k;
    uint32_t* hrow = p.key_hist != nullptr ? p.key_hist + (size_t)bk * kSaHist : nullptr;
    const bool trivial = (k == 0 || k == N);  // no select needed (every CTA agrees)

    // ---- zero what the cluster adds into; B0: nobody adds before everyone has zeroed
    if (tid == 0) {
        ms->ovf = 0;
        ms->fb_n = 0;
        ms->nfb = 0;
        mbar_init(&ms->bar, 1);
        fence_mbarrier_init();
    }
    if (tid == 0) {
        ms->ncand = 0;
        ms->nabove = 0;
    }
    for (int i = tid; i < 2 * kSaHist + kSaHist / 2; i += kSaThreads) hist0[i] = 0u;  // hist0, hist1, hist2
    cl.sync();  // B0

    pdl_wait();  // scores, key_hist and q may come from the preceding kernels

    // ---- start moving: the part's scores (bulk copies), the query rows (cp.async)
    bool staged = p.staged != 0 && np > 0;
    if (staged && tid == 0) {
        mbar_arrive_expect_tx(&ms->bar, (uint32_t)np * 4u);
        constexpr int kChunk = 8192;  // bytes per bulk copy
        for (int off = 0; off < np * 4; off += kChunk)
            bulk_g2s(reinterpret_cast<uint8_t*>(keys_s) + off, reinterpret_cast<const uint8_t*>(srow + p0) + off,
                     (uint32_t)min(kChunk, np * 4 - off), &ms->bar);
    }
    for (int e = tid; p.attend && e < RP * PPR; e += kSaThreads) {
        const int r = e / PPR, part = e % PPR;
        uint8_t* dst = sm + L.oQ + r * Rows::kRowB + part * 16;
        if (r < p.R) {
            const int v = r / p.G, gg = r % p.G;
            const uint8_t* qrow =
                static_cast<const uint8_t*>(p.q) + ((((size_t)b * p.V + v) * p.Hq + kvh * p.G + gg) * D) * 2;
            cp_async16(dst, qrow + part * 16);
        } else {
            *reinterpret_cast<uint4*>(dst) = make_uint4(0u, 0u, 0u, 0u);
        }
    }
    cp_async_commit();
    // the top digit first when the indexer's histogram is given (read straight into
    // registers): it overlaps the staging
    uint32_t d0 = 0, above0 = 0;
    if (!trivial && hrow != nullptr) {
        const uint4* h4 = reinterpret_cast<const uint4*>(hrow) + 4 * (kSaThreads - 1 - tid);
        const uint4 hv[4] = {__ldcg(h4), __ldcg(h4 + 1), __ldcg(h4 + 2), __ldcg(h4 + 3)};
        cta_select_digit_regs<16>(hv, (uint32_t)k, ms, d0, above0);
        d0 &= kSaHist - 1;
    }
    if (staged) {
        const bool ok = mbar_wait(&ms->bar, 0);
        if (__syncthreads_or(!ok)) {  // keep going on the global copy; the result is flagged
            if (tid == 0) report(p.err, SD_DEVERR_TIMEOUT);
            staged = false;
        }
    }
    auto key_at = [&](int i) -> uint32_t {  // i in [p0, p1)
        return float_key(staged ? __uint_as_float(keys_s[i - p0]) : __ldcg(srow + i));
    };

    // ---- otherwise the top digit is counted here and summed over the cluster
    if (!trivial && hrow == nullptr) {
        for (int base = p0 + warp * 32; base < p1; base += kSaThreads) {
            const int i = base + lane;
            const bool valid = i < p1;
            const uint32_t dg = valid ? key_at(i) >> 21 : 0xffffffffu;
            const uint32_t peers = __match_any_sync(0xffffffffu, dg);
            if (valid && lane == __ffs(peers) - 1) atomicAdd(&hist0[dg], (uint32_t)__popc(peers));
        }
        cl.sync();  // every CTA's top-digit counts are complete (and are not changed again)
        cluster_sum_hist(cl, hist0, cand_k, kSaHist, P);  // the candidate area is free until the pass
        __syncthreads();
        cta_select_digit(cand_k, kSaHist, (uint32_t)k, ms, d0, above0);
        d0 &= kSaHist - 1;
    }
    uint32_t krem = (uint32_t)k - above0;
    const uint32_t krem0 = krem;  // still needed from the d0 bin (the fallback restarts there)

    // ---- one pass over the part: the bitmap of the entries above d0's bin (sel), written by
    // lanes 0..U-1 without divergence, and the list of the entries in it (the candidates) with
    // their next digit counted into hist1; then hist1's coarse sums go to every CTA
    if (!trivial) {
        // the d0 bin as the closed float interval [f_lo, f_hi]: a score lies above the bin iff
        // f > f_hi and in it iff f_lo <= f <= f_hi (-0 and +0 compare equal, as their order
        // keys do); the bins next to the infinities and NaN keys compare keys instead
        const uint32_t k_lo = d0 << 21, k_hi = k_lo | 0x1FFFFFu;
        const bool fcmp = d0 > 0x003u && d0 < 0x7FCu;
        const float f_lo = key_float(k_lo), f_hi = key_float(k_hi);
        if (staged) {
            if (fcmp) sa_scan<true, true>(keys_s, srow, p0, p1, nw, d0, f_lo, f_hi, k_hi, sel, tie, cand_k, cand_i, hist1, &ms->ncand, &ms->nabove);
            else sa_scan<true, false>(keys_s, srow, p0, p1, nw, d0, f_lo, f_hi, k_hi, sel, tie, cand_k, cand_i, hist1, &ms->ncand, &ms->nabove);
        } else {
            if (fcmp) sa_scan<false, true>(keys_s, srow, p0, p1, nw, d0, f_lo, f_hi, k_hi, sel, tie, cand_k, cand_i, hist1, &ms->ncand, &ms->nabove);
            else sa_scan<false, false>(keys_s, srow, p0, p1, nw, d0, f_lo, f_hi, k_hi, sel, tie, cand_k, cand_i, hist1, &ms->ncand, &ms->nabove);
        }
        __syncthreads();
        if (tid == 0 && ms->ncand > (uint32_t)kSaCand)  // the list overflowed: every CTA resolves from global
            for (int c = 0; c < P; ++c) atomicOr(cl.map_shared_rank(&ms->ovf, c), 1u);
        // 64 coarse sums of 32 bins each (a warp reads one group, a lane one bin), pushed to
        // every CTA (the fine bins stay here)
        static_assert(kSaHist / kSaCoarse == 32, "a coarse group is one warp's bins");
#pragma unroll 4
        for (int g = warp; g < kSaCoarse; g += kSaWarps) {
            const uint32_t sum = __reduce_add_sync(0xffffffffu, hist1[g * 32 + lane]);
            if (lane < P) cl.map_shared_rank(coarse, lane)[rank * kSaCoarse + g] = sum;
        }
    }
    cl.sync();  // B1: coarse sums and ovf pushed, every hist1 complete; every CTA has read key_hist
    if (hrow != nullptr && rank == 0)
        for (int i = tid; i < kSaHist / 4; i += kSaThreads) reinterpret_cast<uint4*>(hrow)[i] = make_uint4(0u, 0u, 0u, 0u);
    // the listed candidates: the first kSaCand of the part's
    const uint32_t n_cand = min(ms->ncand, (uint32_t)kSaCand);
    uint32_t* fbk = hist0;             // final-bin keys pushed by the cluster (hist0 is done with)
    uint32_t* fbp = hist0 + kSaFb;     // and their positions in the row
    bool fallback = !trivial && ms->ovf != 0u;

    // ---- digit 1 (bits 20..10) from the cluster's sum; candidates above its bin join the
    // selection, those in it (the final bin) are pushed to every CTA with this part's count
    // of entries above the final bin
    uint32_t pre21 = 0;
    if (!trivial && !fallback) {
        // the coarse group holding the krem-th largest, then its 32 fine bins summed over the
        // cluster (one round of remote reads)
        uint32_t* ctot = reinterpret_cast<uint32_t*>(lst);  // lst is free until the final-bin list
        if (tid < kSaCoarse) {
            uint32_t t = 0;
            for (int c = 0; c < P; ++c) t += coarse[c * kSaCoarse + tid];
            ctot[tid] = t;
        }
        if (tid == 0) {
            ms->sel_digit = 0;
            ms->sel_above = 0;
        }
        __syncthreads();
        if (warp == 0) {
            const uint32_t ga = ctot[kSaCoarse - 1 - 2 * lane], gb = ctot[kSaCoarse - 2 - 2 * lane];
            const uint32_t incl = warp_inclusive_scan(ga + gb), excl = incl - ga - gb;
            const uint32_t cross = __ballot_sync(0xffffffffu, excl < krem && krem <= incl);
            if (cross != 0u) {
                const int src = __ffs(cross) - 1;
                uint32_t G = 0, aboveG = 0;
                if (lane == src) {
                    const bool first = excl + ga >= krem;
                    G = (uint32_t)(kSaCoarse - 1 - 2 * lane - (first ? 0 : 1));
                    aboveG = first ? excl : excl + ga;
                }
                G = __shfl_sync(0xffffffffu, G, src);
                aboveG = __shfl_sync(0xffffffffu, aboveG, src);
                const uint32_t bin = G * (kSaHist / kSaCoarse) + 31u - (uint32_t)lane;  // from the top
                uint32_t f = 0;
                for (int c = 0; c < P; ++c) f += cl.map_shared_rank(hist1, c)[bin];
                const uint32_t fi = warp_inclusive_scan(f) + aboveG, fe = fi - f;
                const uint32_t fc = __ballot_sync(0xffffffffu, fe < krem && krem <= fi);
                if (fc != 0u && lane == __ffs(fc) - 1) {
                    ms->sel_digit = bin;
                    ms->sel_above = fe;
                }
            }
        }
        __syncthreads();
        const uint32_t d1 = ms->sel_digit & (kSaHist - 1), ab1 = ms->sel_above;
        krem -= ab1;
        pre21 = (d0 << 11) | d1;
        for (uint32_t cb = (uint32_t)(tid - lane); cb < n_cand; cb += kSaThreads) {  // warp-uniform bounds
            const uint32_t c = cb + (uint32_t)lane;
            bool up = false;
            if (c < n_cand) {
                const uint32_t ck = cand_k[c], ci = cand_i[c], dg = (ck >> 10) & (kSaHist - 1);
                if (dg > d1) {
                    atomicOr(&sel[ci >> 5], 1u << (ci & 31));
                    up = true;
                } else if (dg == d1) {
                    const uint32_t q = atomicAdd(&ms->nfb, 1u);
                    if (q < (uint32_t)kSaList) lst[q] = c;
                }
            }
            const uint32_t nu = (uint32_t)__popc(__ballot_sync(0xffffffffu, up));
            if (lane == 0 && nu != 0u) atomicAdd(&ms->nabove, nu);
        }
        __syncthreads();
        const uint32_t total = ms->nabove;  // this part's entries above the final bin
        const uint32_t nfb = min(ms->nfb, (uint32_t)kSaList);
        if (tid < P) {
            SaMisc* rm = cl.map_shared_rank(ms, tid);
            // a list longer than this CTA keeps pushes the cluster's total past the buffer
            ms->fb_off[tid] = atomicAdd(&rm->fb_n, ms->nfb > (uint32_t)kSaList ? (uint32_t)kSaFb + 1u : ms->nfb);
            rm->dsure[rank] = total;
        }
        __syncthreads();
        for (uint32_t q = tid; q < nfb; q += kSaThreads) {
            const int c = lst[q];
            const uint32_t key = cand_k[c], pos = (uint32_t)p0 + cand_i[c];
            for (int t = 0; t < P; ++t) {
                const uint32_t slot = ms->fb_off[t] + q;
                if (slot < (uint32_t)kSaFb) {
                    cl.map_shared_rank(fbk, t)[slot] = key;
                    cl.map_shared_rank(fbp, t)[slot] = pos;
                }
            }
        }
    }
    cl.sync();  // B2: every CTA holds the row's final-bin entries and the parts' counts above it
    if (!trivial && !fallback && ms->fb_n > (uint32_t)kSaFb) fallback = true;  // same in every CTA

    uint32_t thr = 0, base = 0, take = 0, my_gt = 0, my_eq = 0;
    if (!trivial && !fallback) {
        // ---- the threshold key: the krem-th largest among the final-bin entries
        const uint32_t n_fb = ms->fb_n;
        if (tid < kSaMaxCluster) {
            ms->cgt[tid] = tid < P ? ms->dsure[tid] : 0u;
            ms->ceq[tid] = 0u;
        }
        if (n_fb <= 32u) {
            // few entries (the usual case): one warp ranks them by key, then position (all
            // distinct); the entry ranked krem - 1 holds the threshold key
            if (warp == 0) {
                const bool have = (uint32_t)lane < n_fb;
                const uint32_t ky = have ? fbk[lane] : 0u, ps = have ? fbp[lane] : 0xffffffffu;
                uint32_t rk = 0u;
                for (uint32_t j = 0; j < n_fb; ++j) {
                    const uint32_t kj = __shfl_sync(0xffffffffu, ky, (int)j);
                    const uint32_t pj = __shfl_sync(0xffffffffu, ps, (int)j);
                    rk += (kj > ky || (kj == ky && pj < ps)) ? 1u : 0u;
                }
                const uint32_t hit = __ballot_sync(0xffffffffu, have && rk + 1u == krem);
                const uint32_t tk = __shfl_sync(0xffffffffu, ky, hit != 0u ? __ffs(hit) - 1 : 0);
                const uint32_t ngt = (uint32_t)__popc(__ballot_sync(0xffffffffu, have && ky > tk));
                if (lane == 0) {
                    ms->sel_digit = tk;
                    ms->sel_above = ngt;
                }
            }
            __syncthreads();
            thr = ms->sel_digit;
            krem -= ms->sel_above;
        } else {
            // digit 2 (bits 9..0) of the final-bin entries
            for (int i = tid; i < kSaHist / 2; i += kSaThreads) hist2[i] = 0u;
            __syncthreads();
            for (uint32_t e = tid; e < n_fb; e += kSaThreads) atomicAdd(&hist2[fbk[e] & 1023u], 1u);
            __syncthreads();
            uint32_t d2, ab2;
            cta_select_digit(hist2, kSaHist / 2, krem, ms, d2, ab2);
            d2 &= 1023u;
            krem -= ab2;
            thr = (pre21 << 10) | d2;
        }
        // ---- every part's counts above / equal to the threshold, from the final bin
        for (uint32_t e = tid; e < n_fb; e += kSaThreads) {
            const uint32_t key = fbk[e], r = min(fbp[e] / (uint32_t)p.part, (uint32_t)(P - 1));
            if (key > thr) atomicAdd(&ms->cgt[r], 1u);
            else if (key == thr) atomicAdd(&ms->ceq[r], 1u);
        }
        __syncthreads();
        // ---- the final-bin entries of this part above the threshold join the selection, those
        // equal to it are ties
        for (uint32_t e = tid; e < n_fb; e += kSaThreads) {
            const uint32_t pos = fbp[e];
            if (pos < (uint32_t)p0 || pos >= (uint32_t)p1) continue;
            const uint32_t li = pos - (uint32_t)p0;
            if (fbk[e] > thr) atomicOr(&sel[li >> 5], 1u << (li & 31));
            else if (fbk[e] == thr) atomicOr(&tie[li >> 5], 1u << (li & 31));
        }
        my_gt = ms->cgt[rank];
        my_eq = ms->ceq[rank];
    } else if (fallback) {
        thr = sa_fallback_threshold(srow, N, p.part, P, d0, krem0, hist0, ms, krem);
        my_gt = ms->cgt[rank];
        my_eq = ms->ceq[rank];
    } else if (k == N) {
        my_gt = (uint32_t)np;
        for (int c = tid; c < P; c += kSaThreads) ms->cgt[c] = (uint32_t)min(p.part, N - c * p.part);
        if (tid < kSaMaxCluster) ms->ceq[tid] = 0u;
        __syncthreads();
    } else if (tid < kSaMaxCluster) {  // k == 0
        ms->cgt[tid] = ms->ceq[tid] = 0u;
    }
    __syncthreads();

    // ---- this CTA's ties and its offset in the row's ascending output
    {
        uint32_t eq_before = 0;
        for (int c = 0; c < rank; ++c) {
            const uint32_t ec = ms->ceq[c];
            const uint32_t tc = krem > eq_before ? min(ec, krem - eq_before) : 0u;
            base += ms->cgt[c] + tc;
            eq_before += ec;
        }
        take = krem > eq_before ? min(my_eq, krem - eq_before) : 0u;
    }
    const uint32_t n_mine = base >= (uint32_t)k ? 0u : min(my_gt + take, (uint32_t)k - base);
    auto put = [&](uint32_t at, int pos) {  // at < n_mine
        orow[base + at] = pos;
        if (at < (uint32_t)kSaList) lst[at] = pos;
    };
    __syncthreads();  // lst is rewritten below

    // ---- ordered emit of this part's selection into idx[base, base + n_mine)
    if (k == N) {
        for (int i = tid; i < np; i += kSaThreads) put((uint32_t)i, p0 + i);
    } else if (!trivial && !fallback) {
        // one scan gives each thread the selected and tied entries before its words
        const int W = (nw + kSaThreads - 1) / kSaThreads;  // words per thread
        const int w0 = tid * W, w1 = min(nw, w0 + W);
        uint32_t cs = 0, ct = 0;
        for (int w = w0; w < w1; ++w) {
            cs += __popc(sel[w]);
            ct += __popc(tie[w]);
        }
        uint32_t tot_s, tot_t, sel_before, tie_before;
        cta_exclusive_scan2(cs, ct, ms, sel_before, tie_before, tot_s, tot_t);
        uint32_t ties_left = take > tie_before ? take - tie_before : 0u;
        uint32_t at = sel_before + min(tie_before, take);
        for (int w = w0; w < w1; ++w) {
            uint32_t bits = sel[w], tb = tie[w];
            while (tb != 0u && ties_left > 0u) {  // the lowest-index ties still needed
                const uint32_t low = tb & (0u - tb);
                bits |= low;
                tb ^= low;
                --ties_left;
            }
            while (bits != 0u) {
                const int bpos = __ffs(bits) - 1;
                bits &= bits - 1u;
                if (at < n_mine) put(at, p0 + w * 32 + bpos);
                ++at;
            }
        }
    } else if (!trivial) {
        sa_emit_ordered(staged ? keys_s : nullptr, srow, p0, p1, thr, take, n_mine, ms, orow + base, lst);
    }
    if (!p.attend) {  // selection only: no CTA leaves while the cluster may still read it
        cl.sync();
        return;
    }
    cp_async_wait<0>();  // query rows
    __syncthreads();     // the selection list is complete (shared memory and idx)

    // ---- attention over this CTA's selected rows, kSaWin list rows at a time
    int32_t* src = reinterpret_cast<int32_t*>(sm + L.oSrc);
    RowSource rs;
    rs.k_pool = p.kc + (size_t)bk * p.pool_rows * (D * 2);
    rs.v_pool = p.vc + (size_t)bk * p.pool_rows * (D * 2);
    rs.k_host = p.kh + (size_t)bk * p.T * (D * 2);
    rs.v_host = p.vh + (size_t)bk * p.T * (D * 2);
    const int n_list = (int)n_mine * p.block;  // this CTA's rows, list rows [base*block, +n_list)
    const int list0 = (int)base * p.block, n_all = k * p.block;
    float* lbase = nullptr;
    if (p.logits != nullptr) lbase = p.logits + ((size_t)b * p.V * p.Hq + kvh * p.G) * n_all + list0;
    WarpAcc<D, RP> acc;
    acc.init();
    for (int w0 = 0; w0 < n_list; w0 += kSaWin) {
        const int nwin = min(kSaWin, n_list - w0);
        for (int j = tid; j < nwin; j += kSaThreads) {
            const int jl = w0 + j, e = jl / p.block;
            const int selv = e < kSaList ? lst[e] : orow[base + e];
            const int pos = selv * p.block + jl % p.block;
            int32_t code = pos;
            if (selv < 0 || selv >= N) {  // only with a histogram that does not match the scores
                report(p.err, SD_DEVERR_INDEX);
                code = kNoRow;
            } else if (p.slot_map != nullptr) {
                const int slot = p.slot_map[(size_t)(p.slot_per_head ? bk : b) * p.T + pos];
                if (slot >= 0 && slot < p.pool_rows) {
                    code = slot;
                } else if (slot == -1) {
                    code = -1 - pos;
                } else {
                    report(p.err, SD_DEVERR_SLOT);
                    code = kNoRow;
                }
            }
            src[j] = code;
        }
        __syncthreads();
        auto row_code = [&](int j) -> int32_t { return src[j]; };
        auto logit = [&](int r, int j, float x) {
            if (lbase != nullptr && r < p.R) {
                const int v = r / p.G, gg = r % p.G;
                lbase[((size_t)v * p.Hq + gg) * n_all + w0 + j] = x * kLn2f;
            }
        };
        mma_attend_warp<D, RP>(acc, sm + L.oU + warp * Rows::kWarpBytes, smem_addr(sm + L.oQ), warp, nwin, p.R, rs,
                               p.scale_log2, row_code, logit);
        __syncthreads();  // src is rewritten by the next window
    }

    // ---- this CTA's partial (m, l, O), pushed into the inbox of each query row's owner
    float* mlw = reinterpret_cast<float*>(sm + L.oML);
    float* rowv = reinterpret_cast<float*>(sm + L.oRow);
    float* ow = reinterpret_cast<float*>(sm + L.oU);
    mma_combine_warps<D, RP>(acc, mlw, rowv, ow, p.R);
    const int R = p.R;
    const int own = (R + P - 1) / P;  // query rows per owner
    // the inbox either has its own memory, or reuses H once every CTA is past its selection
    if (!p.inbox_own) cl.sync();  // B3: every CTA has finished its selection and attention
    float* inO = reinterpret_cast<float*>(sm + (p.inbox_own ? L.bytes : L.oH));  // [own][P][D]
    float* inM = inO + own * P * D;                      // [own][P]
    float* inL = inM + own * P;                          // [own][P]
    for (int e = tid; e < R * (D / 4); e += kSaThreads) {
        const int r = e / (D / 4), col = (e % (D / 4)) * 4;
        const int owner = r % P, lr = r / P;
        const float4 o = mma_cta_row4<D, RP>(ow, r, col);
        float* dO = cl.map_shared_rank(inO, owner);
        *reinterpret_cast<float4*>(dO + ((size_t)lr * P + rank) * D + col) = o;
        if (col == 0) {
            cl.map_shared_rank(inM, owner)[lr * P + rank] = rowv[r];
            cl.map_shared_rank(inL, owner)[lr * P + rank] = rowv[RP + r];
        }
    }
    cl.sync();  // B4: every inbox is complete; no shared memory is read across CTAs after this

    // ---- merge this CTA's query rows r = lr * P + rank over the P partials
    for (int e = tid; e < own * (D / 4); e += kSaThreads) {
        const int lr = e / (D / 4), col = (e % (D / 4)) * 4;
        const int r = lr * P + rank;
        if (r >= R) continue;
        float M = -INFINITY;
        for (int s = 0; s < P; ++s) M = fmaxf(M, inM[lr * P + s]);
        float Ls = 0.f;
        float4 o = make_float4(0.f, 0.f, 0.f, 0.f);
        for (int s = 0; s < P; ++s) {
            const float ms_ = inM[lr * P + s];
            if (M == -INFINITY || ms_ == -INFINITY) continue;
            const float wgt = exp2f(ms_ - M);
            Ls = fmaf(inL[lr * P + s], wgt, Ls);
            const float4 x = *reinterpret_cast<const float4*>(inO + ((size_t)lr * P + s) * D + col);
            o.x = fmaf(wgt, x.x, o.x);
            o.y = fmaf(wgt, x.y, o.y);
            o.z = fmaf(wgt, x.z, o.z);
            o.w = fmaf(wgt, x.w, o.w);
        }
        const float inv = Ls > 0.f ? 1.f / Ls : 0.f;
        const int v = r / p.G, gg = r % p.G;
        const size_t qrow = ((size_t)b * p.V + v) * p.Hq + kvh * p.G + gg;
        *reinterpret_cast<float4*>(p.out + qrow * D + col) = make_float4(o.x * inv, o.y * inv, o.z * inv, o.w * inv);
        if (col == 0) p.lse[qrow] = Ls > 0.f ? (M + log2f(Ls)) * kLn2f : -INFINITY;
    }
}

struct SaPlan {
    int P, part, staged, RP, smem;
};

SaPlan plan_for(int N, int D, int RP, int P, bool scores_aligned) {
    SaPlan pl{};
    pl.RP = RP;
    P = std::max(1, std::min(P, kSaMaxCluster));
    P = std::min(P, std::max(1, (N + 255) / 256));
    int part = (N + P - 1) / P;
    part = std::max(kSaPartAlign, (part + kSaPartAlign - 1) / kSaPartAlign * kSaPartAlign);
    pl.P = std::max(1, (N + part - 1) / part);
    pl.part = part;
    const int stages = kMmaWarps * kWStages * 2 * kSub * (D * 2 + 16);
    pl.staged = (scores_aligned && N % 4 == 0 && part * 4 <= stages) ? 1 : 0;
    pl.smem = sa_layout(D, RP, part, pl.staged).bytes;
    return pl;
}

// Clusters of `P` CTAs with `smem` bytes each that the current device runs at once
// (queried once per device and shape, then cached).
template <int D, int RP>
int max_active_clusters(int P, int smem) {
    static std::mutex mu;
    static std::map<std::tuple<int, int, int>, int> cache;
    int dev = 0;
    cudaGetDevice(&dev);
    const auto key = std::make_tuple(dev, P, smem);
    {
        std::lock_guard<std::mutex> g(mu);
        auto it = cache.find(key);
        if (it != cache.end()) return it->second;
    }
    auto kern = select_attend_kernel<D, RP>;
    int n = 0;
    if (cudaFuncSetAttribute(kern, cudaFuncAttributeMaxDynamicSharedMemorySize, smem) == cudaSuccess) {
        cudaLaunchConfig_t cfg{};
        cfg.gridDim = dim3(P, 1, 1);
        cfg.blockDim = dim3(kSaThreads);
        cfg.dynamicSmemBytes = smem;
        cudaLaunchAttribute attr[1];
        attr[0].id = cudaLaunchAttributeClusterDimension;
        attr[0].val.clusterDim.x = P;
        attr[0].val.clusterDim.y = 1;
        attr[0].val.clusterDim.z = 1;
        cfg.attrs = attr;
        cfg.numAttrs = 1;
        if (cudaOccupancyMaxActiveClusters(&n, kern, &cfg) != cudaSuccess) n = 0;
    }
    cudaGetLastError();
    std::lock_guard<std::mutex> g(mu);
    cache[key] = n;
    return n;
}

// Cluster size: the caller's, or the largest P <= 8 (parts of at least 256 scores) whose
// rows * P CTAs all run at once on this GPU with room to spare; P = 1 when even single
// CTAs need several waves.
template <int D, int RP>
SaPlan plan_select_attend(int rows, int N, int requested, bool scores_aligned) {
    if (requested > 0) return plan_for(N, D, RP, requested, scores_aligned);
    for (int P = kSaMaxCluster; P > 1; --P) {
        const SaPlan pl = plan_for(N, D, RP, P, scores_aligned);
        if (pl.P != P) continue;  // N too short for P parts
        // keep a tenth of the clusters' room free: a programmatic launch places clusters while
        // the preceding kernel still holds SMs, and a full GPU would leave one for a second wave
        if (rows * 10 <= max_active_clusters<D, RP>(P, pl.smem) * 9) return pl;
    }
    return plan_for(N, D, RP, 1, scores_aligned);
}

template <int D, int RP>
sd_status launch_select_attend(SelAttParams p, int rows, int requested, bool scores_aligned, cudaStream_t st) {
    const SaPlan pl = plan_select_attend<D, RP>(rows, p.N, requested, scores_aligned);
    if (sa_inbox_bytes(D, p.R, pl.P) > kSaHBytes) {
        set_error("sd_select_attend: merge inbox does not fit (R=%d, P=%d)", p.R, pl.P);
        return SD_ERR_UNSUPPORTED;
    }
    p.part = pl.part;
    p.staged = pl.staged;
    // a separate inbox saves a cluster barrier when two CTAs per SM still fit
    const int inbox = sa_inbox_bytes(D, p.R, pl.P);
    p.inbox_own = pl.smem + inbox <= kSaTwoPerSm ? 1 : 0;
    const int smem = pl.smem + (p.inbox_own ? inbox : 0);
    auto kern = select_attend_kernel<D, RP>;
    SD_CUDA_CHECK(cudaFuncSetAttribute(kern, cudaFuncAttributeMaxDynamicSharedMemorySize, smem),
                  "sd_select_attend: cudaFuncSetAttribute");
    cudaLaunchConfig_t cfg{};
    cfg.gridDim = dim3(pl.P, p.Hkv, p.B);
    cfg.blockDim = dim3(kSaThreads);
    cfg.dynamicSmemBytes = smem;
    cfg.stream = st;
    cudaLaunchAttribute attr[2];
    attr[0].id = cudaLaunchAttributeClusterDimension;
    attr[0].val.clusterDim.x = pl.P;
    attr[0].val.clusterDim.y = 1;
    attr[0].val.clusterDim.z = 1;
    attr[1].id = cudaLaunchAttributeProgrammaticStreamSerialization;
    attr[1].val.programmaticStreamSerializationAllowed = 1;
    cfg.attrs = attr;
    cfg.numAttrs = 2;
    SD_CUDA_CHECK(cudaLaunchKernelEx(&cfg, kern, p), "sd_select_attend: launch");
    return launch_status("sd_select_attend");
}

}  // namespace

// sd_topk's path for few long rows: the cluster kernel's selection alone, one cluster of
// P >= 2 CTAs per row.  Returns false (nothing launched) when the rows are too many for
// clusters of two or more CTAs to run in one wave; the caller then uses its own kernel.
bool topk_by_clusters(const float* scores, int rows, int N, int k, int32_t* idx, uint32_t* key_hist,
                      cudaStream_t st, sd_status* status) {
    if (rows <= 0 || rows > 65535 || k <= 0 || k >= N) return false;
    const bool al = aligned16(scores);
    const SaPlan pl = plan_select_attend<128, 16>(rows, N, 0, al);
    if (pl.P < 2) return false;
    SelAttParams p{};
    p.scores = scores;
    p.key_hist = key_hist;
    p.idx = idx;
    p.N = N;
    p.k = k;
    p.B = 1;
    p.Hkv = rows;
    p.V = 1;
    p.Hq = rows;
    p.G = 1;
    p.R = 1;
    p.T = N;
    p.block = 1;
    p.attend = 0;
    *status = launch_select_attend<128, 16>(p, rows, 0, al, st);
    return true;
}

}  // namespace sd

using namespace sd;

extern "C" sd_status sd_select_attend(const float* scores, int N, uint32_t* key_hist, int32_t* idx,
                                      const sd_attend_args* a, void* stream) {
    clear_error();
    SD_REQUIRE(a != nullptr, "sd_select_attend: null args");
    SD_REQUIRE(a->B >= 0 && a->V >= 1 && a->Hq >= 1 && a->Hkv >= 1 && a->T >= 0 && N >= 0,
               "sd_select_attend: bad sizes (B=%d V=%d Hq=%d Hkv=%d T=%d N=%d)", a->B, a->V, a->Hq, a->Hkv, a->T, N);
    SD_REQUIRE(a->Hq % a->Hkv == 0, "sd_select_attend: Hq must be a multiple of Hkv");
    SD_REQUIRE(a->block >= 1 && (long)N * a->block == a->T,
               "sd_select_attend: N * block (%d * %d) must equal T (%d)", N, a->block, a->T);
    const int k = a->n_idx;
    SD_REQUIRE(k >= 0 && k <= N, "sd_select_attend: n_idx (%d) must be in [0, N=%d]", k, N);
    SD_REQUIRE(a->B <= 65535 && a->Hkv <= 65535, "sd_select_attend: B and Hkv must be <= 65535");
    if (a->dtype != SD_BF16 || (a->d != 64 && a->d != 128)) {
        set_error("sd_select_attend: needs bf16 q/K/V with d 64 or 128 (use sd_topk + sd_gather_attend)");
        return SD_ERR_UNSUPPORTED;
    }
    const int R = (a->Hq / a->Hkv) * a->V;
    if (R > 32) {
        set_error("sd_select_attend: G*V = %d exceeds 32", R);
        return SD_ERR_UNSUPPORTED;
    }
    SD_REQUIRE(a->splits >= 0 && a->splits <= kSaMaxCluster, "sd_select_attend: splits must be in [0, 8]");
    if (a->per_head) {
        set_error("sd_select_attend: per-head selections go through sd_topk + sd_gather_attend");
        return SD_ERR_UNSUPPORTED;
    }
    SD_REQUIRE(a->T < kRingBase && a->pool_rows < kRingBase, "sd_select_attend: T and pool_rows must be < 2^30");
    if (a->ring_w != 0) {
        set_error("sd_select_attend: a draft ring goes through sd_topk + sd_gather_attend");
        return SD_ERR_UNSUPPORTED;
    }
    if (a->tier != nullptr) {
        set_error("sd_select_attend: tiered rows go through sd_topk + sd_gather_attend");
        return SD_ERR_UNSUPPORTED;
    }
    if (a->B == 0) return SD_OK;
    SD_REQUIRE(scores && a->q && a->out && a->lse && (k == 0 || idx), "sd_select_attend: null pointer");
    SD_REQUIRE(aligned16(a->q) && aligned16(a->out), "sd_select_attend: q and out must be 16-byte aligned");
    SD_REQUIRE(key_hist == nullptr || aligned16(key_hist), "sd_select_attend: key_hist must be 16-byte aligned");
    SelAttParams p{};
    p.scores = scores;
    p.key_hist = key_hist;
    p.idx = idx;
    p.N = N;
    p.k = k;
    p.q = a->q;
    p.kc = static_cast<const uint8_t*>(a->k_cache);
    p.vc = static_cast<const uint8_t*>(a->v_cache);
    p.slot_map = a->slot_map;
    p.B = a->B;
    p.V = a->V;
    p.Hq = a->Hq;
    p.Hkv = a->Hkv;
    p.G = a->Hq / a->Hkv;
    p.R = R;
    p.T = a->T;
    p.block = a->block;
    p.scale_log2 = a->scale * 1.44269504088896340736f;
    p.out = a->out;
    p.lse = a->lse;
    p.logits = a->logits;
    p.err = a->err_word;
    p.attend = 1;
    p.slot_per_head = a->slot_per_head;
    SD_REQUIRE(a->slot_per_head == 0 || a->slot_per_head == 1, "sd_select_attend: slot_per_head must be 0 or 1");
    if (a->slot_map != nullptr) {
        SD_REQUIRE(a->pool_rows >= 0, "sd_select_attend: pool_rows must be >= 0");
        SD_REQUIRE(a->k_host && a->v_host, "sd_select_attend: slot_map needs k_host and v_host");
        p.kh = mapped_host_ptr(a->k_host);
        p.vh = mapped_host_ptr(a->v_host);
        SD_REQUIRE(p.kh && p.vh, "sd_select_attend: k_host/v_host must be pinned, mapped host memory");
        SD_REQUIRE(aligned16(a->k_host) && aligned16(a->v_host), "sd_select_attend: host K/V must be 16-byte aligned");
        p.pool_rows = a->pool_rows;
    } else {
        p.pool_rows = a->T;
    }
    if (k > 0 && (a->slot_map == nullptr || a->pool_rows > 0)) {
        SD_REQUIRE(a->k_cache && a->v_cache, "sd_select_attend: null k_cache/v_cache");
        SD_REQUIRE(aligned16(a->k_cache) && aligned16(a->v_cache),
                   "sd_select_attend: k_cache/v_cache must be 16-byte aligned");
    }
    const int rows = a->B * a->Hkv;
    const bool al = aligned16(scores);
    cudaStream_t st = as_stream(stream);
    if (a->d == 128)
        return R <= 16 ? launch_select_attend<128, 16>(p, rows, a->splits, al, st)
                       : launch_select_attend<128, 32>(p, rows, a->splits, al, st);
    return R <= 16 ? launch_select_attend<64, 16>(p, rows, a->splits, al, st)
                   : launch_select_attend<64, 32>(p, rows, a->splits, al, st);
}
