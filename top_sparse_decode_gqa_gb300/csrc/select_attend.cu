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
// part [c*part, (c+1)*part) of the row's N scores:
//   1. the row's top digit (11 bits of the order key) comes from the indexer's histogram;
//      one pass over the part marks every entry above it in a bitmap, keeps the entries of
//      that digit as candidates and counts their next digit;
//   2. the next two digits are resolved over the candidates, each CTA summing the P
//      histograms through distributed shared memory (DSMEM), so every CTA finds the same
//      threshold key and the same number of ties still needed;
//   3. the P (above, equal) counts give each CTA its ties (lowest indices first) and its
//      offset in the row's ascending output; it writes its selected indices there;
//   4. the CTA then attends over its own selected rows with the warp-MMA loop of
//      attend_mma.cuh (all G*V query rows of the group per fetched row);
//   5. the P partial (m, l, O) are merged through DSMEM, each CTA finishing every P-th
//      output column group.
// When a CTA's candidates overflow its buffer, the cluster resolves the digits and the
// ordered emit over the keys themselves instead (same result, more passes).
#include <cooperative_groups.h>

#include <algorithm>

#include "attend_mma.cuh"
#include "sd_common.cuh"
#include "sd_host.h"

namespace cg = cooperative_groups;

namespace sd {
namespace {

constexpr int kSaThreads = kMmaWarps * 32;
constexpr int kSaWarps = kMmaWarps;
constexpr int kSaHist = 2048;      // bins of the 11-bit digits
constexpr int kSaCand = 1024;      // candidates a CTA keeps
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
};

// Shared-memory layout.  Phase-A buffers (histograms, bitmaps, candidates) and phase-B
// buffers (row sources, warp and row statistics, merge weights) share one region: phase B
// starts after the last barrier at which another CTA reads a phase-A buffer.
struct SaLayout {
    int oQ, oU, oA, oHist0, oHist1, oHist2, oSel, oTie, oCandK, oCandI;
    int oSrc, oML, oRow, oW, oMisc, bytes;
};

__host__ __device__ constexpr int sa_align(int x, int a) { return (x + a - 1) / a * a; }

__host__ __device__ inline SaLayout sa_layout(int D, int RP, int part, int staged) {
    SaLayout L{};
    const int row_b = D * 2 + 16;
    const int stages = kMmaWarps * kWStages * 2 * kSub * row_b;
    L.oQ = 0;
    L.oU = sa_align(RP * row_b, 128);
    const int u = sa_align(staged && part * 4 > stages ? part * 4 : stages, 128);
    L.oA = L.oU + u;
    // phase A
    L.oHist0 = L.oA;
    L.oHist1 = L.oHist0 + kSaHist * 4;
    L.oHist2 = L.oHist1 + kSaHist * 4;
    L.oSel = L.oHist2 + (kSaHist / 2) * 4;
    L.oTie = L.oSel + part / 8;
    L.oCandK = L.oTie + part / 8;
    L.oCandI = L.oCandK + kSaCand * 4;
    const int end_a = L.oCandI + kSaCand * 4;
    // phase B
    L.oSrc = L.oA;
    L.oML = L.oSrc + kSaWin * 4;
    L.oRow = L.oML + 2 * kMmaWarps * RP * 4;
    L.oW = L.oRow + 6 * RP * 4;
    const int end_b = L.oW + (kSaMaxCluster + 1) * RP * 4;
    L.oMisc = sa_align(end_a > end_b ? end_a : end_b, 16);
    L.bytes = L.oMisc + 128;
    return L;
}

// Values a CTA publishes to its cluster (at the start of the misc area).
struct SaMisc {
    uint32_t n_cand;   // candidates seen (may exceed kSaCand)
    uint32_t gt, eq;   // entries above / equal to the threshold key
    uint32_t pad0;
    uint32_t wgt[kSaWarps], weq[kSaWarps];  // per-warp counts of the ordered emit
    uint32_t wsum[kSaWarps];
    uint32_t sel_digit, sel_above;
    uint64_t bar;
};

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

// Given the histogram of one digit (nb bins, higher bins = larger keys) of the entries
// still in the running, the digit holding the krem-th largest and how many entries lie in
// higher bins.  Thread t owns bins [nb - per*(t+1), nb - per*t).  If no bin crosses (a
// histogram that does not match the scores) the answer is digit 0, 0 above.
SD_DEVINL void cta_select_digit(const uint32_t* hist, int nb, uint32_t krem, SaMisc* ms, uint32_t& digit,
                                uint32_t& above) {
    const int tid = threadIdx.x;
    if (tid == 0) {
        ms->sel_digit = 0;
        ms->sel_above = 0;
    }
    const int per = nb / kSaThreads;
    const int hi = nb - per * tid;
    uint32_t local = 0;
    for (int b = hi - per; b < hi; ++b) local += hist[b];
    const uint32_t incl = cta_inclusive_scan(local, ms->wsum);
    const uint32_t excl = incl - local;
    if (excl < krem && krem <= incl) {
        uint32_t acc = excl;
        for (int b = hi - 1; b >= hi - per; --b) {
            if (acc + hist[b] >= krem) {
                ms->sel_digit = (uint32_t)b;
                ms->sel_above = acc;
                break;
            }
            acc += hist[b];
        }
    }
    __syncthreads();
    digit = ms->sel_digit;
    above = ms->sel_above;
    __syncthreads();
}

// dst[i] = sum over the cluster's P CTAs of their copy of src[i], i < n (n a multiple of
// 4 * kSaThreads is not required; n is a multiple of 4).
SD_DEVINL void cluster_sum_hist(cg::cluster_group& cl, const uint32_t* src, uint32_t* dst, int n, int P) {
    const uint4* rem[kSaMaxCluster];
#pragma unroll
    for (int c = 0; c < kSaMaxCluster; ++c)
        rem[c] = reinterpret_cast<const uint4*>(cl.map_shared_rank(const_cast<uint32_t*>(src), c < P ? c : 0));
    for (int i = threadIdx.x; i < n / 4; i += kSaThreads) {
        uint4 x[kSaMaxCluster];
#pragma unroll
        for (int c = 0; c < kSaMaxCluster; ++c)
            if (c < P) x[c] = rem[c][i];
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

// Block-wide exclusive prefix sum; also returns the total.
SD_DEVINL uint32_t cta_exclusive_scan(uint32_t v, uint32_t* wsum, uint32_t& total) {
    const uint32_t incl = cta_inclusive_scan(v, wsum);
    __shared__ uint32_t tot;
    if ((int)threadIdx.x == kSaThreads - 1) tot = incl;
    __syncthreads();
    total = tot;
    __syncthreads();
    return incl - v;
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
    uint32_t* sel = reinterpret_cast<uint32_t*>(sm + L.oSel);
    uint32_t* tie = reinterpret_cast<uint32_t*>(sm + L.oTie);
    uint32_t* cand_k = reinterpret_cast<uint32_t*>(sm + L.oCandK);
    uint32_t* cand_i = reinterpret_cast<uint32_t*>(sm + L.oCandI);
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

    if (tid == 0) {
        ms->n_cand = 0;
        mbar_init(&ms->bar, 1);
        fence_mbarrier_init();
    }
    for (int i = tid; i < kSaHist; i += kSaThreads) hist1[i] = 0u;
    for (int i = tid; i < kSaHist / 2; i += kSaThreads) hist2[i] = 0u;
    __syncthreads();

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
    for (int e = tid; e < RP * PPR; e += kSaThreads) {
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

    // ---- the top digit's histogram: from the indexer, or counted here and summed
    uint32_t d0 = 0, above0 = 0;
    const bool trivial = (k == 0 || k == N);  // no select needed (every CTA agrees)
    if (hrow != nullptr) {
        for (int i = tid; i < kSaHist / 4; i += kSaThreads)
            reinterpret_cast<uint4*>(hist0)[i] = __ldcg(reinterpret_cast<const uint4*>(hrow) + i);
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
    if (hrow == nullptr && !trivial) {
        // count the top digit of the part into hist1, then sum the cluster's into hist0
        for (int base = p0 + warp * 32; base < p1; base += kSaThreads) {
            const int i = base + lane;
            const bool valid = i < p1;
            const uint32_t dg = valid ? key_at(i) >> 21 : 0xffffffffu;
            const uint32_t peers = __match_any_sync(0xffffffffu, dg);
            if (valid && lane == __ffs(peers) - 1) atomicAdd(&hist1[dg], (uint32_t)__popc(peers));
        }
        cl.sync();
        cluster_sum_hist(cl, hist1, hist0, kSaHist, P);
        cl.sync();  // every CTA has read the others' hist1
        for (int i = tid; i < kSaHist; i += kSaThreads) hist1[i] = 0u;
    }
    __syncthreads();
    if (!trivial) cta_select_digit(hist0, kSaHist, (uint32_t)k, ms, d0, above0);
    d0 &= kSaHist - 1;
    uint32_t krem = (uint32_t)k - above0;

    // ---- one pass over the part: bitmap of entries above d0, candidates of digit d0 and
    // the histogram of their next digit
    if (!trivial) {
        const uint32_t lt = lanemask_lt();
        constexpr int U = 8;
        for (int g0 = warp; g0 < nw; g0 += U * kSaWarps) {
            uint32_t kk[U];
#pragma unroll
            for (int u = 0; u < U; ++u) {
                const int i = p0 + (g0 + u * kSaWarps) * 32 + lane;
                kk[u] = (g0 + u * kSaWarps < nw && i < p1) ? key_at(i) : 0u;
            }
#pragma unroll
            for (int u = 0; u < U; ++u) {
                const int gw = g0 + u * kSaWarps;
                if (gw >= nw) break;
                const int li = gw * 32 + lane;
                const bool valid = p0 + li < p1;
                const uint32_t dg = kk[u] >> 21;
                const uint32_t sure = __ballot_sync(0xffffffffu, valid && dg > d0);
                if (lane == 0) {
                    sel[gw] = sure;
                    tie[gw] = 0u;
                }
                const bool in = valid && dg == d0;
                if (in) atomicAdd(&hist1[(kk[u] >> 10) & (kSaHist - 1)], 1u);
                const uint32_t m = __ballot_sync(0xffffffffu, in);
                if (m != 0u) {
                    const int leader = __ffs(m) - 1;
                    uint32_t at = 0;
                    if (lane == leader) at = atomicAdd(&ms->n_cand, (uint32_t)__popc(m));
                    at = __shfl_sync(0xffffffffu, at, leader);
                    const uint32_t slot = at + __popc(m & lt);
                    if (in && slot < (uint32_t)kSaCand) {
                        cand_k[slot] = kk[u];
                        cand_i[slot] = (uint32_t)li;
                    }
                }
            }
        }
    }
    cl.sync();  // B1: hist1, n_cand published; every CTA has read key_hist
    if (hrow != nullptr && rank == 0)
        for (int i = tid; i < kSaHist / 4; i += kSaThreads) reinterpret_cast<uint4*>(hrow)[i] = make_uint4(0u, 0u, 0u, 0u);
    bool overflow = false;
#pragma unroll
    for (int c = 0; c < kSaMaxCluster; ++c)
        if (c < P) overflow |= cl.map_shared_rank(&ms->n_cand, c)[0] > (uint32_t)kSaCand;
    const uint32_t n_cand = min(ms->n_cand, (uint32_t)kSaCand);

    uint32_t thr = 0;
    uint32_t my_gt = 0, my_eq = 0;
    if (!trivial) {
        // ---- digit 1 (bits 20..10): sum of the cluster's hist1 into hist0
        cluster_sum_hist(cl, hist1, hist0, kSaHist, P);
        __syncthreads();
        uint32_t d1, ab1;
        cta_select_digit(hist0, kSaHist, krem, ms, d1, ab1);
        d1 &= kSaHist - 1;
        krem -= ab1;
        const uint32_t pre21 = (d0 << 11) | d1;
        // ---- digit 2 (bits 9..0) over the entries with those 21 top bits
        if (!overflow) {
            for (uint32_t c = tid; c < n_cand; c += kSaThreads) {
                const uint32_t ck = cand_k[c];
                if ((ck >> 10) == pre21) atomicAdd(&hist2[ck & 1023u], 1u);
            }
        } else {
            for (int base = p0 + warp * 32; base < p1; base += kSaThreads) {
                const int i = base + lane;
                const bool valid = i < p1;
                const uint32_t kk = valid ? key_at(i) : 0u;
                const bool in = valid && (kk >> 10) == pre21;
                const uint32_t peers = __match_any_sync(0xffffffffu, in ? (kk & 1023u) : 0xffffffffu);
                if (in && lane == __ffs(peers) - 1) atomicAdd(&hist2[kk & 1023u], (uint32_t)__popc(peers));
            }
        }
        cl.sync();  // B2: hist2 published; nobody reads hist1 any more
        cluster_sum_hist(cl, hist2, hist1, kSaHist / 2, P);
        __syncthreads();
        uint32_t d2, ab2;
        cta_select_digit(hist1, kSaHist / 2, krem, ms, d2, ab2);
        d2 &= 1023u;
        krem -= ab2;
        thr = (pre21 << 10) | d2;
        // ---- this part's counts above / equal to the threshold
        if (!overflow) {
            uint32_t gt = 0, eq = 0;
            for (int w = tid; w < nw; w += kSaThreads) gt += __popc(sel[w]);
            for (uint32_t c = tid; c < n_cand; c += kSaThreads) {
                gt += cand_k[c] > thr;
                eq += cand_k[c] == thr;
            }
            gt = __reduce_add_sync(0xffffffffu, gt);
            eq = __reduce_add_sync(0xffffffffu, eq);
            if (lane == 0) {
                ms->wgt[warp] = gt;
                ms->weq[warp] = eq;
            }
        } else {
            // warp w scans the contiguous segment [p0 + w*seg, p0 + (w+1)*seg)
            const int seg = ((np + kSaWarps - 1) / kSaWarps + 31) / 32 * 32;
            const int s0 = p0 + warp * seg, s1 = min(p1, s0 + seg);
            uint32_t gt = 0, eq = 0;
            for (int base = s0; base < s1; base += 32) {
                const int i = base + lane;
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
#pragma unroll
        for (int w = 0; w < kSaWarps; ++w) {
            my_gt += ms->wgt[w];
            my_eq += ms->weq[w];
        }
    } else if (k == N) {
        my_gt = (uint32_t)np;
    }
    if (tid == 0) {
        ms->gt = my_gt;
        ms->eq = my_eq;
    }
    cl.sync();  // B3: counts published; nobody reads a histogram any more

    // ---- this CTA's ties and its offset in the row's ascending output
    uint32_t base = 0, take = 0;
    {
        uint32_t eq_before = 0;
        for (int c = 0; c < rank; ++c) {
            const SaMisc* rm = cl.map_shared_rank(ms, c);
            const uint32_t gc = rm->gt, ec = rm->eq;
            const uint32_t tc = krem > eq_before ? min(ec, krem - eq_before) : 0u;
            base += gc + tc;
            eq_before += ec;
        }
        take = krem > eq_before ? min(my_eq, krem - eq_before) : 0u;
    }
    const uint32_t n_mine = base >= (uint32_t)k ? 0u : min(my_gt + take, (uint32_t)k - base);

    // ---- ordered emit of this part's selection into idx[base, base + n_mine)
    if (k == N) {
        for (int i = tid; i < np; i += kSaThreads) orow[p0 + i] = p0 + i;
    } else if (!trivial && !overflow) {
        for (uint32_t c = tid; c < n_cand; c += kSaThreads) {
            const uint32_t ck = cand_k[c], ci = cand_i[c];
            if (ck > thr) atomicOr(&sel[ci >> 5], 1u << (ci & 31));
            else if (ck == thr) atomicOr(&tie[ci >> 5], 1u << (ci & 31));
        }
        __syncthreads();
        const int W = (nw + kSaThreads - 1) / kSaThreads;  // words per thread
        const int w0 = tid * W, w1 = min(nw, w0 + W);
        uint32_t cnt = 0, total;
        for (int w = w0; w < w1; ++w) cnt += __popc(tie[w]);
        uint32_t before = cta_exclusive_scan(cnt, ms->wsum, total);
        for (int w = w0; w < w1; ++w) {
            uint32_t bits = tie[w];
            while (bits != 0u && before < take) {
                const uint32_t low = bits & (0u - bits);
                sel[w] |= low;
                bits ^= low;
                ++before;
            }
        }
        __syncthreads();
        cnt = 0;
        for (int w = w0; w < w1; ++w) cnt += __popc(sel[w]);
        uint32_t at = cta_exclusive_scan(cnt, ms->wsum, total);
        for (int w = w0; w < w1; ++w) {
            uint32_t bits = sel[w];
            while (bits != 0u) {
                const int bpos = __ffs(bits) - 1;
                bits &= bits - 1u;
                if (at < n_mine) orow[base + at] = p0 + w * 32 + bpos;
                ++at;
            }
        }
    } else if (!trivial) {
        const int seg = ((np + kSaWarps - 1) / kSaWarps + 31) / 32 * 32;
        const int s0 = p0 + warp * seg, s1 = min(p1, s0 + seg);
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
            if (pick && at < n_mine) orow[base + at] = i;
            pos += __popc(pm);
            eq_seen += __popc(eqm);
        }
    }
    cp_async_wait<0>();  // query rows
    __syncthreads();     // this CTA's idx entries are visible to all its threads

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
            const int jl = w0 + j;
            const int selv = orow[base + jl / p.block];
            const int pos = selv * p.block + jl % p.block;
            int32_t code = pos;
            if (selv < 0 || selv >= N) {  // only with a histogram that does not match the scores
                report(p.err, SD_DEVERR_INDEX);
                code = kNoRow;
            } else if (p.slot_map != nullptr) {
                const int slot = p.slot_map[(size_t)b * p.T + pos];
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
        mma_attend_warp<D, RP>(acc, sm + L.oU + warp * Rows::kWarpBytes, smem_addr(sm + L.oQ), warp, nwin, rs,
                               p.scale_log2, row_code, logit);
        __syncthreads();  // src is rewritten by the next window
    }

    // ---- this CTA's partial (m, l, O): O summed over the warps into ow[0]
    float* mlw = reinterpret_cast<float*>(sm + L.oML);
    float* rowv = reinterpret_cast<float*>(sm + L.oRow);
    float* ow = reinterpret_cast<float*>(sm + L.oU);
    mma_combine_warps<D, RP>(acc, mlw, rowv, ow);
    for (int e = tid; e < p.R * (D / 4); e += kSaThreads) {
        const int r = e / (D / 4), col = (e % (D / 4)) * 4;
        const float4 o = mma_cta_row4<D, RP>(ow, r, col);
        *reinterpret_cast<float4*>(ow + (size_t)r * D + col) = o;
    }
    cl.sync();  // B4: every CTA's partial is published

    // ---- merge: weights of the P partials per query row, then every P-th column group
    float* wts = reinterpret_cast<float*>(sm + L.oW);  // [P][RP] weight / L, then [RP] lse
    if (tid < p.R) {
        const int r = tid;
        float mc[kSaMaxCluster], lc[kSaMaxCluster];
        float M = -INFINITY;
#pragma unroll
        for (int c = 0; c < kSaMaxCluster; ++c)
            if (c < P) {
                const float* rv = cl.map_shared_rank(rowv, c);
                mc[c] = rv[r];
                lc[c] = rv[RP + r];
                M = fmaxf(M, mc[c]);
            }
        float Ls = 0.f;
#pragma unroll
        for (int c = 0; c < kSaMaxCluster; ++c)
            if (c < P && M != -INFINITY && mc[c] != -INFINITY) Ls = fmaf(lc[c], exp2f(mc[c] - M), Ls);
#pragma unroll
        for (int c = 0; c < kSaMaxCluster; ++c)
            if (c < P) wts[c * RP + r] = (Ls > 0.f && mc[c] != -INFINITY) ? exp2f(mc[c] - M) / Ls : 0.f;
        if (r % P == rank) {
            const int v = r / p.G, gg = r % p.G;
            p.lse[((size_t)b * p.V + v) * p.Hq + kvh * p.G + gg] = Ls > 0.f ? (M + log2f(Ls)) * kLn2f : -INFINITY;
        }
    }
    __syncthreads();
    const float* rem_o[kSaMaxCluster];
#pragma unroll
    for (int c = 0; c < kSaMaxCluster; ++c) rem_o[c] = cl.map_shared_rank(ow, c < P ? c : 0);
    const int items = p.R * (D / 4);
    for (int e = rank + P * tid; e < items; e += P * kSaThreads) {
        const int r = e / (D / 4), col = (e % (D / 4)) * 4;
        float4 x[kSaMaxCluster];
#pragma unroll
        for (int c = 0; c < kSaMaxCluster; ++c)
            if (c < P) x[c] = *reinterpret_cast<const float4*>(rem_o[c] + (size_t)r * D + col);
        float4 o = make_float4(0.f, 0.f, 0.f, 0.f);
#pragma unroll
        for (int c = 0; c < kSaMaxCluster; ++c)
            if (c < P) {
                const float wgt = wts[c * RP + r];
                o.x = fmaf(wgt, x[c].x, o.x);
                o.y = fmaf(wgt, x[c].y, o.y);
                o.z = fmaf(wgt, x[c].z, o.z);
                o.w = fmaf(wgt, x[c].w, o.w);
            }
        const int v = r / p.G, gg = r % p.G;
        const size_t qrow = ((size_t)b * p.V + v) * p.Hq + kvh * p.G + gg;
        *reinterpret_cast<float4*>(p.out + qrow * D + col) = o;
    }
    cl.sync();  // B5: no CTA leaves while another may still read its shared memory
}

struct SaPlan {
    int P, part, staged, RP, smem;
};

// Cluster size and part length: enough CTAs to fill the GPU (two per SM at these shared
// memory sizes), at most 8 per cluster, at least 256 scores per part.
SaPlan plan_select_attend(int rows, int N, int D, int R, int requested, bool scores_aligned) {
    SaPlan pl{};
    pl.RP = R <= 16 ? 16 : 32;
    int P;
    if (requested > 0) {
        P = requested;
    } else {
        const int slots = num_sms() * 2;
        P = rows > 0 ? slots / rows : 1;
    }
    P = std::max(1, std::min(P, kSaMaxCluster));
    P = std::min(P, std::max(1, (N + 255) / 256));
    int part = (N + P - 1) / P;
    part = std::max(kSaPartAlign, (part + kSaPartAlign - 1) / kSaPartAlign * kSaPartAlign);
    pl.P = std::max(1, (N + part - 1) / part);
    pl.part = part;
    const int row_b = D * 2 + 16;
    const int stages = kMmaWarps * kWStages * 2 * kSub * row_b;
    pl.staged = (scores_aligned && N % 4 == 0 && part * 4 <= stages) ? 1 : 0;
    pl.smem = sa_layout(D, pl.RP, part, pl.staged).bytes;
    return pl;
}

template <int D, int RP>
sd_status launch_select_attend(const SelAttParams& p, const SaPlan& pl, cudaStream_t st) {
    auto kern = select_attend_kernel<D, RP>;
    SD_CUDA_CHECK(cudaFuncSetAttribute(kern, cudaFuncAttributeMaxDynamicSharedMemorySize, pl.smem),
                  "sd_select_attend: cudaFuncSetAttribute");
    cudaLaunchConfig_t cfg{};
    cfg.gridDim = dim3(pl.P, p.Hkv, p.B);
    cfg.blockDim = dim3(kSaThreads);
    cfg.dynamicSmemBytes = pl.smem;
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

const uint8_t* mapped_host_ptr(const void* h) {
    cudaPointerAttributes at{};
    if (cudaPointerGetAttributes(&at, h) != cudaSuccess) {
        cudaGetLastError();
        return nullptr;
    }
    if (at.type != cudaMemoryTypeHost || at.devicePointer == nullptr) return nullptr;
    return static_cast<const uint8_t*>(at.devicePointer);
}

}  // namespace
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
    const SaPlan pl = plan_select_attend(a->B * a->Hkv, N, a->d, R, a->splits, aligned16(scores));
    p.part = pl.part;
    p.staged = pl.staged;
    cudaStream_t st = as_stream(stream);
    if (a->d == 128)
        return pl.RP == 16 ? launch_select_attend<128, 16>(p, pl, st) : launch_select_attend<128, 32>(p, pl, st);
    return pl.RP == 16 ? launch_select_attend<64, 16>(p, pl, st) : launch_select_attend<64, 32>(p, pl, st);
}
