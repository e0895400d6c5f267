// block_step.cu -- sd_decode_step for block selection over short score rows: one
// thread-block cluster per KV group runs the group's whole decode step in one launch.
//
// SparDA (gist.science summary), sec. 2 item 1 and "Indexador de Previsao Compacto": the
// indexer scores blocks of the cache by a dot product with one compact key per block, the
// top-k blocks are kept, and attention runs over the tokens of those blocks only.
// "Esparsidade de Contexto no Tempo de Inferencia" (gist.science summary), sec. 2: the
// selection is exact (Oracle top-k); sec. 3C: traffic O(k*block*d) instead of O(T*d).
// Adaptive DHiSparse (news page), "Metodologia": the query rows of a group share every
// fetched row.  Ties go to the lower block index (the pages are silent).
//
// Computes what sd_index_score -> sd_topk -> sd_gather_attend computes (scores and index
// sets bit for bit; attention in its own summation order).  The C CTAs of the cluster of KV
// group g = (b, kvh):
//   1. score: CTA r scores its contiguous share of the group's N block keys (tiled TMA,
//      128 keys per ring stage, mma.sync), into its copy of the group's score row in shared
//      memory and into `scores`;
//   2. select: after a cluster barrier every CTA copies its peers' shares out of their shared
//      memory (distributed shared memory) and runs the same exact radix select (8-bit
//      digits, ties to the lower index), so all hold the same ascending list of k blocks;
//      CTA 0 writes it to `idx`;
//   3. attend: CTA r streams its contiguous share of the list's k*block rows through the
//      ring in 64-row stages of K and V (each block's rows as whole 16- or 32-row runs of
//      tiled TMA, 128-byte swizzle); consumer warps 0-3 each keep their own online softmax
//      over the 32-row halves they take, for all G*V query rows of the group (the transposed
//      tile: keys and output columns on the M side of the mma, the query rows on the N side);
//   4. merge: the four warps' states merge into the CTA's (m, l, O); after a second cluster
//      barrier each CTA merges a slice of the output over the C CTAs' states, in rank order
//      (deterministic), and writes out and lse; a third barrier keeps every CTA's shared
//      memory in place until its peers have read it.
// Warp 4 issues the copies.  No CTA waits on another outside the cluster's own hardware
// barriers, so clusters never wait on each other.  Every mbarrier wait is bounded: one that
// runs out sets SD_DEVERR_TIMEOUT, the CTA stops working but still passes the cluster
// barriers, and it lets its copies in flight land before it exits.
#include <cooperative_groups.h>

#include <algorithm>
#include <cmath>

#include "sd_host.h"
#include "step_tiles.cuh"
#include "tc_common.cuh"

namespace cg = cooperative_groups;

namespace sd {
namespace {

constexpr int kBsCons = 4;                    // consumer warps 0-3
constexpr int kBsProd = kBsCons;              // producer warp 4
constexpr int kBsThreads = 32 * (kBsCons + 1);
constexpr int kBsSlot = 32768;                // ring stage: 128 keys, or 64 K and V rows
constexpr int kBsStageKeys = 128;
constexpr int kBsStageRows = 64;
constexpr int kBsMaxN = 8192;                 // blocks per group this path takes
constexpr int kBsMaxCluster = 8;
constexpr int kBsPartO = 0;                   // after the attention, in the ring: warps' states
constexpr int kBsPartML = kBsCons * 16 * 128 * 4;
static_assert(kBsPartML + kBsCons * 16 * 8 <= 2 * kBsSlot, "the warps' states fit in two ring stages");
// The merge inbox: from each CTA of the cluster, its O for the (query row, 4 columns) items
// this CTA owns (item i on CTA i % C, slot i / C: C * ceil(R*32 / C) <= 16*32 + 7 float4), then
// its (m, l) of every query row (C * 16 float2).
constexpr int kBsInboxBytes = (16 * 32 + kBsMaxCluster) * 16 + kBsMaxCluster * 16 * 8;

struct BsParams {
    const uint8_t* q_idx;  // [NG, V, 128] 16-bit
    const uint8_t* q;      // [B, V, Hq, 128] bf16
    float* scores;         // [NG, N]
    int32_t* idx;          // [NG, k]
    float* out;            // [B, V, Hq, 128]
    float* lse;            // [B, V, Hq]
    int32_t* err;
    int V, Hq, Hkv, G, R, T, N, k, block;
    int br;                // rows per TMA run: min(block, 32)
    int nc;                // keys per CTA share (a multiple of 128)
    int ns;                // ring stages (even)
    int glg, gcnt;         // the selection's group maxima, taken while scoring: groups of
                           // 2^glg keys, gcnt of them (glg = -1: no bound, the radix select)
    int kr, cact;          // each of the cact CTAs holding keys bounds the top kr of its groups
    int oQ, oQi, oScore, oSel, oHist, oScan, oGmax, oInbox, oAux, oBars, oMisc;  // shared memory offsets
    float scale_log2;
    unsigned long long wait_ns;
};

// Exclusive prefix sum of one value per thread over the CTA (kBsThreads), via wt[8].
SD_DEVINL uint32_t bs_scan_excl(uint32_t v, uint32_t* wt) {
    const int lane = threadIdx.x & 31, warp = threadIdx.x >> 5;
    uint32_t x = v;
#pragma unroll
    for (int o = 1; o < 32; o <<= 1) {
        const uint32_t y = __shfl_up_sync(0xffffffffu, x, o);
        if (lane >= o) x += y;
    }
    if (lane == 31) wt[warp] = x;
    __syncthreads();
    uint32_t r = x - v;
    for (int u = 0; u < warp; ++u) r += wt[u];
    __syncthreads();
    return r;
}

// Exact top-k of sc[0 .. N) (1 <= k < N), ties to the lower index: the k indices in
// ascending order into sel[0 .. k).  Radix select on the order-preserving key, 8 bits per
// pass from the top (it stops early once the digit's bin holds exactly the entries still
// needed): each thread loads 8 keys before it counts any, so the loads overlap, and counts
// with plain shared atomics.  Then one ordered pass: thread t owns entries [t*per, t*per +
// per), and two prefix sums give each its first tie rank and its first output slot.
SD_DEVINL void bs_select(const float* sc, int N, int k, int32_t* sel, uint32_t* hist, uint32_t* wt, int* bc) {
    const int tid = threadIdx.x, lane = tid & 31, warp = tid >> 5;
    uint32_t prefix = 0u, pmask = 0u;
    int krem = k;
#pragma unroll 1
    for (int pass = 0; pass < 4; ++pass) {
        const int shift = 24 - 8 * pass;
        for (int i = tid; i < 256; i += kBsThreads) hist[i] = 0u;
        __syncthreads();
        for (int base = tid; base < N; base += 8 * kBsThreads) {
            uint32_t kk[8];
#pragma unroll
            for (int u = 0; u < 8; ++u) {
                const int i = base + u * kBsThreads;
                kk[u] = i < N ? float_key(sc[i]) : 0u;
            }
#pragma unroll
            for (int u = 0; u < 8; ++u) {
                const int i = base + u * kBsThreads;
                if (i < N && (kk[u] & pmask) == prefix) atomicAdd(&hist[(kk[u] >> shift) & 255u], 1u);
            }
        }
        __syncthreads();
        if (warp == 0) {  // lane l owns bins 255 - 8l - j, j < 8 (lane 0 the top ones)
            uint32_t loc = 0u;
#pragma unroll
            for (int j = 0; j < 8; ++j) loc += hist[255 - 8 * lane - j];
            uint32_t x = loc;
#pragma unroll
            for (int o = 1; o < 32; o <<= 1) {
                const uint32_t y = __shfl_up_sync(0xffffffffu, x, o);
                if (lane >= o) x += y;
            }
            uint32_t above = x - loc;
            if (above < (uint32_t)krem && (uint32_t)krem <= above + loc) {
                for (int j = 0; j < 8; ++j) {
                    const int bin = 255 - 8 * lane - j;
                    const uint32_t c = hist[bin];
                    if (above + c >= (uint32_t)krem) {
                        bc[0] = bin;
                        bc[1] = (int)above;
                        bc[2] = (int)c;
                        break;
                    }
                    above += c;
                }
            }
        }
        __syncthreads();
        const uint32_t dg = (uint32_t)bc[0];
        krem -= bc[1];
        prefix |= dg << shift;
        pmask |= 255u << shift;
        if (bc[2] == krem) break;  // every entry left in the bin is taken: no tie to break
    }
    // entries above the prefix, and the first krem equal to it
    const int per = (N + kBsThreads - 1) / kBsThreads;
    const int i0 = tid * per, i1 = min(N, i0 + per);
    uint32_t gt = 0u, eq = 0u;
    for (int i = i0; i < i1; ++i) {
        const uint32_t mk = float_key(sc[i]) & pmask;
        gt += mk > prefix ? 1u : 0u;
        eq += mk == prefix ? 1u : 0u;
    }
    const uint32_t eq_before = bs_scan_excl(eq, wt);
    const uint32_t take = (uint32_t)max(0, min((int)eq, krem - (int)eq_before));
    uint32_t pos = bs_scan_excl(gt + take, wt);
    uint32_t seen = 0u;
    for (int i = i0; i < i1; ++i) {
        const uint32_t mk = float_key(sc[i]) & pmask;
        const bool on = mk > prefix || (mk == prefix && seen++ < take);
        if (on && pos < (uint32_t)k) sel[pos] = i;
        pos += on ? 1u : 0u;
    }
    __syncthreads();
}

constexpr int kBsCandCap = 512;   // candidates of a group, over all the cluster's CTAs
constexpr int kBsMaxGroups = 512;  // group maxima of a group's keys

// The k entries marked in bits[0 .. ceil(N/32)) written ascending into sel[0 .. k): thread t
// owns bitmap words [t*W, t*W + W) and one prefix sum gives its first output slot.
SD_DEVINL void bs_emit_bits(const uint32_t* bits, int N, int k, int32_t* sel, uint32_t* wt) {
    const int tid = threadIdx.x;
    const int NW = (N + 31) / 32;
    const int W = (NW + kBsThreads - 1) / kBsThreads;
    const int w0 = tid * W, w1 = min(NW, w0 + W);
    uint32_t n = 0u;
    for (int w = w0; w < w1; ++w) n += (uint32_t)__popc(bits[w]);
    uint32_t pos = bs_scan_excl(n, wt);
    for (int w = w0; w < w1; ++w) {
        uint32_t b = bits[w];
        while (b != 0u) {
            const int bp = __ffs(b) - 1;
            b &= b - 1u;
            if (pos < (uint32_t)k) sel[pos] = w * 32 + bp;
            ++pos;
        }
    }
    __syncthreads();
}

template <bool F16, int NQ>
__global__ void __launch_bounds__(kBsThreads, 2)
    block_step_kernel(const __grid_constant__ CUtensorMap kmap, const __grid_constant__ CUtensorMap kvk,
                      const __grid_constant__ CUtensorMap kvv, const BsParams p) {
    extern __shared__ uint8_t smem_raw[];
    const uint32_t raw = smem_addr(smem_raw);
    uint8_t* sm = smem_raw + ((1024u - (raw & 1023u)) & 1023u);
    cg::cluster_group cl = cg::this_cluster();
    const int C = (int)cl.num_blocks(), r = (int)cl.block_rank();
    const int g = (int)blockIdx.x / C, b = g / p.Hkv, kvh = g % p.Hkv;
    const int tid = threadIdx.x, warp = tid >> 5, lane = tid & 31;
    uint64_t* full = reinterpret_cast<uint64_t*>(sm + p.oBars);
    uint64_t* empty = full + p.ns;
    uint64_t* qbar = empty + p.ns;  // the query rows
    volatile int* abort_flag = reinterpret_cast<volatile int*>(sm + p.oMisc);
    float* sc = reinterpret_cast<float*>(sm + p.oScore);
    uint32_t* gmx = reinterpret_cast<uint32_t*>(sm + p.oGmax);  // the group maxima, by group
    int32_t* sel = reinterpret_cast<int32_t*>(sm + p.oSel);
    const uint32_t ring = smem_addr(sm);
    const uint64_t lim = p.wait_ns;

    if (tid == 0) {
        for (int s = 0; s < p.ns; ++s) {
            mbar_init(&full[s], 1);   // the producer's arrival with the stage's bytes
            mbar_init(&empty[s], 2);  // the two consumer warps of the stage
        }
        mbar_init(qbar, 1);
        *abort_flag = 0;
        reinterpret_cast<uint32_t*>(sm + p.oAux)[kBsMaxCluster] = 0u;  // this CTA's candidate count
        fence_mbarrier_init();
    }
    __syncthreads();
    // every CTA of the cluster has started before any writes into a peer's shared memory: an
    // arrival now, the wait just before the first such write
    asm volatile("barrier.cluster.arrive.relaxed.aligned;" ::: "memory");
    pdl_wait();  // the inputs are the preceding kernels' results

    // this CTA's shares: keys [j_begin, j_end), attention stages [s0, s1)
    const int j_begin = r * p.nc, j_end = min(p.N, j_begin + p.nc);
    const int n_sc = j_end > j_begin ? (j_end - j_begin + kBsStageKeys - 1) / kBsStageKeys : 0;
    const int n_rows = p.k * p.block;
    const int S = (n_rows + kBsStageRows - 1) / kBsStageRows;
    const int s0 = (int)((long long)r * S / C), s1 = (int)((long long)(r + 1) * S / C);
    const int n_at = s1 - s0;
    const uint64_t pol = l2_evict_first_policy();
    int n_issued = 0;  // stages the producer filled (its lane 0)
    // the next free ring stage for sequence number n (lane 0 of the producer)
    auto take_stage = [&](int n) -> bool {
        if (n < p.ns) return true;
        const int s = n % p.ns;
        if (ds_wait(&empty[s], (uint32_t)((n / p.ns - 1) & 1), abort_flag, lim)) return true;
        *abort_flag = 1;
        return false;
    };

    // ---------------------------------------------------------------- 1. score
    if (warp == kBsProd) {
        if (lane == 0) {
            // the query rows first (they gate the scoring): attention rows v*G + gi, indexer rows
            const uint32_t gb = (uint32_t)p.G * 256u;
            mbar_arrive_expect_tx(qbar, (uint32_t)p.V * (gb + 256u));
            for (int v = 0; v < p.V; ++v)
                bulk_g2s(sm + p.oQ + v * gb, p.q + (((size_t)b * p.V + v) * p.Hq + (size_t)kvh * p.G) * 256, gb, qbar);
            bulk_g2s(sm + p.oQi, p.q_idx + (size_t)g * p.V * 256, (uint32_t)p.V * 256u, qbar);
            for (int n = 0; n < n_sc; ++n) {
                if (!take_stage(n)) break;
                const int s = n % p.ns;
                uint8_t* st = sm + s * kBsSlot;
                const int row = g * p.N + j_begin + n * kBsStageKeys;
                mbar_arrive_expect_tx(&full[s], kBsSlot);
#pragma unroll
                for (int t = 0; t < 2; ++t) {
                    tma_load_2d_hint(st + t * 16384, &kmap, 0, row + 64 * t, &full[s], pol);
                    tma_load_2d_hint(st + t * 16384 + 8192, &kmap, 64, row + 64 * t, &full[s], pol);
                }
                n_issued = n + 1;
            }
        }
        __syncwarp();
        asm volatile("barrier.cluster.wait.aligned;" ::: "memory");
    } else {
        // zero the padding query rows (attention rows R..15, indexer rows V..7), then wait for
        // the copied ones; the consumer warps' own barrier
        for (int i = tid; i < 24 * 16; i += 32 * kBsCons) {
            const int row = i >> 4;
            if (row < 16 ? row >= p.R : row - 16 >= p.V)
                reinterpret_cast<uint4*>(sm + (row < 16 ? p.oQ : p.oQi - 16 * 256))[i] = make_uint4(0u, 0u, 0u, 0u);
        }
        warp_wait(qbar, 0u, abort_flag, lim);
        asm volatile("bar.sync 1, %0;" ::"n"(32 * kBsCons) : "memory");
        asm volatile("barrier.cluster.wait.aligned;" ::: "memory");
        const int t = warp & 1;  // stage n goes to warps 2(n % 2) and 2(n % 2) + 1, tile t each
        for (int n = warp >> 1; n < n_sc; n += 2) {
            const int s = n % p.ns;
            if (!warp_wait(&full[s], (uint32_t)((n / p.ns) & 1), abort_flag, lim)) break;
            const int jt = j_begin + n * kBsStageKeys + 64 * t;
            float* sbuf = sc + jt;  // the score row has room for every CTA's whole share
            score_tile<F16>(ring + s * kBsSlot + t * 16384, smem_addr(sm + p.oQi), lane, p.V, sbuf);
            __syncwarp();
            if (lane == 0) mbar_arrive(&empty[s]);
            // the scores go to `scores` and into every peer's copy of the score row
            uint32_t key[2];
#pragma unroll
            for (int h = 0; h < 2; ++h) {
                const int j = jt + 32 * h + lane;
                const float v = sbuf[32 * h + lane];
                if (j < j_end) {
                    p.scores[(size_t)g * p.N + j] = v;
                    for (int c = 0; c < C; ++c)
                        if (c != r) *cl.map_shared_rank(sc + j, c) = v;
                }
                key[h] = float_key(v);
            }
            if (p.glg >= 0) {  // the selection's group maxima of these 64 keys (groups of <= 64)
                const int gsz = 1 << p.glg;
                if (gsz == 64) {
                    const uint32_t m = __reduce_max_sync(0xffffffffu, max(key[0], key[1]));
                    if (lane == 0 && (jt >> 6) < p.gcnt) gmx[jt >> 6] = m;
                } else {
#pragma unroll
                    for (int h = 0; h < 2; ++h) {
                        uint32_t m = key[h];
                        for (int o = 1; o < gsz; o <<= 1) m = max(m, __shfl_xor_sync(0xffffffffu, m, o));
                        const int j = jt + 32 * h + lane;
                        if ((lane & (gsz - 1)) == 0 && (j >> p.glg) < p.gcnt) gmx[j >> p.glg] = m;
                    }
                }
            }
        }
        if (p.glg >= 0 && j_begin < p.N) {
            // this CTA's bound: the kr-th largest maximum of its share's whole groups (kr of its
            // entries, in distinct groups, reach it), pushed to every CTA of the cluster
            asm volatile("bar.sync 1, %0;" ::"n"(32 * kBsCons) : "memory");
            if (warp == 0) {
                const int g0 = j_begin >> p.glg, g1 = min(p.gcnt, j_end >> p.glg);
                uint32_t lb = 0u;
                for (int base = g0; base < g1; base += 32) {
                    const int i = base + lane;
                    if (i < g1) {
                        const uint32_t v = gmx[i];
                        int gt = 0, ge = 0;
                        for (int u = g0; u < g1; ++u) {
                            const uint32_t w = gmx[u];
                            gt += w > v ? 1 : 0;
                            ge += w >= v ? 1 : 0;
                        }
                        if (gt < p.kr && p.kr <= ge) lb = v;
                    }
                }
                lb = __reduce_max_sync(0xffffffffu, lb);  // every lane that found it found the same value
                if (lane < C) *cl.map_shared_rank(reinterpret_cast<uint32_t*>(sm + p.oAux) + r, lane) = lb;
            }
        }
    }
    __syncwarp();
    cl.sync();  // (1) every CTA holds the whole score row and every CTA's bound

    // ---------------------------------------------------------------- 2. select
    {
        if (p.k == p.N) {
            for (int i = tid; i < p.N; i += kBsThreads) sel[i] = i;
            __syncthreads();
        } else if (p.k > 0) {
            uint32_t* wt = reinterpret_cast<uint32_t*>(sm + p.oScan);
            int* bc = reinterpret_cast<int*>(sm + p.oScan + 32);
            bool done = false;
            if (p.glg >= 0) {
                // L = the least of the CTAs' bounds: each holding CTA has kr >= k / cact entries
                // at or above its own, so the top k all reach L.  Each CTA ranks the candidates
                // (entries >= L) of the whole row: it takes those of its own share and pushes them
                // into region r of every CTA's ring (idle between the phases), with their count.
                const uint32_t* lbs = reinterpret_cast<const uint32_t*>(sm + p.oAux);
                uint32_t* lcnt = reinterpret_cast<uint32_t*>(sm + p.oAux) + kBsMaxCluster;
                uint32_t L = 0xffffffffu;
                for (int c = 0; c < p.cact; ++c) L = min(L, lbs[c]);
                uint32_t* cnt = reinterpret_cast<uint32_t*>(sm);  // [C] candidates from each CTA
                unsigned long long* cand = reinterpret_cast<unsigned long long*>(sm + 64);  // [C][capr], then the list
                uint32_t* bits = reinterpret_cast<uint32_t*>(sm + 64 + 2 * kBsCandCap * 8);  // [ceil(N / 32)]
                const int capr = kBsCandCap / C;
                for (int w = tid; w < (p.N + 31) / 32; w += kBsThreads) bits[w] = 0u;
                const uint32_t lt = lanemask_lt();
                for (int base = j_begin + warp * 32; base < j_end; base += kBsThreads) {
                    const int i = base + lane;
                    const uint32_t key = i < j_end ? float_key(sc[i]) : 0u;
                    const bool on = i < j_end && key >= L;
                    const uint32_t m = __ballot_sync(0xffffffffu, on);
                    if (m == 0u) continue;
                    uint32_t at = 0u;
                    if (lane == 0) at = atomicAdd(lcnt, (uint32_t)__popc(m));
                    at = __shfl_sync(0xffffffffu, at, 0) + (uint32_t)__popc(m & lt);
                    if (on && at < (uint32_t)capr) {
                        const unsigned long long v = ((unsigned long long)key << 32) | (0xffffffffu - (uint32_t)i);
                        for (int c = 0; c < C; ++c) *cl.map_shared_rank(cand + r * capr + at, c) = v;
                    }
                }
                __syncthreads();
                if (tid < C) *cl.map_shared_rank(cnt + r, tid) = *lcnt;  // above capr: overflow
                cl.sync();  // (1b) every CTA holds every CTA's candidates
                bool ovf = false;
                for (int c = 0; c < C; ++c) ovf = ovf || cnt[c] > (uint32_t)capr;
                if (!ovf) {
                    // the regions as one list, then the rank of each candidate among all of them
                    // (order key, then the lower index), eight loads in flight per thread
                    unsigned long long* lst = cand + kBsCandCap;  // [total], after the regions
                    int total = 0;
                    for (int c = 0; c < C; ++c) {
                        const int n = (int)cnt[c];
                        for (int s2 = tid; s2 < n; s2 += kBsThreads) lst[total + s2] = cand[c * capr + s2];
                        total += n;
                    }
                    __syncthreads();
                    for (int q = tid; q < total; q += kBsThreads) {
                        const unsigned long long v = lst[q];
                        int r0 = 0, r1 = 0;
                        int t = 0;
                        for (; t + 8 <= total; t += 8) {
                            unsigned long long u[8];
#pragma unroll
                            for (int e = 0; e < 8; ++e) u[e] = lst[t + e];
#pragma unroll
                            for (int e = 0; e < 8; e += 2) {
                                r0 += u[e] > v ? 1 : 0;
                                r1 += u[e + 1] > v ? 1 : 0;
                            }
                        }
                        for (; t < total; ++t) r0 += lst[t] > v ? 1 : 0;
                        if (r0 + r1 < p.k) {
                            const uint32_t i = 0xffffffffu - (uint32_t)(v & 0xffffffffull);
                            atomicOr(&bits[i >> 5], 1u << (i & 31));
                        }
                    }
                    __syncthreads();
                    bs_emit_bits(bits, p.N, p.k, sel, wt);
                    done = true;
                }
            }
            if (!done)  // no bound, or too many entries reach it (heavy ties): radix over the row
                bs_select(sc, p.N, p.k, sel, reinterpret_cast<uint32_t*>(sm + p.oHist), wt, bc);
        }
        if (r == 0)
            for (int i = tid; i < p.k; i += kBsThreads) p.idx[(size_t)g * p.k + i] = sel[i];
    }

    // ---------------------------------------------------------------- 3. attend
    AttAccT<NQ> acc;
    if (warp == kBsProd) {
        if (lane == 0 && !*abort_flag) {
            for (int a = 0; a < n_at; ++a) {
                const int n = n_sc + a;
                if (!take_stage(n)) break;
                const int s = n % p.ns;
                uint8_t* st = sm + s * kBsSlot;
                const int j0 = (s0 + a) * kBsStageRows;
                mbar_arrive_expect_tx(&full[s], kBsSlot);
                for (int q = 0; q < kBsStageRows; q += p.br) {
                    // a run past the list's end loads the stage's first run again (masked out)
                    const int jr = j0 + q < n_rows ? j0 + q : j0;
                    const int e = jr / p.block;
                    const int row = g * p.T + sel[e] * p.block + (jr - e * p.block);
                    uint8_t* dk = st + (q >> 5) * 16384 + (q & 31) * 128;
                    tma_load_2d_hint(dk, &kvk, 0, row, &full[s], pol);
                    tma_load_2d_hint(dk + 4096, &kvk, 64, row, &full[s], pol);
                    tma_load_2d_hint(dk + 8192, &kvv, 0, row, &full[s], pol);
                    tma_load_2d_hint(dk + 12288, &kvv, 64, row, &full[s], pol);
                }
                n_issued = n + 1;
            }
        }
    } else {
        att_init_t(acc);
        uint32_t qf[8][NQ][2];
        load_q_frags_t<NQ>(smem_addr(sm + p.oQ), lane, qf);
        const int h = warp & 1;
        for (int a = 0; a < n_at; ++a) {
            const int n = n_sc + a;
            if ((n & 1) != (warp >> 1)) continue;
            if (*abort_flag) break;
            const int s = n % p.ns;
            if (!warp_wait(&full[s], (uint32_t)((n / p.ns) & 1), abort_flag, lim)) break;
            const int jb = (s0 + a) * kBsStageRows + 32 * h;
            const int nv = max(0, min(32, n_rows - jb));
            const uint32_t valid = nv >= 32 ? 0xffffffffu : ((1u << nv) - 1u);
            const uint32_t kb = ring + s * kBsSlot + h * 16384;
            if (valid != 0u) attend_stage_t<NQ>(kb, kb + 8192, lane, qf, valid, p.scale_log2, acc);
            __syncwarp();
            if (lane == 0) mbar_arrive(&empty[s]);
        }
    }
    __syncthreads();
    if (tid == 32 * kBsProd && *abort_flag) {
        // let every stage issued but not consumed land before the ring is reused
        for (int n = max(0, n_issued - p.ns); n < n_issued; ++n)
            mbar_wait(&full[n % p.ns], (uint32_t)((n / p.ns) & 1), lim);
        mbar_wait(qbar, 0u, lim);
    }
    pdl_launch_dependents();
    __syncthreads();

    // ---------------------------------------------------------------- 4. merge
    float* wo = reinterpret_cast<float*>(sm + kBsPartO);     // [4][16][128]
    float2* wml = reinterpret_cast<float2*>(sm + kBsPartML);  // [4][16]
    const int ipc = (p.R * 32 + C - 1) / C;  // inbox slots: items a CTA owns
    float4* in_o = reinterpret_cast<float4*>(sm + p.oInbox);                        // [C][ipc]
    float2* in_ml = reinterpret_cast<float2*>(sm + p.oInbox + C * ipc * 16);        // [C][16]
    if (warp < kBsCons) {  // O^T fragments: column 16md + g8 (+8) of query row 8nq + 2t4 + e
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
    // the CTA's state: (query row, 4 columns) items over the four warps' states
    for (int i = tid; i < p.R * 32; i += kBsThreads) {
        const int row = i >> 5, c4 = i & 31;
        float2 ml[kBsCons];
        float4 o[kBsCons];
#pragma unroll
        for (int w = 0; w < kBsCons; ++w) {
            ml[w] = wml[w * 16 + row];
            o[w] = reinterpret_cast<const float4*>(wo + (w * 16 + row) * 128)[c4];
        }
        float M = -INFINITY;
#pragma unroll
        for (int w = 0; w < kBsCons; ++w) M = fmaxf(M, ml[w].x);
        float L = 0.f;
        float4 O = make_float4(0.f, 0.f, 0.f, 0.f);
#pragma unroll
        for (int w = 0; w < kBsCons; ++w) {
            const float f = ml[w].x == -INFINITY ? 0.f : exp2f(ml[w].x - M);
            L = fmaf(ml[w].y, f, L);
            O.x = fmaf(o[w].x, f, O.x);
            O.y = fmaf(o[w].y, f, O.y);
            O.z = fmaf(o[w].z, f, O.z);
            O.w = fmaf(o[w].w, f, O.w);
        }
        // pushed to the item's owner; the row's (M, L) to every CTA (item (row, c4 < C) is
        // CTA c4's, as 32 is a multiple of C)
        *cl.map_shared_rank(in_o + r * ipc + i / C, i % C) = O;
        if (c4 < C) *cl.map_shared_rank(in_ml + r * 16 + row, c4) = make_float2(M, L);
    }
    cl.sync();  // (2) every CTA's state is in its owners' inboxes
    // the output: the items this CTA owns, each merging the C CTAs' states in rank order
    for (int i = tid * C + r; i < p.R * 32; i += kBsThreads * C) {
        const int row = i >> 5, c4 = i & 31;
        float2 ml[kBsMaxCluster];
        float4 o[kBsMaxCluster];
#pragma unroll
        for (int c = 0; c < kBsMaxCluster; ++c) {
            if (c < C) {
                ml[c] = in_ml[c * 16 + row];
                o[c] = in_o[c * ipc + i / C];
            }
        }
        float M = -INFINITY;
#pragma unroll
        for (int c = 0; c < kBsMaxCluster; ++c)
            if (c < C) M = fmaxf(M, ml[c].x);
        float L = 0.f;
        float4 O = make_float4(0.f, 0.f, 0.f, 0.f);
#pragma unroll
        for (int c = 0; c < kBsMaxCluster; ++c) {
            if (c >= C) continue;
            const float f = ml[c].x == -INFINITY ? 0.f : exp2f(ml[c].x - M);
            L = fmaf(ml[c].y, f, L);
            O.x = fmaf(o[c].x, f, O.x);
            O.y = fmaf(o[c].y, f, O.y);
            O.z = fmaf(o[c].z, f, O.z);
            O.w = fmaf(o[c].w, f, O.w);
        }
        const int v = row / p.G, gi = row % p.G;
        const size_t qrow = ((size_t)b * p.V + v) * p.Hq + (size_t)kvh * p.G + gi;
        const float inv = L > 0.f ? 1.f / L : 0.f;
        reinterpret_cast<float4*>(p.out + qrow * 128)[c4] = make_float4(O.x * inv, O.y * inv, O.z * inv, O.w * inv);
        if (c4 == 0) p.lse[qrow] = L > 0.f ? (M + log2f(L)) * 0.69314718055994530942f : -INFINITY;
    }
    // nothing reads a peer's shared memory after (2): the CTA may leave
    if (tid == 0 && *abort_flag) report(p.err, SD_DEVERR_TIMEOUT);
}

struct BsPlan {
    int C, ns, nc, per_sm, bytes;
    int oQ, oQi, oScore, oSel, oHist, oScan, oGmax, oInbox, oAux, oBars, oMisc;
};

int align_up(int x, int a) { return (x + a - 1) / a * a; }

BsPlan layout_for(int N, int k, int C, int ns) {
    BsPlan pl{};
    pl.C = C;
    pl.ns = ns;
    pl.nc = align_up((N + C - 1) / C, kBsStageKeys);
    int off = ns * kBsSlot;
    pl.oQ = off;
    off += 16 * 256;
    pl.oQi = off;
    off += 8 * 256;
    pl.oScore = off;
    off += align_up(C * pl.nc * 4, 16);
    pl.oSel = off;
    off += align_up(std::max(k, 1) * 4, 16);
    pl.oHist = off;
    off += 256 * 4;
    pl.oScan = off;
    off += 64;
    pl.oGmax = off;
    off += kBsMaxGroups * 4;
    pl.oInbox = off;
    off += kBsInboxBytes;
    pl.oAux = off;
    off += 64;
    pl.oBars = off;
    off += align_up((2 * ns + 1) * 8, 16);
    pl.oMisc = off;
    off += 16;
    pl.bytes = off + 1024;  // slack for the 1024-byte alignment of the ring
    return pl;
}

// Cluster size C (the largest of 8, 4, 2, 1 whose NG*C CTAs fit in one wave at two CTAs per
// SM) and ring depth: two CTAs per SM with the deepest ring that leaves room for both when
// the CTAs outnumber the SMs, else one CTA per SM with up to eight stages.  The depth is
// even: stage n goes to slot n % ns and consumer pair n % 2, so a pair only ever meets its
// own slots, in order, and never waits on a slot's phase while that slot is two phases
// behind (an mbarrier's parity could not tell those apart).
BsPlan plan_block_step(int NG, int N, int k) {
    int dev = 0;
    cudaGetDevice(&dev);
    int per_sm_smem = 0, reserved = 0;
    cudaDeviceGetAttribute(&per_sm_smem, cudaDevAttrMaxSharedMemoryPerMultiprocessor, dev);
    cudaDeviceGetAttribute(&reserved, cudaDevAttrReservedSharedMemoryPerBlock, dev);
    const int optin = max_smem_optin();
    const int sms = num_sms();
    int C = 1;
    for (int c = kBsMaxCluster; c >= 1; c /= 2)
        if ((long long)NG * c <= 2LL * sms) {
            C = c;
            break;
        }
    const int per_sm = (long long)NG * C > sms ? 2 : 1;
    const int budget = std::min(optin, per_sm_smem / per_sm - reserved);
    BsPlan best = layout_for(N, k, C, 2);
    for (int ns = 4; ns <= 8; ns += 2) {  // even: each consumer pair keeps its own stages
        const BsPlan pl = layout_for(N, k, C, ns);
        if (pl.bytes > budget) break;
        best = pl;
    }
    best.per_sm = per_sm;
    return best;
}

}  // namespace

bool block_step_eligible(const sd_decode_step_args* a) {
    const int bl = a->block;
    const bool runs = bl % 16 == 0 && (bl <= 32 ? 32 % bl == 0 : bl % 32 == 0);
    const int N = a->T / bl;
    return runs && N <= kBsMaxN && layout_for(N, a->n_idx, 1, 2).bytes <= max_smem_optin();
}

sd_status block_step_launch(const sd_decode_step_args* a, cudaStream_t st) {
    const char* who = "sd_decode_step";
    const int NG = a->B * a->Hkv, N = a->T / a->block;
    const BsPlan pl = plan_block_step(NG, N, a->n_idx);
    SD_REQUIRE(pl.bytes <= max_smem_optin(), "%s: the group's score row does not fit in shared memory", who);
    const bool f16 = a->key_dtype == SD_F16;
    const int br = std::min(a->block, 32);
    CUtensorMap kmap, kvk, kvv;
    if (!make_tensor_map_2d(&kmap, a->keys, (uint64_t)NG * N, 128, 64, f16) ||
        !make_tensor_map_2d(&kvk, a->k_cache, (uint64_t)NG * a->T, 128, br, false) ||
        !make_tensor_map_2d(&kvv, a->v_cache, (uint64_t)NG * a->T, 128, br, false)) {
        set_error("%s: cuTensorMapEncodeTiled failed", who);
        return SD_ERR_CUDA;
    }
    BsParams p{};
    p.q_idx = static_cast<const uint8_t*>(a->q_idx);
    p.q = static_cast<const uint8_t*>(a->q);
    p.scores = a->scores;
    p.idx = a->idx;
    p.out = a->out;
    p.lse = a->lse;
    p.err = a->err_word;
    p.V = a->V;
    p.Hq = a->Hq;
    p.Hkv = a->Hkv;
    p.G = a->Hq / a->Hkv;
    p.R = p.G * a->V;
    p.T = a->T;
    p.N = N;
    p.k = a->n_idx;
    p.block = a->block;
    p.br = br;
    p.nc = pl.nc;
    p.ns = pl.ns;
    p.oQ = pl.oQ;
    p.oQi = pl.oQi;
    p.oScore = pl.oScore;
    p.oSel = pl.oSel;
    p.oHist = pl.oHist;
    p.oScan = pl.oScan;
    p.oGmax = pl.oGmax;
    p.oInbox = pl.oInbox;
    p.oAux = pl.oAux;
    // the selection's group maxima are taken while scoring when its fast path applies and a
    // group (2^glg keys, glg <= 6) lies within one 64-key scoring tile
    p.glg = -1;
    p.gcnt = 0;
    p.cact = (N + pl.nc - 1) / pl.nc;
    p.kr = (p.k + p.cact - 1) / std::max(1, p.cact);
    if (p.k > 0 && p.k < N) {
        int lg = 2;
        while ((N >> (lg + 1)) >= 2 * p.k) ++lg;
        const int G = (N >> lg) & ~3;
        // every CTA holding keys needs kr whole groups of its own share for its bound
        bool enough = G >= p.k && G >= 4 && G <= kBsMaxGroups && lg <= 6;
        for (int c = 0; enough && c < p.cact; ++c) {
            const int j0 = c * pl.nc, j1 = std::min(N, j0 + pl.nc);
            enough = std::min(G, j1 >> lg) - (j0 >> lg) >= p.kr;
        }
        if (enough) {
            p.glg = lg;
            p.gcnt = G;
        }
    }
    p.oBars = pl.oBars;
    p.oMisc = pl.oMisc;
    p.scale_log2 = a->scale * 1.44269504088896340736f;
    p.wait_ns = a->wait_limit_ns > 0 ? (unsigned long long)a->wait_limit_ns : (unsigned long long)kWaitDeadlineNs;
    const bool nq1 = p.R <= 8;  // query rows in one tile of 8, else two
    auto kern = f16 ? (nq1 ? block_step_kernel<true, 1> : block_step_kernel<true, 2>)
                    : (nq1 ? block_step_kernel<false, 1> : block_step_kernel<false, 2>);
    SD_CUDA_CHECK(cudaFuncSetAttribute(kern, cudaFuncAttributeMaxDynamicSharedMemorySize, pl.bytes),
                  "sd_decode_step: cudaFuncSetAttribute");
    cudaLaunchConfig_t cfg{};
    cfg.gridDim = dim3((unsigned)(NG * pl.C));
    cfg.blockDim = dim3(kBsThreads);
    cfg.dynamicSmemBytes = (size_t)pl.bytes;
    cfg.stream = st;
    cudaLaunchAttribute attr[2];
    attr[0].id = cudaLaunchAttributeClusterDimension;
    attr[0].val.clusterDim.x = (unsigned)pl.C;
    attr[0].val.clusterDim.y = 1;
    attr[0].val.clusterDim.z = 1;
    attr[1].id = cudaLaunchAttributeProgrammaticStreamSerialization;
    attr[1].val.programmaticStreamSerializationAllowed = 1;
    cfg.attrs = attr;
    cfg.numAttrs = 2;
    SD_CUDA_CHECK(cudaLaunchKernelEx(&cfg, kern, kmap, kvk, kvv, p), "sd_decode_step: launch");
    return launch_status(who);
}

}  // namespace sd
