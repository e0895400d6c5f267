// decode_step.cu -- one whole sparse decode step (indexer, top-k, gather-attend) in one
// persistent launch.
//
// SparDA (gist.science summary), sec. 2 "Indexador de Previsao Compacto": one indexer head
// per KV group scores every cached token (or block, sec. 2 item 1) with a dot product and no
// softmax.  "Esparsidade de Contexto no Tempo de Inferencia" (gist.science summary), sec. 2:
// exact (Oracle) top-k feeding a sparse decode kernel; sec. 3C: traffic O(k*d) instead of
// O(N*d).  Adaptive DHiSparse (news page), "Metodologia": the query rows of a group share
// every fetched row.  Ties in the selection go to the lower index (the pages are silent).
//
// Computes what sd_index_score -> sd_topk -> sd_gather_attend computes (scores and index
// sets bit for bit; attention in its own summation order), for K/V resident in HBM.
//
// The work of a step is a list of tasks taken from one device counter (one per claim):
//   scoring task (g, part)   128 indexer keys of KV group g, as two 16 KB stages of 64 keys
//                            (tiled TMA, 128-byte swizzle) -> scores (mma.sync m16n8k16;
//                            products of integer-valued keys and queries are exact, so are the
//                            fp32 sums) and their 11-bit order-key digits added to the group's
//                            histogram;
//   attention task (g, part) up to 128 selected rows of group g, as up to four stages of 32 K
//                            and V rows (tiled TMA for whole 32-row runs of a block, 16-byte
//                            cp.async for scattered rows): exact online softmax over them for
//                            all G*V query rows of the group, written as one partial (m, l, O).
// The list puts the scoring tasks of group g + L before the attention tasks of group g, so the
// attention of early groups overlaps the scoring of later ones (L, the lag, covers the time a
// group's selection takes).  The CTA that claims a group's last scoring task owns its top-k:
// it runs it once every scoring task of the group is counted; the group's attention tasks
// wait (bounded) for it.  The CTA that claims a group's last attention task likewise merges
// the group's partials, in task order, once they are all counted.  The owners are whichever
// CTAs happened to claim those tasks, so the selections spread over the GPU.
//
// A CTA (one per SM) runs four independent pipelines: producer warp 4 + w claims tasks and
// fills the two 16 KB ring slots of consumer warp w, which runs each task alone (so four
// tasks are worked on at once while the next stages load, and a task waiting for its group's
// selection holds up only its own pipeline) and posts a record per finished task.  Warp 8
// keeps the books: it counts the records into the device-scope counters (one fence per batch
// and fire-and-forget adds) and hands the selections and merges this CTA owns, once their
// groups are complete, to warps 9-10.  Every wait is bounded; a wait that runs out sets
// SD_DEVERR_TIMEOUT, every role leaves at its next wait, and the CTA lets its copies in flight
// land before it exits.
#include <algorithm>
#include <cmath>

#include "sd_host.h"
#include "step_tiles.cuh"
#include "tc_common.cuh"

namespace sd {
namespace {

constexpr int kDsCons = 4;                           // pipelines: consumer warps 0-3
constexpr int kDsProd0 = kDsCons;                    // producer warps 4-7
constexpr int kDsBook = 2 * kDsCons;                 // bookkeeping warp 8
constexpr int kDsSel0 = kDsBook + 1;                 // selection warps 9-10
constexpr int kDsSelW = 2;
constexpr int kDsThreads = 32 * (kDsSel0 + kDsSelW);
constexpr int kDsST = 32 * kDsSelW;                  // selection threads
constexpr int kDsStages = 2 * kDsCons;               // ring slots: two per pipeline
constexpr int kDsData = 16384;                       // keys, or K then V rows, of one stage
constexpr int kDsQSlot = 4096;                       // the stage's query rows (<= 16 of 256 B)
constexpr int kDsStage = kDsData + kDsQSlot;
constexpr int kDsKeyRows = 64;                       // indexer keys per scoring stage
constexpr int kDsScoreStages = 2;                    // stages per scoring task
constexpr int kDsTaskKeys = kDsKeyRows * kDsScoreStages;
constexpr int kDsRows = 32;                          // K/V rows per attention stage
constexpr int kDsTaskStages = 4;                     // stages per attention task
constexpr int kDsTaskRows = kDsRows * kDsTaskStages;  // selected rows per attention task
constexpr int kDsBins = 2048;                        // 11-bit digits of the order key
constexpr int kDsCand = 1024;                        // candidates kept in shared memory
constexpr int kDsMaxN = 32768;                       // scores per group the selection handles
constexpr int kDsMaxR = 16;                          // query rows per group
constexpr int kDsRecW = 16;                          // records in flight per pipeline
constexpr int kDsJobsW = 16;                         // owned selections / merges per producer
constexpr int kDsChunk = 32 * kDsST;                 // scores per chunk of a pass over them
constexpr int kDsClaim = 1;                          // tasks a producer claims per atomic
constexpr int kDsSelScratch = (kDsBins * 4 + 2 * (kDsMaxN / 8) + 2 * kDsCand * 4) / 8;  // float2 slots
constexpr int kDsMaxMerge = kDsSelScratch - kDsMaxR;  // (partial, row) pairs a merge takes

enum : int { kTaskScore = 0, kTaskAttend = 1, kTaskEnd = 2, kTaskFin = 3 };

struct StageMeta {
    int kind, g, task, j0, nrows, sgi, nst, pad;
    uint32_t valid, pad1, pad2, pad3;
};

struct DsLayout {
    static constexpr int oHist = kDsStages * kDsStage;        // u32[2048]
    static constexpr int oSel = oHist + kDsBins * 4;          // u32[kDsMaxN / 32]
    static constexpr int oTie = oSel + kDsMaxN / 8;           // u32[kDsMaxN / 32]
    static constexpr int oCandIdx = oTie + kDsMaxN / 8;       // i32[kDsCand]
    static constexpr int oCandKey = oCandIdx + kDsCand * 4;   // u32[kDsCand]
    static constexpr int oChunk = oCandKey + kDsCand * 4;     // f32[2][kDsChunk]
    static constexpr int oScore = oChunk + 2 * kDsChunk * 4;  // f32[4][64] per consumer warp
    static constexpr int oMeta = oScore + kDsCons * 64 * 4;   // StageMeta[kDsStages]
    static constexpr int oBars = oMeta + kDsStages * (int)sizeof(StageMeta);
    // full[S], empty[S], rec_full[4][R], rec_free[4][R], chunk[2]
    static constexpr int kBars = 2 * kDsStages + 2 * kDsCons * kDsRecW + 2;
    static constexpr int oRec = oBars + kBars * 8;            // int2[4][kDsRecW]
    static constexpr int oJobs = oRec + kDsCons * kDsRecW * 8;  // int[2][4][kDsJobsW]: selections, merges
    static constexpr int oMisc = oJobs + 2 * kDsCons * kDsJobsW * 4;  // flags, ring indices, broadcast
    static constexpr int kMisc = 512;
    static constexpr int kBytes = oMisc + kMisc + 1024;       // + slack for 1024-byte alignment
    static_assert(kDsStage % 1024 == 0, "stages must stay 1024-byte aligned (128-byte swizzle)");
    static_assert(oChunk - oHist == kDsSelScratch * 8, "the selection scratch is one area");
    static_assert(kBytes <= 232448, "shared memory per CTA");
};

// Offsets in the misc area.
constexpr int kMiAbort = 0, kMiBusy = 4, kMiWork = 8 /* kind, group */, kMiCandN = 16, kMiCpar = 20 /* [2] */,
              kMiConsumed = 32 /* [4] */, kMiIssued = 48 /* [4] */, kMiJobIdx = 64 /* [4 producers][4] */,
              kMiBc = 128 /* [16] */, kMiWt = 192 /* [kDsSelW] */;

struct DsParams {
    const uint8_t* q_idx;  // [NG, V, 128] 16-bit
    const uint8_t* q;      // [B, V, Hq, 128] bf16
    const uint8_t* kc;     // [NG * T, 128] bf16
    const uint8_t* vc;
    float* scores;         // [NG, N]
    int32_t* idx;          // [NG, k]
    float* out;            // [B, V, Hq, 128]
    float* lse;            // [B, V, Hq]
    int32_t* err;
    uint32_t* ctrl;        // [0] next task, [1] CTAs finished
    uint32_t* gstate;      // [NG][4]: scoring tasks done, attention tasks done, selection ready
    uint32_t* hist;        // [NG][2048]
    float* part_o;         // [NG][AG][R][128]
    float* part_ml;        // [NG][AG][R][2]
    int B, V, Hq, Hkv, G, R, T, N, k, block, NG, SG, AG, L, n_rows;
    int tma_blocks;        // block % 32 == 0: a stage's 32 rows are one contiguous run
    float scale_log2;
    unsigned long long wait_ns;
    uint32_t total;
};

struct Task {
    int kind, g, part;
};

// Task t of the list: units u = 0 .. NG + L - 1, unit u holding the scoring tasks of group u
// (u < NG) and then the attention tasks of group u - L (u >= L).
SD_DEVINL Task decode_task(const DsParams& p, uint32_t t) {
    const uint32_t a = (uint32_t)p.L * (uint32_t)p.SG;
    if (t < a) return {kTaskScore, (int)(t / p.SG), (int)(t % p.SG)};
    t -= a;
    const uint32_t u = (uint32_t)(p.SG + p.AG);
    const uint32_t b = (uint32_t)(p.NG - p.L) * u;
    if (t < b) {
        const int uu = p.L + (int)(t / u), r = (int)(t % u);
        if (r < p.SG) return {kTaskScore, uu, r};
        return {kTaskAttend, uu - p.L, r - p.SG};
    }
    t -= b;
    return {kTaskAttend, p.NG - p.L + (int)(t / p.AG), (int)(t % p.AG)};
}

// ------------------------------------------------------------------ selection

struct SelSmem {
    uint32_t* hist;   // [2048]
    uint32_t* sel;    // [kDsMaxN / 32]
    uint32_t* tie;    // [kDsMaxN / 32]
    int32_t* cidx;    // [kDsCand]
    uint32_t* ckey;   // [kDsCand]
    float2* scratch;  // the five arrays above as one [kDsSelScratch] float2 area (merges)
    float* chunk;     // [2][kDsChunk]
    uint64_t* cbar;   // [2] chunk barriers
    volatile uint32_t* cpar;  // [2] their next parities
    volatile uint32_t* cand_n;
    int* bc;          // broadcast scalars [16]
    uint32_t* wt;     // per-warp scan totals [kDsSelW]
    volatile int* abort_flag;
    uint64_t lim;
};

// Barrier of the kDsST selection threads (hardware named barrier 1).  Every selection warp
// passes the same sequence of these barriers: a selection's or a merge's control flow
// depends only on values shared through shared memory, and nothing inside either waits on
// another role (the chunk copies it waits for are its own, with bounded waits), so no
// selection warp can be left waiting here.
SD_DEVINL void sel_bar() { asm volatile("bar.sync 1, %0;" ::"n"(kDsST) : "memory"); }

// Sum of v over the selection threads above this one (descending: up = false) or below it
// (ascending: up = true), in every thread.
SD_DEVINL uint32_t sel_scan_excl(uint32_t v, int sst, const SelSmem& S, bool up) {
    const int lane = sst & 31, w = sst >> 5;
    uint32_t x = v;
#pragma unroll
    for (int o = 1; o < 32; o <<= 1) {
        const uint32_t y = up ? __shfl_up_sync(0xffffffffu, x, o) : __shfl_down_sync(0xffffffffu, x, o);
        if (up ? lane >= o : lane + o < 32) x += y;
    }
    if (lane == (up ? 31 : 0)) S.wt[w] = x;
    sel_bar();
    uint32_t r = x - v;
#pragma unroll
    for (int u = 0; u < kDsSelW; ++u)
        if (up ? u < w : u > w) r += S.wt[u];
    sel_bar();  // wt may be reused after this
    return r;
}

// In the 2048-bin histogram S.hist, the bin d where the count of entries in bins above d is
// < target <= that count plus hist[d] (1 <= target <= the total): writes d, the count above
// and hist[d] to S.bc[o .. o+2], visible to every thread on return.
SD_DEVINL void sel_find_bin(uint32_t target, int o, int sst, const SelSmem& S) {
    constexpr int per = kDsBins / kDsST;
    const uint32_t* h = S.hist + sst * per;
    uint32_t loc = 0;
#pragma unroll 8
    for (int j = 0; j < per; ++j) loc += h[(j + sst) & (per - 1)];
    const uint32_t above = sel_scan_excl(loc, sst, S, false);
    if (above < target && target <= above + loc) {
        uint32_t cum = above;
        for (int j = per - 1; j >= 0; --j) {
            const uint32_t c = h[j];
            if (cum + c >= target) {
                S.bc[o] = sst * per + j;
                S.bc[o + 1] = (int)cum;
                S.bc[o + 2] = (int)c;
                break;
            }
            cum += c;
        }
    }
    sel_bar();
}

enum : int { kPassFirst, kPassSelD, kPassHist2, kPassSelP22, kPassHist3, kPassSelThr, kPassSelTie };

struct PassArg {
    int mode, D;
    uint32_t p22, thr;
};

// For pass modes other than kPassFirst: whether an entry with order key `key` sets its bit in
// the selection (sel) and tie bitmaps, and the histogram bin it adds to (hbin >= 0).
SD_DEVINL void pass_decide(const PassArg& a, uint32_t key, bool& sel, bool& tie, int& hbin) {
    const bool inD = (int)(key >> 21) == a.D;
    sel = tie = false;
    hbin = -1;
    switch (a.mode) {
        case kPassSelD: sel = inD; break;
        case kPassHist2: hbin = inD ? (int)((key >> 10) & 2047u) : -1; break;
        case kPassSelP22: sel = inD && (key >> 10) >= a.p22; break;
        case kPassHist3: hbin = (key >> 10) == a.p22 ? (int)(key & 1023u) : -1; break;
        case kPassSelThr: sel = inD && key >= a.thr; break;
        default:  // kPassSelTie
            sel = inD && key > a.thr;
            tie = inD && key == a.thr;
            break;
    }
}

// One pass over the group's N scores (N a multiple of 4) in chunks of kDsChunk, through two
// shared-memory buffers filled by 1-D bulk copies (one copy in flight while the other chunk is
// read).  In a chunk, selection thread t owns bitmap word t (scores 32t .. 32t + 31 of the
// chunk) and builds its bits in a register, so no bitmap update is atomic.  kPassFirst sets
// the bits above digit D and keeps the digit-D entries as candidates, allocated once per warp
// and chunk.  Ends with a selection barrier.
SD_DEVINL void score_pass(const PassArg& a, const float* sc, int N, int sst, const SelSmem& S) {
    const int lane = sst & 31;
    const int nch = (N + kDsChunk - 1) / kDsChunk;
    uint32_t par0 = S.cpar[0], par1 = S.cpar[1];
    float* chunk = S.chunk;
    uint64_t* cbar = S.cbar;
    auto issue = [&](int c, int b) {
        const uint32_t bytes = (uint32_t)min(kDsChunk, N - c * kDsChunk) * 4u;
        mbar_arrive_expect_tx(&cbar[b], bytes);
        bulk_g2s(chunk + b * kDsChunk, sc + (size_t)c * kDsChunk, bytes, &cbar[b]);
    };
    if (sst == 0) {
        // the scores were written by other CTAs (generic stores, acquired through the group's
        // counter); order that before these async-proxy reads
        asm volatile("fence.proxy.async.global;" ::: "memory");
        issue(0, 0);
        if (nch > 1) issue(1, 1);
    }
    uint32_t* sel = S.sel;
    uint32_t* tie = S.tie;
    for (int c = 0; c < nch; ++c) {
        const int b = c & 1;
        if (!mbar_wait(&cbar[b], b ? par1 : par0, S.lim)) *S.abort_flag = 1;
        if (b) par1 ^= 1u;
        else par0 ^= 1u;
        const int base = c * kDsChunk + 32 * sst;  // this thread's 32 scores
        const int nin = max(0, min(32, N - base));
        const float4* b4 = reinterpret_cast<const float4*>(chunk + b * kDsChunk) + 8 * sst;
        // the thread's 32 keys in read order: key[4j + e] is score 4 * ((j + sst) & 7) + e of its
        // word (the rotated order makes a quarter warp read 8 distinct bank groups)
        uint32_t key[32];
#pragma unroll
        for (int j = 0; j < 8; ++j) {
            const float4 v = b4[(j + sst) & 7];
            key[4 * j + 0] = float_key(v.x);
            key[4 * j + 1] = float_key(v.y);
            key[4 * j + 2] = float_key(v.z);
            key[4 * j + 3] = float_key(v.w);
        }
        const int w = base >> 5;
        if (a.mode == kPassFirst) {
            uint32_t above = 0, cnt = 0;
#pragma unroll
            for (int e = 0; e < 32; ++e) {
                const int bp = 4 * (((e >> 2) + sst) & 7) + (e & 3);
                const int dg = (int)(key[e] >> 21);
                const uint32_t in = bp < nin ? 1u : 0u;
                above |= (in & (dg > a.D ? 1u : 0u)) << bp;
                cnt += in & (dg == a.D ? 1u : 0u);
            }
            if (nin > 0) sel[w] = above;
            // candidates: one shared atomic per warp, then each thread writes its own
            uint32_t incl = cnt;
#pragma unroll
            for (int o = 1; o < 32; o <<= 1) {
                const uint32_t y = __shfl_up_sync(0xffffffffu, incl, o);
                if (lane >= o) incl += y;
            }
            uint32_t wbase = 0;
            if (lane == 31 && incl > 0) wbase = atomicAdd(const_cast<uint32_t*>(S.cand_n), incl);
            wbase = __shfl_sync(0xffffffffu, wbase, 31);
            uint32_t slot = wbase + incl - cnt;
            if (cnt > 0) {
#pragma unroll
                for (int e = 0; e < 32; ++e) {
                    const int bp = 4 * (((e >> 2) + sst) & 7) + (e & 3);
                    if (bp < nin && (int)(key[e] >> 21) == a.D) {
                        if (slot < (uint32_t)kDsCand) {
                            S.cidx[slot] = base + bp;
                            S.ckey[slot] = key[e];
                        }
                        ++slot;
                    }
                }
            }
        } else {
            uint32_t sw = 0, tw = 0;
#pragma unroll
            for (int e = 0; e < 32; ++e) {
                const int bp = 4 * (((e >> 2) + sst) & 7) + (e & 3);
                bool sl, tl;
                int hb;
                pass_decide(a, key[e], sl, tl, hb);
                const uint32_t in = bp < nin ? 1u : 0u;
                sw |= (in & (sl ? 1u : 0u)) << bp;
                tw |= (in & (tl ? 1u : 0u)) << bp;
                if (in && hb >= 0) atomicAdd(&S.hist[hb], 1u);
            }
            if (sw) sel[w] |= sw;
            if (tw) tie[w] |= tw;
        }
        sel_bar();  // every thread is done with buffer b
        if (sst == 0 && c + 2 < nch) {
            fence_proxy_async_shared();
            issue(c + 2, b);
        }
    }
    if (sst == 0) {
        S.cpar[0] = par0;
        S.cpar[1] = par1;
    }
    sel_bar();
}

// One pass over the candidates (every one has digit D; never kPassFirst).  Ends with a
// selection barrier.
SD_DEVINL void cand_pass(const PassArg& a, int n, int sst, const SelSmem& S) {
    for (int c = sst; c < n; c += kDsST) {
        bool sl, tl;
        int hb;
        const int i = S.cidx[c];
        pass_decide(a, S.ckey[c], sl, tl, hb);
        if (sl) atomicOr(&S.sel[i >> 5], 1u << (i & 31));
        if (tl) atomicOr(&S.tie[i >> 5], 1u << (i & 31));
        if (hb >= 0) atomicAdd(&S.hist[hb], 1u);
    }
    sel_bar();
}

// The group's exact top-k: ascending indices of the k entries first in (score desc, index
// asc), written to p.idx[g]; the group's histogram is read and zeroed.  All kDsST selection
// threads call it.
SD_DEVINL void select_group(const DsParams& p, int g, int sst, const SelSmem& S) {
    const int N = p.N, k = p.k;
    const float* sc = p.scores + (size_t)g * N;
    uint32_t* gh = p.hist + (size_t)g * kDsBins;
    int32_t* out = p.idx + (size_t)g * k;

    // 1. the top digit D from the histogram the scoring tasks built (then zeroed for next time)
#pragma unroll 4
    for (int j = sst; j < kDsBins / 4; j += kDsST) {
        uint4* g4 = reinterpret_cast<uint4*>(gh) + j;
        *reinterpret_cast<uint4*>(S.hist + 4 * j) = __ldcg(g4);
        __stcg(g4, make_uint4(0u, 0u, 0u, 0u));
    }
    const int NW = (N + 31) >> 5;
    for (int w = sst; w < NW; w += kDsST) S.sel[w] = S.tie[w] = 0u;
    if (sst == 0) *S.cand_n = 0u;
    sel_bar();
    if (k == 0) return;
    sel_find_bin((uint32_t)k, 0, sst, S);
    PassArg a{kPassFirst, S.bc[0], 0u, 0u};
    const uint32_t nD = (uint32_t)S.bc[2];
    const uint32_t krem = (uint32_t)k - (uint32_t)S.bc[1];

    // 2. one pass over the scores: digits above D are selected, digit D entries become candidates
    score_pass(a, sc, N, sst, S);
    const bool overflow = nD > (uint32_t)kDsCand;
    // 3. the threshold among the digit-D entries: bits 20..10, then 9..0, each a histogram
    // pass over the candidates (or over the scores again when the candidates overflowed)
    auto digit_pass = [&](int mode) {
        a.mode = mode;
        if (overflow) score_pass(a, sc, N, sst, S);
        else cand_pass(a, (int)nD, sst, S);
    };
    uint32_t ties_take = 0;
    if (krem == nD) {
        digit_pass(kPassSelD);
    } else {
        for (int j = sst; j < kDsBins; j += kDsST) S.hist[j] = 0u;
        sel_bar();
        digit_pass(kPassHist2);
        sel_find_bin(krem, 3, sst, S);
        a.p22 = ((uint32_t)a.D << 11) | (uint32_t)S.bc[3];
        const uint32_t krem2 = krem - (uint32_t)S.bc[4];
        if (krem2 == (uint32_t)S.bc[5]) {
            digit_pass(kPassSelP22);
        } else {
            for (int j = sst; j < kDsBins; j += kDsST) S.hist[j] = 0u;
            sel_bar();
            digit_pass(kPassHist3);
            sel_find_bin(krem2, 6, sst, S);
            a.thr = (a.p22 << 10) | (uint32_t)S.bc[6];
            const uint32_t krem3 = krem2 - (uint32_t)S.bc[7];
            if (krem3 == (uint32_t)S.bc[8]) {
                digit_pass(kPassSelThr);
            } else {
                ties_take = krem3;
                digit_pass(kPassSelTie);
            }
        }
    }

    // 4. emit ascending: the selected entries, and the first ties_take ties in index order
    const int wpt = (NW + kDsST - 1) / kDsST;
    const int w0 = min(NW, sst * wpt), w1 = min(NW, w0 + wpt);
    uint32_t cs = 0, ct = 0;
    for (int w = w0; w < w1; ++w) {
        cs += (uint32_t)__popc(S.sel[w]);
        ct += (uint32_t)__popc(S.tie[w]);
    }
    const uint32_t tie_before = sel_scan_excl(ct, sst, S, true);
    const uint32_t take = ties_take > tie_before ? min(ct, ties_take - tie_before) : 0u;
    uint32_t pos = sel_scan_excl(cs + take, sst, S, true);
    uint32_t taken = 0;
    for (int w = w0; w < w1; ++w) {
        uint32_t sw = S.sel[w], tw = S.tie[w];
        while (tw != 0u && taken < take) {
            const uint32_t low = tw & (0u - tw);
            sw |= low;
            tw ^= low;
            ++taken;
        }
        while (sw != 0u) {
            const int bit = __ffs(sw) - 1;
            if (pos < (uint32_t)k) out[pos] = w * 32 + bit;
            ++pos;
            sw &= sw - 1u;
        }
    }
}

// The group's output: the merge of its AG attention partials in task order.  All kDsST
// selection threads call it: the partials' (m, l) go to shared memory, warp u reduces rows
// u, u + kDsSelW, ... (the row maximum M and sum L over the partials) and turns each
// partial's m into its weight 2^(m - M) / L, then every (row, 4-column) pair sums its
// partials.
SD_DEVINL void merge_group(const DsParams& p, int g, int sst, const SelSmem& S) {
    const int NP = p.AG, R = p.R;
    const int lane = sst & 31, sw = sst >> 5;
    const int b = g / p.Hkv, kvh = g % p.Hkv;
    const size_t base = (size_t)g * NP * R;
    float2* ml = S.scratch;              // [NP * R]: (m, l), then (weight, -)
    float2* rowML = S.scratch + NP * R;  // [R]: (M, L)
    const float2* gml = reinterpret_cast<const float2*>(p.part_ml) + base;
    for (int e = sst; e < NP * R; e += kDsST) ml[e] = __ldcg(gml + e);
    sel_bar();
    for (int r = sw; r < R; r += kDsSelW) {
        float M = -INFINITY;
        for (int t = lane; t < NP; t += 32) M = fmaxf(M, ml[t * R + r].x);
        M = warp_max(M);
        float Ls = 0.f;
        for (int t = lane; t < NP; t += 32) {
            const float2 x = ml[t * R + r];
            if (x.x != -INFINITY) Ls = fmaf(x.y, exp2f(x.x - M), Ls);
        }
        Ls = warp_sum(Ls);
        for (int t = lane; t < NP; t += 32) {
            const float mt = ml[t * R + r].x;
            ml[t * R + r].x = (mt == -INFINITY || !(Ls > 0.f)) ? 0.f : exp2f(mt - M) / Ls;
        }
        if (lane == 0) rowML[r] = make_float2(M, Ls);
    }
    sel_bar();
    for (int pr = sst; pr < R * 32; pr += kDsST) {
        const int r = pr >> 5, c4 = pr & 31;
        const float4* po = reinterpret_cast<const float4*>(p.part_o + (base + r) * 128) + c4;
        float4 o = make_float4(0.f, 0.f, 0.f, 0.f);
        for (int t0 = 0; t0 < NP; t0 += 16) {
            float4 x[16];
#pragma unroll
            for (int u = 0; u < 16; ++u)
                x[u] = t0 + u < NP ? __ldcg(po + (size_t)(t0 + u) * R * 32) : make_float4(0.f, 0.f, 0.f, 0.f);
#pragma unroll
            for (int u = 0; u < 16; ++u) {
                const float wgt = t0 + u < NP ? ml[(t0 + u) * R + r].x : 0.f;
                o.x = fmaf(wgt, x[u].x, o.x);
                o.y = fmaf(wgt, x[u].y, o.y);
                o.z = fmaf(wgt, x[u].z, o.z);
                o.w = fmaf(wgt, x[u].w, o.w);
            }
        }
        const int v = r / p.G, gi = r % p.G;
        const size_t qrow = ((size_t)b * p.V + v) * p.Hq + (size_t)kvh * p.G + gi;
        reinterpret_cast<float4*>(p.out + qrow * 128)[c4] = o;
        if (c4 == 0) {
            const float2 x = rowML[r];
            p.lse[qrow] = x.y > 0.f ? (x.x + log2f(x.y)) * 0.69314718055994530942f : -INFINITY;
        }
    }
    sel_bar();  // the scratch may be reused after this
}

// ------------------------------------------------------------------ the kernel

template <bool F16>
__global__ void __launch_bounds__(kDsThreads, 1)
    decode_step_kernel(const __grid_constant__ CUtensorMap kmap, const __grid_constant__ CUtensorMap kvk,
                       const __grid_constant__ CUtensorMap kvv, const DsParams p) {
    using L = DsLayout;
    extern __shared__ uint8_t smem_raw[];
    const uint32_t raw = smem_addr(smem_raw);
    uint8_t* sm = smem_raw + ((1024u - (raw & 1023u)) & 1023u);
    uint64_t* full = reinterpret_cast<uint64_t*>(sm + L::oBars);
    uint64_t* empty = full + kDsStages;
    uint64_t* rec_full = empty + kDsStages;       // [4][kDsRecW]
    uint64_t* rec_free = rec_full + kDsCons * kDsRecW;
    uint64_t* cbar = rec_free + kDsCons * kDsRecW;
    StageMeta* meta = reinterpret_cast<StageMeta*>(sm + L::oMeta);
    int2* rec = reinterpret_cast<int2*>(sm + L::oRec);  // [4][kDsRecW]
    volatile int* jobs = reinterpret_cast<volatile int*>(sm + L::oJobs);  // [2][4][kDsJobsW]
    uint8_t* misc = sm + L::oMisc;
    volatile int* abort_flag = reinterpret_cast<volatile int*>(misc + kMiAbort);
    volatile int* busy = reinterpret_cast<volatile int*>(misc + kMiBusy);
    volatile int* work = reinterpret_cast<volatile int*>(misc + kMiWork);
    volatile uint32_t* consumed = reinterpret_cast<volatile uint32_t*>(misc + kMiConsumed);
    volatile uint32_t* issued = reinterpret_cast<volatile uint32_t*>(misc + kMiIssued);
    volatile uint32_t* jidx = reinterpret_cast<volatile uint32_t*>(misc + kMiJobIdx);  // [w][sel head, tail, mer head, tail]
    const uint64_t lim = p.wait_ns;

    const int tid = threadIdx.x, warp = tid >> 5, lane = tid & 31;
    if (tid == 0) {
        for (int s = 0; s < kDsStages; ++s) {
            mbar_init(&full[s], 32);
            mbar_init(&empty[s], 1);  // the pipeline's consumer warp
        }
        for (int r = 0; r < kDsCons * kDsRecW; ++r) {
            mbar_init(&rec_full[r], 1);
            mbar_init(&rec_free[r], 1);
        }
        mbar_init(&cbar[0], 1);
        mbar_init(&cbar[1], 1);
        for (int j = 0; j < L::kMisc / 4; ++j) reinterpret_cast<volatile uint32_t*>(misc)[j] = 0u;
        fence_mbarrier_init();
    }
    __syncthreads();
    pdl_wait();  // the inputs and the workspace counters are the preceding kernels' results

    if (warp >= kDsProd0 && warp < kDsProd0 + kDsCons) {
        // ------------------------------------------------------------ producer of pipeline w
        const int w = warp - kDsProd0;
        const uint64_t pol = l2_evict_first_policy();
        uint32_t n = 0;  // stages filled into the pipeline: stage n is slot 2w + (n & 1)
        bool ok = true;
        auto take_slot = [&]() -> int {  // the next free slot (all lanes), -1 on an abort
            const int s = 2 * w + (int)(n & 1u);
            return warp_wait(&empty[s], ((n >> 1) & 1u) ^ 1u, abort_flag, lim) ? s : -1;
        };
        // this CTA owns a selection (which 0) or merge (1) of group g: queued for the bookkeeper
        auto own = [&](int which, int g) -> bool {
            bool got = true;
            if (lane == 0) {
                volatile uint32_t* hd = jidx + 4 * w + 2 * which;  // head, tail
                volatile int* ring = jobs + (which * kDsCons + w) * kDsJobsW;
                if (hd[1] - hd[0] >= (uint32_t)kDsJobsW) {
                    const uint64_t t0 = globaltimer_ns();
                    while (hd[1] - hd[0] >= (uint32_t)kDsJobsW) {
                        __nanosleep(256);
                        if (*abort_flag || globaltimer_ns() - t0 > lim) {
                            got = false;
                            break;
                        }
                    }
                }
                if (got) {
                    ring[hd[1] % kDsJobsW] = g;
                    __threadfence_block();
                    hd[1] = hd[1] + 1u;
                }
            }
            return __shfl_sync(0xffffffffu, got ? 1 : 0, 0) != 0;
        };
        uint32_t t_next = 0, t_end = 0;  // the claimed tasks not yet started
        int ready_g = -1;                // the last group seen with its selection published
        while (ok) {
            if (t_next == t_end) {  // claim the next kDsClaim tasks of the list in one atomic
                uint32_t t0 = 0;
                if (lane == 0) t0 = atomicAdd(&p.ctrl[0], (uint32_t)kDsClaim);
                t_next = __shfl_sync(0xffffffffu, t0, 0);
                t_end = t_next + kDsClaim;
            }
            const uint32_t t = t_next++;
            if (t >= p.total) {  // the pipeline's end marker
                const int s = take_slot();
                if (s < 0) {
                    ok = false;
                    break;
                }
                if (lane == 0) meta[s].kind = kTaskEnd;
                __syncwarp();
                mbar_arrive(&full[s]);
                ++n;
                break;
            }
            const Task tk = decode_task(p, t);
            if (tk.kind == kTaskScore) {
                if (tk.part == p.SG - 1 && !own(0, tk.g)) {
                    ok = false;
                    break;
                }
                const int j0t = tk.part * kDsTaskKeys;
                const int nst = min(kDsScoreStages, (p.N - j0t + kDsKeyRows - 1) / kDsKeyRows);
                for (int sgi = 0; sgi < nst; ++sgi) {
                    const int s = take_slot();
                    if (s < 0) {
                        ok = false;
                        break;
                    }
                    uint8_t* st = sm + s * kDsStage;
                    const int j0 = j0t + sgi * kDsKeyRows;
                    if (lane == 0) {
                        StageMeta& m = meta[s];
                        m.kind = kTaskScore;
                        m.g = tk.g;
                        m.j0 = j0;
                        m.nrows = min(kDsKeyRows, p.N - j0);
                        m.sgi = sgi;
                        m.nst = nst;
                        const uint32_t qb = (uint32_t)p.V * 256u;
                        mbar_arrive_expect_tx(&full[s], kDsData + qb);
                        const int row = tk.g * p.N + j0;
                        tma_load_2d_hint(st, &kmap, 0, row, &full[s], pol);
                        tma_load_2d_hint(st + kDsData / 2, &kmap, 64, row, &full[s], pol);
                        bulk_g2s(st + kDsData, p.q_idx + (size_t)tk.g * qb, qb, &full[s]);
                    } else {
                        mbar_arrive(&full[s]);
                    }
                    ++n;
                }
                continue;
            }
            if (tk.part == p.AG - 1 && !own(1, tk.g)) {
                ok = false;
                break;
            }
            // attention task: wait for the group's selection (published once per launch: a group
            // seen ready stays ready until its last attention task is done)
            if (tk.g != ready_g) {
                uint32_t* ready = p.gstate + (size_t)tk.g * 4 + 2;
                bool got = true;
                if (lane == 0 && ld_acquire_gpu(ready) == 0u) {
                    const uint64_t t0 = globaltimer_ns();
                    for (;;) {
                        __nanosleep(256);
                        if (ld_acquire_gpu(ready) != 0u) break;
                        if (*abort_flag || globaltimer_ns() - t0 > lim) {
                            got = false;
                            break;
                        }
                    }
                }
                if (__shfl_sync(0xffffffffu, got ? 1 : 0, 0) == 0) {
                    ok = false;
                    break;
                }
                (void)ld_acquire_gpu(ready);  // every lane reads the selection after this
                ready_g = tk.g;
            }
            const int g = tk.g, b = g / p.Hkv, kvh = g % p.Hkv;
            const int r0 = tk.part * kDsTaskRows;
            const int rows = max(0, min(kDsTaskRows, p.n_rows - r0));
            const int nst = rows > 0 ? (rows + kDsRows - 1) / kDsRows : 1;
            const uint32_t qbytes = (uint32_t)p.G * 256u;
            const int32_t* sel_row = p.idx + (size_t)g * p.k;
            // every selected row of the task at once (one round trip): lane l resolves task row
            // 32q + l, q < kDsTaskStages, to its K/V row (-1: none, or skipped as out of range)
            long long src[kDsTaskStages];
#pragma unroll
            for (int q = 0; q < kDsTaskStages; ++q) {
                const int jr = 32 * q + lane;
                src[q] = -1;
                if (jr < rows) {
                    const int j = r0 + jr;
                    const int e = j / p.block;
                    const int sel = __ldcg(sel_row + e);
                    if (sel >= 0 && sel < p.N)
                        src[q] = (long long)g * p.T + (long long)sel * p.block + (j - e * p.block);
                    else
                        report(p.err, SD_DEVERR_INDEX);
                }
            }
#pragma unroll
            for (int sgi = 0; sgi < kDsTaskStages; ++sgi) {
                if (sgi >= nst || !ok) break;
                const int s = take_slot();
                if (s < 0) {
                    ok = false;
                    break;
                }
                uint8_t* st = sm + s * kDsStage;
                const int nrows = max(0, min(kDsRows, rows - sgi * kDsRows));
                const long long ra = src[sgi];
                // one contiguous run of 32 rows (an aligned part of one block)?
                long long run0 = -1;
                if (p.tma_blocks && nrows == kDsRows) run0 = __shfl_sync(0xffffffffu, ra, 0);
                const uint32_t valid = __ballot_sync(0xffffffffu, ra >= 0);
                if (lane == 0) {
                    StageMeta& m = meta[s];
                    m.kind = kTaskAttend;
                    m.g = g;
                    m.task = tk.part;
                    m.j0 = r0 + sgi * kDsRows;
                    m.nrows = nrows;
                    m.sgi = sgi;
                    m.nst = nst;
                    m.valid = run0 >= 0 ? 0xffffffffu : valid;
                }
                if (run0 >= 0) {
                    if (lane == 0) {
                        mbar_arrive_expect_tx(&full[s], kDsData + (uint32_t)p.V * qbytes);
                        tma_load_2d_hint(st, &kvk, 0, (int)run0, &full[s], pol);
                        tma_load_2d_hint(st + 4096, &kvk, 64, (int)run0, &full[s], pol);
                        tma_load_2d_hint(st + 8192, &kvv, 0, (int)run0, &full[s], pol);
                        tma_load_2d_hint(st + 12288, &kvv, 64, (int)run0, &full[s], pol);
                        for (int v = 0; v < p.V; ++v)
                            bulk_g2s(st + kDsData + v * qbytes,
                                     p.q + (((size_t)b * p.V + v) * p.Hq + (size_t)kvh * p.G) * 256, qbytes, &full[s]);
                    } else {
                        mbar_arrive(&full[s]);
                    }
                } else {
                    if (lane == 0) {
                        mbar_expect_tx(&full[s], (uint32_t)p.V * qbytes);
                        for (int v = 0; v < p.V; ++v)
                            bulk_g2s(st + kDsData + v * qbytes,
                                     p.q + (((size_t)b * p.V + v) * p.Hq + (size_t)kvh * p.G) * 256, qbytes, &full[s]);
                    }
                    // lanes 8q .. 8q + 7 move one 128-byte line of row 4i + q (zeros for rows skipped)
                    const int c = lane & 7;
#pragma unroll
                    for (int it = 0; it < 8; ++it) {
                        const int row = 4 * it + (lane >> 3);
                        const long long sr = __shfl_sync(0xffffffffu, ra, row);
                        const bool on = sr >= 0;
                        const size_t off = on ? ((size_t)sr * 128 + (size_t)c * 8) * 2 : 0;
#pragma unroll
                        for (int h = 0; h < 2; ++h) {
                            const uint32_t dst = swz(kDsRows, row, 8 * h + c);
                            cp_async16_zfill(st + dst, p.kc + off + h * 128, on ? 16u : 0u);
                            cp_async16_zfill(st + kDsData / 2 + dst, p.vc + off + h * 128, on ? 16u : 0u);
                        }
                    }
                    // lanes 1-31 arrive when their copies land; lane 0 holds the phase open until
                    // its copies land too and arrives itself (release: publishes the metadata)
                    if (lane == 0) {
                        cp_async_mbar_arrive(&full[s]);
                        mbar_arrive(&full[s]);
                    } else {
                        cp_async_mbar_arrive_noinc(&full[s]);
                    }
                }
                ++n;
            }
        }
        if (!ok) *abort_flag = 1;
        if (lane == 0) issued[w] = n;
    } else if (warp < kDsCons) {
        // ------------------------------------------------------------ consumer of pipeline w
        const int w = warp;
        float* sbuf = reinterpret_cast<float*>(sm + L::oScore) + w * 64;
        uint32_t qf[8][4];
        AttAcc acc;
        const bool two_halves = p.R > 8;
        bool ok = true;
        uint32_t nrec = 0;  // records posted
        for (uint32_t n = 0;; ++n) {
            const int s = 2 * w + (int)(n & 1u);
            if (!warp_wait(&full[s], (n >> 1) & 1u, abort_flag, lim)) {
                ok = false;
                break;
            }
            const StageMeta m = meta[s];
            const uint8_t* st = sm + s * kDsStage;
            bool post = m.kind == kTaskEnd;
            if (m.kind == kTaskScore) {
                score_tile<F16>(smem_addr(st), smem_addr(st + kDsData), lane, p.V, sbuf);
                __syncwarp();
                if (lane == 0) mbar_arrive(&empty[s]);
#pragma unroll
                for (int h = 0; h < 2; ++h) {
                    const int rl = 32 * h + lane;
                    const bool in = rl < m.nrows;
                    const float v = sbuf[rl];
                    if (in) p.scores[(size_t)m.g * p.N + m.j0 + rl] = v;
                    const uint32_t dg = float_key(v) >> 21;
                    const uint32_t peers = __match_any_sync(0xffffffffu, in ? dg : 0xffffffffu);
                    if (in && lane == __ffs(peers) - 1)
                        atomicAdd(&p.hist[(size_t)m.g * kDsBins + dg], (uint32_t)__popc(peers));
                }
                post = m.sgi == m.nst - 1;
            } else if (m.kind == kTaskAttend) {
                load_q_frags(smem_addr(st + kDsData), lane, p.R, qf);
                if (m.sgi == 0) {
#pragma unroll
                    for (int nt = 0; nt < 16; ++nt)
#pragma unroll
                        for (int e = 0; e < 4; ++e) acc.o[nt][e] = 0.f;
                    acc.m[0] = acc.m[1] = -INFINITY;
                    acc.l[0] = acc.l[1] = 0.f;
                }
                attend_stage(smem_addr(st), smem_addr(st) + kDsData / 2, lane, qf, two_halves, m.valid, p.scale_log2, acc);
                __syncwarp();
                if (lane == 0) mbar_arrive(&empty[s]);
                if (m.sgi == m.nst - 1) {  // the task's partial
                    const int g8 = lane >> 2, t4 = lane & 3;
                    const size_t pb = ((size_t)m.g * p.AG + m.task) * p.R;
#pragma unroll
                    for (int hf = 0; hf < 2; ++hf) {
                        const int r = g8 + 8 * hf;
                        if (r >= p.R) continue;
#pragma unroll
                        for (int nt = 0; nt < 16; ++nt)
                            *reinterpret_cast<float2*>(p.part_o + (pb + r) * 128 + 8 * nt + 2 * t4) =
                                make_float2(acc.o[nt][2 * hf], acc.o[nt][2 * hf + 1]);
                        if (t4 == 0)
                            *reinterpret_cast<float2*>(p.part_ml + (pb + r) * 2) = make_float2(acc.m[hf], acc.l[hf]);
                    }
                    post = true;
                }
            }
            if (lane == 0) consumed[w] = n + 1;
            if (post) {  // the task's record: its kind and group (an end marker for kTaskEnd)
                const int slot = w * kDsRecW + (int)(nrec % kDsRecW);
                if (nrec >= (uint32_t)kDsRecW &&
                    !warp_wait(&rec_free[slot], ((nrec / kDsRecW) & 1u) ^ 1u, abort_flag, lim)) {
                    ok = false;
                    break;
                }
                if (lane == 0) rec[slot] = make_int2(m.kind, m.g);
                __syncwarp();  // the warp's stores before its arrival (release)
                if (lane == 0) mbar_arrive(&rec_full[slot]);
                ++nrec;
            }
            if (m.kind == kTaskEnd) break;
        }
        if (!ok) *abort_flag = 1;
    } else if (warp == kDsBook) {
        // ------------------------------------------------------------ bookkeeping
        uint32_t ra[kDsCons] = {0u, 0u, 0u, 0u};  // records taken per pipeline
        int ends = 0;
        uint64_t last_progress = globaltimer_ns();
        bool fin = false;
        while (!fin) {
            bool progress = false;
            // 1. the records each pipeline posted so far move the groups' counters: one fence for
            // the batch (release of the consumers' stores behind the records), then plain adds
#pragma unroll
            for (int w = 0; w < kDsCons; ++w) {
                int nb = 0;
                if (lane == 0)
                    while (nb < kDsRecW && mbar_try_wait(&rec_full[w * kDsRecW + (ra[w] + nb) % kDsRecW],
                                                         ((ra[w] + nb) / kDsRecW) & 1u))
                        ++nb;
                nb = __shfl_sync(0xffffffffu, nb, 0);
                if (nb == 0) continue;
                progress = true;
                int kind = -1, gg = 0;
                if (lane < nb) {
                    const int r = w * kDsRecW + (int)((ra[w] + lane) % kDsRecW);
                    (void)mbar_try_wait(&rec_full[r], ((ra[w] + lane) / kDsRecW) & 1u);  // acquire
                    const int2 rc = rec[r];
                    kind = rc.x;
                    gg = rc.y;
                    mbar_arrive(&rec_free[r]);
                }
                fence_acq_rel_gpu();
                if (lane < nb && kind != kTaskEnd)
                    atomicAdd(&p.gstate[(size_t)gg * 4 + (kind == kTaskScore ? 0 : 1)], 1u);
                ends += __popc(__ballot_sync(0xffffffffu, lane < nb && kind == kTaskEnd));
                ra[w] += (uint32_t)nb;
            }
            // 2. when the selection warps are idle: an owned selection or merge whose group is
            // complete (acquire), or the end
            int post = -1, pg = 0;
            if (lane == 0 && *busy == 0) {
                bool pending = false;
                for (int which = 0; which < 2 && post < 0; ++which)
                    for (int w = 0; w < kDsCons && post < 0; ++w) {
                        volatile uint32_t* hd = jidx + 4 * w + 2 * which;
                        if (hd[0] == hd[1]) continue;
                        pending = true;
                        __threadfence_block();
                        const int g = jobs[(which * kDsCons + w) * kDsJobsW + hd[0] % kDsJobsW];
                        const uint32_t target = (uint32_t)(which == 0 ? p.SG : p.AG);
                        if (ld_acquire_gpu(&p.gstate[(size_t)g * 4 + which]) == target) {
                            post = which == 0 ? kTaskScore : kTaskAttend;
                            pg = g;
                            hd[0] = hd[0] + 1u;
                        }
                    }
                const uint64_t now = globaltimer_ns();
                if (post >= 0 || progress) {
                    last_progress = now;
                } else if (ends == kDsCons && !pending) {
                    post = kTaskFin;  // no more records, no owned work left
                } else if (*abort_flag || now - last_progress > lim) {
                    *abort_flag = 1;
                    post = kTaskFin;
                }
            } else if (lane == 0 && (*abort_flag || globaltimer_ns() - last_progress > lim)) {
                // the selection warps are busy; on an abort, wait for them (bounded) and end
                const uint64_t t0 = globaltimer_ns();
                while (*busy != 0 && globaltimer_ns() - t0 < lim) __nanosleep(256);
                *abort_flag = 1;
                post = kTaskFin;
            }
            post = __shfl_sync(0xffffffffu, post, 0);
            pg = __shfl_sync(0xffffffffu, pg, 0);
            if (post >= 0) {
                if (lane == 0) {
                    work[0] = post;
                    work[1] = pg;
                    *busy = 1;
                    __threadfence_block();
                }
                __syncwarp();
                // hand it to the selection warps (they wait at barrier 2)
                asm volatile("bar.arrive 2, %0;" ::"n"(32 + kDsST) : "memory");
                fin = post == kTaskFin;
            } else if (!progress) {
                __nanosleep(64);
            }
        }
    } else {
        // ------------------------------------------------------------ selection
        const int sst = tid - 32 * kDsSel0;
        SelSmem S;
        S.hist = reinterpret_cast<uint32_t*>(sm + L::oHist);
        S.sel = reinterpret_cast<uint32_t*>(sm + L::oSel);
        S.tie = reinterpret_cast<uint32_t*>(sm + L::oTie);
        S.cidx = reinterpret_cast<int32_t*>(sm + L::oCandIdx);
        S.ckey = reinterpret_cast<uint32_t*>(sm + L::oCandKey);
        S.scratch = reinterpret_cast<float2*>(sm + L::oHist);
        S.chunk = reinterpret_cast<float*>(sm + L::oChunk);
        S.cbar = cbar;
        S.cpar = reinterpret_cast<volatile uint32_t*>(misc + kMiCpar);
        S.cand_n = reinterpret_cast<volatile uint32_t*>(misc + kMiCandN);
        S.bc = reinterpret_cast<int*>(misc + kMiBc);
        S.wt = reinterpret_cast<uint32_t*>(misc + kMiWt);
        S.abort_flag = abort_flag;
        S.lim = lim;
        for (;;) {
            asm volatile("bar.sync 2, %0;" ::"n"(32 + kDsST) : "memory");  // the bookkeeper's hand-off
            const int wk = work[0], wg = work[1];
            if (wk == kTaskFin) break;
            if (wk == kTaskScore) {
                select_group(p, wg, sst, S);
                sel_bar();  // every part of the selection is written: publish it
                if (sst == 0) {
                    p.gstate[(size_t)wg * 4 + 0] = 0u;
                    fence_acq_rel_gpu();
                    st_release_gpu(p.gstate + (size_t)wg * 4 + 2, 1u);
                }
            } else {
                merge_group(p, wg, sst, S);
                if (sst == 0) {
                    p.gstate[(size_t)wg * 4 + 1] = 0u;
                    p.gstate[(size_t)wg * 4 + 2] = 0u;
                }
            }
            sel_bar();
            if (sst == 0) {
                __threadfence_block();
                *busy = 0;
            }
        }
    }

    __syncthreads();
    if (tid == 0) {
        if (*abort_flag) {
            report(p.err, SD_DEVERR_TIMEOUT);
            // let the stages filled but not consumed land before the CTA exits
            for (int w = 0; w < kDsCons; ++w)
                for (uint32_t j = consumed[w]; j < issued[w]; ++j)
                    mbar_wait(&full[2 * w + (int)(j & 1u)], (j >> 1) & 1u, lim);
        }
        // the last CTA to finish resets the task counter for the next call
        __threadfence();
        if (atomicAdd(&p.ctrl[1], 1u) == gridDim.x - 1u) {
            p.ctrl[0] = 0u;
            p.ctrl[1] = 0u;
        }
    }
}

}  // namespace

namespace {

struct StepPlan {
    int NG, N, SG, AG, R, L, n_rows;
    size_t o_gstate, o_hist, o_part_o, o_part_ml, bytes;
};

size_t round256(size_t x) { return (x + 255) & ~size_t(255); }

StepPlan plan_step(const sd_decode_step_args* a) {
    StepPlan sp{};
    sp.NG = a->B * a->Hkv;
    sp.N = a->block > 0 ? a->T / a->block : 0;
    sp.SG = std::max(1, (sp.N + kDsTaskKeys - 1) / kDsTaskKeys);
    sp.n_rows = a->n_idx * a->block;
    sp.AG = std::max(1, (sp.n_rows + kDsTaskRows - 1) / kDsTaskRows);
    sp.R = (a->Hkv > 0 ? a->Hq / a->Hkv : 0) * a->V;
    if (a->lag > 0) {
        sp.L = a->lag;
    } else {
        // the lag covers ~15 us of the whole GPU's streaming (a group's selection and the
        // latency of its last scoring stages) at ~6.5 TB/s
        const double unit_bytes = (double)sp.N * 256.0 + (double)sp.n_rows * 512.0;
        const double unit_us = unit_bytes / 6.5e6;
        sp.L = (int)std::ceil(15.0 / std::max(unit_us, 1e-3));
    }
    sp.L = std::max(1, std::min(sp.L, std::max(1, sp.NG)));
    size_t off = 256;  // ctrl
    sp.o_gstate = off;
    off += round256((size_t)sp.NG * 16);
    sp.o_hist = off;
    off += round256((size_t)sp.NG * kDsBins * 4);
    sp.o_part_o = off;
    off += round256((size_t)sp.NG * sp.AG * sp.R * 128 * 4);
    sp.o_part_ml = off;
    off += round256((size_t)sp.NG * sp.AG * sp.R * 2 * 4);
    sp.bytes = off;
    return sp;
}

sd_status validate_step(const sd_decode_step_args* a) {
    const char* who = "sd_decode_step";
    SD_REQUIRE(a != nullptr, "%s: null args", who);
    SD_REQUIRE(a->B >= 0 && a->V >= 1 && a->Hq >= 1 && a->Hkv >= 1 && a->T >= 1 && a->block >= 1 && a->n_idx >= 0,
               "%s: bad sizes (B=%d V=%d Hq=%d Hkv=%d T=%d block=%d n_idx=%d)", who, a->B, a->V, a->Hq, a->Hkv,
               a->T, a->block, a->n_idx);
    SD_REQUIRE(a->Hq % a->Hkv == 0, "%s: Hq must be a multiple of Hkv", who);
    SD_REQUIRE(a->T % a->block == 0, "%s: T must be a multiple of block", who);
    SD_REQUIRE(a->n_idx <= a->T / a->block, "%s: n_idx must be <= T / block", who);
    SD_REQUIRE(a->key_dtype == SD_BF16 || a->key_dtype == SD_F16, "%s: key_dtype must be SD_BF16 or SD_F16", who);
    SD_REQUIRE(a->lag >= 0, "%s: lag must be >= 0", who);
    if (a->d != 128 || a->d_idx != 128) {
        set_error("%s: d and d_idx must be 128 (got %d, %d)", who, a->d, a->d_idx);
        return SD_ERR_UNSUPPORTED;
    }
    if (a->V > 8 || (a->Hq / a->Hkv) * a->V > kDsMaxR) {
        set_error("%s: V <= 8 and (Hq/Hkv)*V <= %d query rows per group are supported", who, kDsMaxR);
        return SD_ERR_UNSUPPORTED;
    }
    const int N = a->T / a->block;
    if (N > kDsMaxN || (N & 3) != 0) {
        set_error("%s: T / block must be a multiple of 4 and at most %d (got %d)", who, kDsMaxN, N);
        return SD_ERR_UNSUPPORTED;
    }
    SD_REQUIRE((long long)a->B * a->Hkv * a->T < (1LL << 31), "%s: B*Hkv*T must be < 2^31", who);
    SD_REQUIRE((long long)a->n_idx * a->block <= (1LL << 30), "%s: selection too large", who);
    const long long ag = std::max(1LL, ((long long)a->n_idx * a->block + kDsTaskRows - 1) / kDsTaskRows);
    if (ag * (a->Hq / a->Hkv) * a->V > kDsMaxMerge) {
        set_error("%s: %lld selected rows per group with %d query rows exceed the merge (at most %d (partial, row) pairs)",
                  who, (long long)a->n_idx * a->block, (a->Hq / a->Hkv) * a->V, kDsMaxMerge);
        return SD_ERR_UNSUPPORTED;
    }
    return SD_OK;
}

}  // namespace
}  // namespace sd

using namespace sd;

extern "C" size_t sd_decode_step_workspace_bytes(const sd_decode_step_args* a) {
    if (validate_step(a) != SD_OK) return 0;
    return plan_step(a).bytes;
}

extern "C" sd_status sd_decode_step(const sd_decode_step_args* a, void* stream) {
    clear_error();
    const sd_status vs = validate_step(a);
    if (vs != SD_OK) return vs;
    if (a->B == 0) return SD_OK;
    const char* who = "sd_decode_step";
    SD_REQUIRE(a->q_idx && a->keys && a->q && a->k_cache && a->v_cache && a->scores && a->out && a->lse &&
                   (a->idx || a->n_idx == 0),
               "%s: null pointer argument", who);
    SD_REQUIRE(aligned16(a->q_idx) && aligned16(a->keys) && aligned16(a->q) && aligned16(a->k_cache) &&
                   aligned16(a->v_cache) && aligned16(a->out) && aligned16(a->scores),
               "%s: q_idx, keys, q, k_cache, v_cache, scores and out must be 16-byte aligned", who);
    const StepPlan sp = plan_step(a);
    SD_REQUIRE(a->workspace != nullptr && a->workspace_bytes >= sp.bytes,
               "%s: workspace of %zu bytes needed (got %zu)", who, sp.bytes, a->workspace_bytes);
    SD_REQUIRE((reinterpret_cast<uintptr_t>(a->workspace) & 255u) == 0, "%s: workspace must be 256-byte aligned", who);
    if (block_step_eligible(a)) return block_step_launch(a, as_stream(stream));
    const bool f16 = a->key_dtype == SD_F16;
    CUtensorMap kmap, kvk, kvv;
    if (!make_tensor_map_2d(&kmap, a->keys, (uint64_t)sp.NG * sp.N, 128, kDsKeyRows, f16) ||
        !make_tensor_map_2d(&kvk, a->k_cache, (uint64_t)sp.NG * a->T, 128, kDsRows, false) ||
        !make_tensor_map_2d(&kvv, a->v_cache, (uint64_t)sp.NG * a->T, 128, kDsRows, false)) {
        set_error("%s: cuTensorMapEncodeTiled failed", who);
        return SD_ERR_CUDA;
    }
    uint8_t* ws = static_cast<uint8_t*>(a->workspace);
    DsParams p{};
    p.q_idx = static_cast<const uint8_t*>(a->q_idx);
    p.q = static_cast<const uint8_t*>(a->q);
    p.kc = static_cast<const uint8_t*>(a->k_cache);
    p.vc = static_cast<const uint8_t*>(a->v_cache);
    p.scores = a->scores;
    p.idx = a->idx;
    p.out = a->out;
    p.lse = a->lse;
    p.err = a->err_word;
    p.ctrl = reinterpret_cast<uint32_t*>(ws);
    p.gstate = reinterpret_cast<uint32_t*>(ws + sp.o_gstate);
    p.hist = reinterpret_cast<uint32_t*>(ws + sp.o_hist);
    p.part_o = reinterpret_cast<float*>(ws + sp.o_part_o);
    p.part_ml = reinterpret_cast<float*>(ws + sp.o_part_ml);
    p.B = a->B;
    p.V = a->V;
    p.Hq = a->Hq;
    p.Hkv = a->Hkv;
    p.G = a->Hq / a->Hkv;
    p.R = sp.R;
    p.T = a->T;
    p.N = sp.N;
    p.k = a->n_idx;
    p.block = a->block;
    p.NG = sp.NG;
    p.SG = sp.SG;
    p.AG = sp.AG;
    p.L = sp.L;
    p.n_rows = sp.n_rows;
    p.tma_blocks = a->block % kDsRows == 0 ? 1 : 0;
    p.scale_log2 = a->scale * 1.44269504088896340736f;
    p.wait_ns = a->wait_limit_ns > 0 ? (unsigned long long)a->wait_limit_ns : (unsigned long long)kWaitDeadlineNs;
    SD_REQUIRE((long long)sp.NG * (sp.SG + sp.AG) < (1LL << 31) - 64, "%s: too many tasks", who);
    p.total = (uint32_t)((long long)sp.NG * (sp.SG + sp.AG));
    auto kern = f16 ? decode_step_kernel<true> : decode_step_kernel<false>;
    SD_CUDA_CHECK(cudaFuncSetAttribute(kern, cudaFuncAttributeMaxDynamicSharedMemorySize, DsLayout::kBytes),
                  "sd_decode_step: cudaFuncSetAttribute");
    const unsigned grid = (unsigned)std::max(1, std::min(num_sms(), (int)std::min<long long>(p.total, 1 << 30)));
    SD_CUDA_CHECK(launch_pdl(kern, dim3(grid), dim3(kDsThreads), (size_t)DsLayout::kBytes, as_stream(stream), kmap,
                             kvk, kvv, p),
                  "sd_decode_step: launch");
    return launch_status(who);
}
