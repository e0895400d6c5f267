// topk.cu -- exact top-k per row, ties to the lower index, ascending output.
//
// "Esparsidade de Contexto no Tempo de Inferencia" (gist.science summary), sec. 2
// "Mecanismos de Esparsidade": Oracle Top-K is the exact selection of the k highest-
// scoring tokens; SparDA (gist.science summary), sec. 2 item 1, selects top-k blocks the
// same way.  The pages are silent on ties; the lower index wins.
//
// Rows of at most 4096 entries: one 256-thread CTA per row, the row in registers, four 8-bit
// radix passes (topk_small_kernel).
// Rows of 16384 entries or more, when clusters of two or more CTAs per row fit in one wave,
// go to the cluster selection of select_attend.cu (each CTA owns a part of the row; the
// digits are summed over distributed shared memory).  Otherwise one CTA per row (1024
// threads; 512 threads, two CTAs per SM, when the rows outnumber the SMs and the first
// digit's histogram is given).  Scores become order-preserving
// uint32 keys (kept in shared memory when the row fits and several passes read it).  A radix select with 11/11/10-bit digits finds the
// k-th largest key `thr` and how many entries equal to it are still needed (`krem`).  A
// final ordered pass gives each warp a contiguous segment of the row: per-warp counts,
// a 32-entry scan, and warp ballots emit every key > thr and the first krem keys == thr
// in ascending index order.
#include <algorithm>

#include "sd_common.cuh"
#include "sd_host.h"

namespace sd {
namespace {

constexpr int kTkThreads = 1024;  // threads of the plain kernel, and the most any variant has
constexpr int kTkWarps = kTkThreads / 32;
constexpr int kHistBins = 2048;

// Block-wide inclusive prefix sum of one value per thread (NT threads).
template <int NT>
SD_DEVINL uint32_t block_inclusive_scan(uint32_t v, uint32_t* wsum) {
    const int lane = threadIdx.x & 31, warp = threadIdx.x >> 5;
#pragma unroll
    for (int o = 1; o < 32; o <<= 1) {
        const uint32_t n = __shfl_up_sync(0xffffffffu, v, o);
        if (lane >= o) v += n;
    }
    if (lane == 31) wsum[warp] = v;
    __syncthreads();
    if (warp == 0) {
        uint32_t w = lane < NT / 32 ? wsum[lane] : 0u;
#pragma unroll
        for (int o = 1; o < 32; o <<= 1) {
            const uint32_t n = __shfl_up_sync(0xffffffffu, w, o);
            if (lane >= o) w += n;
        }
        wsum[lane] = w;
    }
    __syncthreads();
    const uint32_t off = warp > 0 ? wsum[warp - 1] : 0u;
    __syncthreads();
    return v + off;
}

struct TopkShared {
    uint32_t hist[kHistBins];
    uint32_t wsum[32];
    uint32_t sel_digit, sel_above, cand_n;
    uint32_t cnt_gt[kTkWarps], cnt_eq[kTkWarps], base_out[kTkWarps], eq_before[kTkWarps];
};

// Given the histogram of one digit (nb bins, higher bins = larger keys) of the entries
// still in the running, pick the digit holding the krem-th largest: returns it and how
// many of those entries lie in higher bins.  Thread t owns bins [nb - per*(t+1), nb - per*t).
template <int NT>
SD_DEVINL void select_digit(TopkShared& sh, uint32_t nb, int krem, uint32_t& digit, uint32_t& above) {
    const int tid = threadIdx.x;
    if (tid == 0) {  // defined even if no bin crosses (a histogram that does not match)
        sh.sel_digit = 0;
        sh.sel_above = 0;
    }
    const int per = (int)nb / NT;
    const int hi = (int)nb - per * tid;
    uint32_t local = 0;
    for (int b = hi - per; b < hi; ++b) local += sh.hist[b];
    const uint32_t incl = block_inclusive_scan<NT>(local, sh.wsum);
    const uint32_t excl = incl - local;
    if (excl < (uint32_t)krem && (uint32_t)krem <= incl) {
        uint32_t acc = excl;
        for (int b = hi - 1; b >= hi - per; --b) {
            if (acc + sh.hist[b] >= (uint32_t)krem) {
                sh.sel_digit = (uint32_t)b;
                sh.sel_above = acc;
                break;
            }
            acc += sh.hist[b];
        }
    }
    __syncthreads();
    digit = sh.sel_digit;
    above = sh.sel_above;
    __syncthreads();
}

// Histogram pass over all N keys: counts the digit (kk >> shift) & (nb - 1) of every key
// whose bits under pmask equal prefix (warp-aggregated shared atomics).
template <int NT, typename KeyAt>
SD_DEVINL void hist_pass_all(TopkShared& sh, KeyAt key_at, int N, uint32_t prefix, uint32_t pmask,
                             int shift, uint32_t nb) {
    const int tid = threadIdx.x, lane = tid & 31, warp = tid >> 5;
    for (int b = tid; b < kHistBins; b += NT) sh.hist[b] = 0;
    __syncthreads();
    for (int base = warp * 32; base < N; base += NT) {
        const int i = base + lane;
        const bool valid = i < N;
        const uint32_t kk = valid ? key_at(i) : 0u;
        const bool in = valid && (kk & pmask) == prefix;
        const uint32_t dg = (kk >> shift) & (nb - 1);
        const uint32_t peers = __match_any_sync(0xffffffffu, in ? dg : 0xffffffffu);
        if (in && lane == __ffs(peers) - 1) atomicAdd(&sh.hist[dg], (uint32_t)__popc(peers));
    }
    __syncthreads();
}

// Ordered emit: every key > thr and the first krem keys == thr (lowest indices), written
// in ascending index order.  Warp w scans the contiguous segment [w*seg, (w+1)*seg).
template <int NT, typename KeyAt>
SD_DEVINL void emit_selected(TopkShared& sh, KeyAt key_at, int N, int k, uint32_t thr, int krem,
                             int32_t* orow) {
    constexpr int NWP = NT / 32;
    const int tid = threadIdx.x, lane = tid & 31, warp = tid >> 5;
    const int seg = ((N + NWP - 1) / NWP + 31) / 32 * 32;
    const int s0 = warp * seg, s1 = min(N, s0 + seg);
    uint32_t gt = 0, eq = 0;
    for (int base = s0; base < s1; base += 32) {
        const int i = base + lane;
        const bool valid = i < s1;
        const uint32_t kk = valid ? key_at(i) : 0u;
        gt += __popc(__ballot_sync(0xffffffffu, valid && kk > thr));
        eq += __popc(__ballot_sync(0xffffffffu, valid && kk == thr));
    }
    if (lane == 0) {
        sh.cnt_gt[warp] = gt;
        sh.cnt_eq[warp] = eq;
    }
    __syncthreads();
    if (tid == 0) {
        uint32_t eqb = 0, ob = 0;
        for (int w = 0; w < NWP; ++w) {
            sh.eq_before[w] = eqb;
            const int take = max(0, min((int)sh.cnt_eq[w], krem - (int)eqb));
            sh.base_out[w] = ob;
            ob += sh.cnt_gt[w] + (uint32_t)take;
            eqb += sh.cnt_eq[w];
        }
    }
    __syncthreads();
    uint32_t eq_seen = sh.eq_before[warp], pos = sh.base_out[warp];
    const uint32_t lt = lanemask_lt();
    for (int base = s0; base < s1; base += 32) {
        const int i = base + lane;
        const bool valid = i < s1;
        const uint32_t kk = valid ? key_at(i) : 0u;
        const bool is_gt = valid && kk > thr;
        const bool is_eq = valid && kk == thr;
        const uint32_t eqm = __ballot_sync(0xffffffffu, is_eq);
        const bool sel = is_gt || (is_eq && (int)(eq_seen + __popc(eqm & lt)) < krem);
        const uint32_t selm = __ballot_sync(0xffffffffu, sel);
        const uint32_t at = pos + __popc(selm & lt);
        if (sel && at < (uint32_t)k) orow[at] = i;
        pos += __popc(selm);
        eq_seen += __popc(eqm);
    }
}

// Loads the scores of row `srow` (raw fp32 bits; order keys are made on use) into keys_s.
// A 16-byte aligned row goes in with one bulk copy (TMA) completed on `bar`; otherwise each
// thread loads 8 scores before storing any, so every thread keeps 8 loads in flight.
// Returns false (uniformly) if the bulk copy did not complete in time.
SD_DEVINL bool stage_keys(const float* srow, int N, uint32_t* keys_s, uint64_t* bar) {
    const int tid = threadIdx.x;
    const bool bulk = ((reinterpret_cast<uintptr_t>(srow) | (uintptr_t)(N * 4)) & 15u) == 0;
    if (bulk) {
        if (tid == 0) {
            mbar_init(bar, 1);
            fence_mbarrier_init();
            mbar_arrive_expect_tx(bar, (uint32_t)N * 4u);
            bulk_g2s(keys_s, srow, (uint32_t)N * 4u, bar);
        }
        __syncthreads();
        const bool ok = mbar_wait(bar, 0);
        if (__syncthreads_or(!ok)) return false;
    } else {
        for (int base = tid; base < N; base += 8 * kTkThreads) {
            float v[8];
#pragma unroll
            for (int u = 0; u < 8; ++u) {
                const int i = base + u * kTkThreads;
                v[u] = i < N ? srow[i] : 0.f;
            }
#pragma unroll
            for (int u = 0; u < 8; ++u) {
                const int i = base + u * kTkThreads;
                if (i < N) keys_s[i] = __float_as_uint(v[u]);
            }
        }
    }
    __syncthreads();
    return true;
}

// Digit layout of the 32-bit order key: 11 + 11 + 10 bits, most significant first.
__device__ constexpr int kShift[3] = {21, 10, 0};

// Plain variant: three histogram passes over the row, then the ordered emit.
__global__ void __launch_bounds__(kTkThreads, 1)
    topk_kernel(const float* __restrict__ scores, int N, int k, int32_t* __restrict__ idx_out,
                int cache_keys, int32_t* err_word) {
    extern __shared__ __align__(16) uint32_t keys_s[];
    __shared__ TopkShared sh;
    __shared__ __align__(8) uint64_t stage_bar;
    const int tid = threadIdx.x;
    const float* srow = scores + (size_t)blockIdx.x * N;
    int32_t* orow = idx_out + (size_t)blockIdx.x * k;
    pdl_wait();
    pdl_launch_dependents();
    if (k == 0) return;
    if (k == N) {
        for (int i = tid; i < N; i += kTkThreads) orow[i] = i;
        return;
    }
    if (cache_keys && !stage_keys(srow, N, keys_s, &stage_bar)) {
        if (tid == 0) report(err_word, SD_DEVERR_TIMEOUT);
        return;
    }
    auto key_at = [&](int i) -> uint32_t { return float_key(cache_keys ? __uint_as_float(keys_s[i]) : srow[i]); };
    uint32_t prefix = 0, pmask = 0;
    int krem = k;
#pragma unroll 1
    for (int pass = 0; pass < 3; ++pass) {
        const uint32_t nb = pass == 2 ? 1024u : 2048u;
        hist_pass_all<kTkThreads>(sh, key_at, N, prefix, pmask, kShift[pass], nb);
        uint32_t dg, above;
        select_digit<kTkThreads>(sh, nb, krem, dg, above);
        prefix |= dg << kShift[pass];
        pmask |= (nb - 1) << kShift[pass];
        krem -= (int)above;
    }
    emit_selected<kTkThreads>(sh, key_at, N, k, prefix, krem, orow);
}

// Short rows (N <= kSmallN): one 256-thread CTA per row holds the whole row in registers —
// warp w the entries [w*32*EPT, (w+1)*32*EPT), lane l those at 32j + l, so the loads coalesce
// whatever the row's alignment — and resolves the threshold key in four 8-bit radix passes
// over warp-private shared histograms (equal digits of a warp merged with one match, one
// atomic per distinct digit).  The emit goes in index order: one scan over the warps of the
// packed (above, equal) counts, then ballots within each warp.  A key histogram passed in is
// only cleared: ranking a row this short from registers costs less than reading the seed.
constexpr int kSmallThreads = 256;
constexpr int kSmallWarps = kSmallThreads / 32;
constexpr int kSmallN = 4096;

struct SmallShared {
    uint32_t h[2][kSmallWarps][256];  // per-warp histograms, alternating between passes
    uint32_t wtot[3][kSmallWarps];
    uint32_t dig[2], abv[2];
};

template <int EPT>
__global__ void __launch_bounds__(kSmallThreads)
    topk_small_kernel(const float* __restrict__ scores, int N, int k, int32_t* __restrict__ idx_out,
                      uint32_t* __restrict__ key_hist) {
    static_assert(kSmallThreads == 256, "thread t owns radix bin 255 - t");
    static_assert(kSmallWarps * 32 * EPT <= 65535, "packed 16-bit counts");
    __shared__ SmallShared sh;
    const int tid = threadIdx.x, lane = tid & 31, warp = tid >> 5;
    const float* srow = scores + (size_t)blockIdx.x * N;
    int32_t* orow = idx_out + (size_t)blockIdx.x * k;
    pdl_wait();
    pdl_launch_dependents();
    const int seg0 = warp * 32 * EPT;
    uint32_t kk[EPT];
#pragma unroll
    for (int j = 0; j < EPT; ++j) {
        const int i = seg0 + 32 * j + lane;
        kk[j] = i < N ? float_key(__ldcg(srow + i)) : 0u;
    }
    if (key_hist != nullptr) {
        uint32_t* hrow = key_hist + (size_t)blockIdx.x * kHistBins;
        for (int b = tid; b < kHistBins; b += kSmallThreads) hrow[b] = 0u;
    }
    if (k == 0) return;
    if (k == N) {
        for (int i = tid; i < N; i += kSmallThreads) orow[i] = i;
        return;
    }
    uint32_t prefix = 0, pmask = 0;
    int krem = k;
#pragma unroll 1
    for (int pass = 0; pass < 4; ++pass) {
        const int shift = 24 - 8 * pass, buf = pass & 1;
        uint32_t* wh = sh.h[buf][warp];
        // this buffer was last read two passes ago, before the barriers of the pass between
        for (int b = lane; b < 256; b += 32) wh[b] = 0u;
        __syncwarp();
#pragma unroll
        for (int j = 0; j < EPT; ++j) {
            const bool in = seg0 + 32 * j + lane < N && (kk[j] & pmask) == prefix;
            if (__any_sync(0xffffffffu, in)) {
                const uint32_t dg = (kk[j] >> shift) & 255u;
                const uint32_t peers = __match_any_sync(0xffffffffu, in ? dg : 0xffffffffu);
                if (in && lane == __ffs(peers) - 1) atomicAdd(&wh[dg], (uint32_t)__popc(peers));
            }
        }
        __syncthreads();
        // thread t owns bin 255 - t: an inclusive scan over t counts the keys at or above it
        const int bin = 255 - tid;
        uint32_t c = 0;
#pragma unroll
        for (int w = 0; w < kSmallWarps; ++w) c += sh.h[buf][w][bin];
        uint32_t incl = c;
#pragma unroll
        for (int o = 1; o < 32; o <<= 1) {
            const uint32_t n = __shfl_up_sync(0xffffffffu, incl, o);
            if (lane >= o) incl += n;
        }
        if (lane == 31) sh.wtot[buf][warp] = incl;
        __syncthreads();
        for (int w = 0; w < warp; ++w) incl += sh.wtot[buf][w];
        const uint32_t excl = incl - c;
        if (excl < (uint32_t)krem && (uint32_t)krem <= incl) {
            sh.dig[buf] = (uint32_t)bin;
            sh.abv[buf] = excl;
        }
        __syncthreads();
        prefix |= sh.dig[buf] << shift;
        pmask |= 255u << shift;
        krem -= (int)sh.abv[buf];
    }
    const uint32_t thr = prefix;
    uint32_t gt = 0, eq = 0;
#pragma unroll
    for (int j = 0; j < EPT; ++j) {
        const bool valid = seg0 + 32 * j + lane < N;
        gt += (valid && kk[j] > thr) ? 1u : 0u;
        eq += (valid && kk[j] == thr) ? 1u : 0u;
    }
    const uint32_t packed = __reduce_add_sync(0xffffffffu, (gt << 16) | eq);
    if (lane == 0) sh.wtot[2][warp] = packed;
    __syncthreads();
    uint32_t before = 0;
    for (int w = 0; w < warp; ++w) before += sh.wtot[2][w];
    uint32_t eq_seen = before & 0xffffu;
    uint32_t pos = (before >> 16) + min(eq_seen, (uint32_t)krem);
    const uint32_t lt = lanemask_lt();
#pragma unroll
    for (int j = 0; j < EPT; ++j) {
        const int i = seg0 + 32 * j + lane;
        const bool valid = i < N;
        const bool is_gt = valid && kk[j] > thr;
        const bool is_eq = valid && kk[j] == thr;
        const uint32_t eqm = __ballot_sync(0xffffffffu, is_eq);
        const bool sel = is_gt || (is_eq && eq_seen + __popc(eqm & lt) < (uint32_t)krem);
        const uint32_t selm = __ballot_sync(0xffffffffu, sel);
        const uint32_t at = pos + __popc(selm & lt);
        if (sel && at < (uint32_t)k) orow[at] = i;
        pos += __popc(selm);
        eq_seen += __popc(eqm);
    }
}

constexpr int kCandCap = 4096;
constexpr int kClusterMinN = 16384;  // rows at least this long go to the cluster selection

// Bits 0..7 of x moved to bits 0, 4, ..., 28 (the others cleared).
SD_DEVINL uint32_t spread8(uint32_t x) {
    x = (x | (x << 12)) & 0x000F000Fu;
    x = (x | (x << 6)) & 0x03030303u;
    return (x | (x << 3)) & 0x11111111u;
}

// Block-wide exclusive prefix sum of one value per thread; also returns the total.
template <int NT>
SD_DEVINL uint32_t block_exclusive_scan(uint32_t v, uint32_t* wsum, uint32_t& total) {
    const uint32_t incl = block_inclusive_scan<NT>(v, wsum);
    if ((int)threadIdx.x == NT - 1) wsum[0] = incl;
    __syncthreads();
    total = wsum[0];
    __syncthreads();
    return incl - v;
}

// Histogram-seeded variant, bitmap emit.  The first digit's histogram comes from
// sd_index_score and picks the top digit d0.  One pass over the row, read straight from
// global memory (the scores were just written, so mostly from L2), marks every entry whose
// digit is above d0 in a selection bitmap (a warp's 32 consecutive entries = one bitmap
// word, written from a ballot) and collects the entries of digit d0 (candidates, with their
// indices; a warp reserves the slots of 8 words with one shared atomic).  The last 21 bits are resolved
// among the candidates; candidates above the threshold join the bitmap, those equal to it
// go to a tie bitmap of which a prefix scan keeps the lowest-index ones still needed; a
// prefix scan over the selection bitmap writes the indices in ascending order.  Falls back
// to full passes when the candidates exceed their buffer.  Leaves the histogram zeroed.
template <int NT>
__global__ void __launch_bounds__(NT, kTkThreads / NT)
    topk_hist_kernel(const float* __restrict__ scores, int N, int k, int32_t* __restrict__ idx_out,
                     uint32_t* __restrict__ key_hist) {
    constexpr int NWP = NT / 32;
    extern __shared__ __align__(16) uint32_t dyn[];
    __shared__ TopkShared sh;
    const int NW = (N + 31) / 32;  // bitmap words
    uint32_t* cand_key = dyn;
    uint32_t* cand_idx = cand_key + kCandCap;
    uint32_t* sel = cand_idx + kCandCap;
    uint32_t* tie = sel + NW;
    const int tid = threadIdx.x, lane = tid & 31, warp = tid >> 5;
    const float* srow = scores + (size_t)blockIdx.x * N;
    int32_t* orow = idx_out + (size_t)blockIdx.x * k;
    uint32_t* hrow = key_hist + (size_t)blockIdx.x * kHistBins;
    pdl_wait();
    pdl_launch_dependents();
    {
        // every load before any store: a load queued behind the store to the same row of
        // bins, one at a time, cost ~4 us each
        static_assert(kHistBins % NT == 0, "bins per thread");
        uint32_t hv[kHistBins / NT];
#pragma unroll
        for (int i = 0; i < kHistBins / NT; ++i) hv[i] = __ldcg(hrow + tid + i * NT);
#pragma unroll
        for (int i = 0; i < kHistBins / NT; ++i) {
            sh.hist[tid + i * NT] = hv[i];
            hrow[tid + i * NT] = 0u;
        }
    }
    for (int w = tid; w < NW; w += NT) {
        sel[w] = 0u;
        tie[w] = 0u;
    }
    if (tid == 0) sh.cand_n = 0;
    __syncthreads();
    if (k == 0) return;
    if (k == N) {
        for (int i = tid; i < N; i += NT) orow[i] = i;
        return;
    }
    auto key_at = [&](int i) -> uint32_t { return float_key(__ldcg(srow + i)); };
    uint32_t d0, above;
    select_digit<NT>(sh, 2048u, k, d0, above);
    d0 &= (kHistBins - 1);
    int krem = k - (int)above;
    if (sh.hist[d0] > (uint32_t)kCandCap) {
        // too many candidates for the buffer: resolve the remaining digits over the row
        uint32_t prefix = d0 << 21, pmask = 0x7ffu << 21;
#pragma unroll 1
        for (int pass = 1; pass < 3; ++pass) {
            const uint32_t nb = pass == 2 ? 1024u : 2048u;
            hist_pass_all<NT>(sh, key_at, N, prefix, pmask, kShift[pass], nb);
            uint32_t dg, ab;
            select_digit<NT>(sh, nb, krem, dg, ab);
            prefix |= dg << kShift[pass];
            pmask |= (nb - 1) << kShift[pass];
            krem -= (int)ab;
        }
        emit_selected<NT>(sh, key_at, N, k, prefix, krem, orow);
        return;
    }
    // ---- one pass: bitmap of entries above d0, candidates of digit d0
    const uint32_t lt = lanemask_lt();
    if (((reinterpret_cast<uintptr_t>(srow) | (uintptr_t)N) & 3u) == 0 &&
        (reinterpret_cast<uintptr_t>(srow) & 15u) == 0) {
        // 16-byte loads: lane l holds entries 4l..4l+3 of a 128-entry chunk (4 bitmap words)
        const float4* srow4 = reinterpret_cast<const float4*>(srow);
        const int NCH = (N + 127) / 128;
        constexpr int U = 4;  // chunks a warp loads before using any
        for (int c0 = warp; c0 < NCH; c0 += U * NWP) {
            float4 f[U];
#pragma unroll
            for (int u = 0; u < U; ++u) {
                const int c = c0 + u * NWP;
                const int e = c * 128 + lane * 4;
                f[u] = (c < NCH && e < N) ? __ldcg(srow4 + e / 4) : make_float4(0.f, 0.f, 0.f, 0.f);
            }
#pragma unroll
            for (int u = 0; u < U; ++u) {
                const int c = c0 + u * NWP;
                if (c >= NCH) break;
                const bool valid = c * 128 + lane * 4 < N;
                const uint32_t kk[4] = {float_key(f[u].x), float_key(f[u].y), float_key(f[u].z), float_key(f[u].w)};
                uint32_t m[4], word = 0, n_in = 0, before = 0;
#pragma unroll
                for (int j = 0; j < 4; ++j) {
                    const uint32_t dg = kk[j] >> 21;
                    const uint32_t sure = __ballot_sync(0xffffffffu, valid && dg > d0);
                    m[j] = __ballot_sync(0xffffffffu, valid && dg == d0);
                    // bitmap word w holds lanes 8w..8w+7: entry 4(l-8w)+j is bit l of ballot j
                    word |= spread8((sure >> (8 * (lane & 3))) & 0xffu) << j;
                    n_in += __popc(m[j]);
                    before += __popc(m[j] & lt);
                }
                if (lane < 4 && 4 * c + lane < NW) sel[4 * c + lane] = word;
                if (n_in != 0u) {  // one reservation for the chunk's candidates
                    uint32_t at = 0;
                    if (lane == 0) at = atomicAdd(&sh.cand_n, n_in);
                    uint32_t slot = __shfl_sync(0xffffffffu, at, 0) + before;
#pragma unroll
                    for (int j = 0; j < 4; ++j) {
                        if ((m[j] >> lane) & 1u) {
                            if (slot < (uint32_t)kCandCap) {
                                cand_key[slot] = kk[j];
                                cand_idx[slot] = (uint32_t)(c * 128 + lane * 4 + j);
                            }
                            ++slot;
                        }
                    }
                }
            }
        }
    } else {
        constexpr int U = 8;  // 32-entry groups a warp loads before using any
        for (int g0 = warp; g0 < NW; g0 += U * NWP) {
            uint32_t kk[U], m[U];
#pragma unroll
            for (int u = 0; u < U; ++u) {
                const int i = (g0 + u * NWP) * 32 + lane;
                kk[u] = (g0 + u * NWP < NW && i < N) ? key_at(i) : 0u;
            }
            uint32_t n_in = 0;
#pragma unroll
            for (int u = 0; u < U; ++u) {
                const int gw = g0 + u * NWP;
                const int i = gw * 32 + lane;
                const bool valid = gw < NW && i < N;
                const uint32_t dg = kk[u] >> 21;
                const uint32_t sure = __ballot_sync(0xffffffffu, valid && dg > d0);
                if (lane == 0 && gw < NW) sel[gw] = sure;
                m[u] = __ballot_sync(0xffffffffu, valid && dg == d0);
                n_in += __popc(m[u]);
            }
            if (n_in != 0u) {  // one reservation for the batch's candidates
                uint32_t at = 0;
                if (lane == 0) at = atomicAdd(&sh.cand_n, n_in);
                at = __shfl_sync(0xffffffffu, at, 0);
#pragma unroll
                for (int u = 0; u < U; ++u) {
                    const uint32_t slot = at + __popc(m[u] & lt);
                    if (((m[u] >> lane) & 1u) && slot < (uint32_t)kCandCap) {
                        cand_key[slot] = kk[u];
                        cand_idx[slot] = (uint32_t)((g0 + u * NWP) * 32 + lane);
                    }
                    at += __popc(m[u]);
                }
            }
        }
    }
    __syncthreads();
    const uint32_t n_cand = min(sh.cand_n, (uint32_t)kCandCap);
    // ---- remaining 21 bits among the candidates
    uint32_t prefix = d0 << 21, pmask = 0x7ffu << 21;
#pragma unroll 1
    for (int pass = 1; pass < 3; ++pass) {
        const uint32_t nb = pass == 2 ? 1024u : 2048u;
        const int shift = kShift[pass];
        for (int b = tid; b < kHistBins; b += NT) sh.hist[b] = 0;
        __syncthreads();
        for (uint32_t c = tid; c < n_cand; c += NT) {
            const uint32_t ck = cand_key[c];
            if ((ck & pmask) == prefix) atomicAdd(&sh.hist[(ck >> shift) & (nb - 1)], 1u);
        }
        __syncthreads();
        uint32_t dg, ab;
        select_digit<NT>(sh, nb, krem, dg, ab);
        prefix |= dg << shift;
        pmask |= (nb - 1) << shift;
        krem -= (int)ab;
    }
    const uint32_t thr = prefix;
    for (uint32_t c = tid; c < n_cand; c += NT) {
        const uint32_t ck = cand_key[c], ci = cand_idx[c];
        if (ck > thr) atomicOr(&sel[ci >> 5], 1u << (ci & 31));
        else if (ck == thr) atomicOr(&tie[ci >> 5], 1u << (ci & 31));
    }
    __syncthreads();
    // ---- keep the krem lowest-index ties; thread t owns words [t*W, t*W + W)
    const int W = (NW + NT - 1) / NT;
    const int w0 = tid * W, w1 = min(NW, w0 + W);
    {
        uint32_t cnt = 0;
        for (int w = w0; w < w1; ++w) cnt += __popc(tie[w]);
        uint32_t total;
        uint32_t before = block_exclusive_scan<NT>(cnt, sh.wsum, total);
        for (int w = w0; w < w1; ++w) {
            uint32_t bits = tie[w];
            while (bits != 0u && (int)before < krem) {
                const uint32_t low = bits & (0u - bits);
                sel[w] |= low;
                bits ^= low;
                ++before;
            }
        }
    }
    __syncthreads();
    // ---- ascending emit from the selection bitmap
    {
        uint32_t cnt = 0;
        for (int w = w0; w < w1; ++w) cnt += __popc(sel[w]);
        uint32_t total;
        uint32_t at = block_exclusive_scan<NT>(cnt, sh.wsum, total);
        for (int w = w0; w < w1; ++w) {
            uint32_t bits = sel[w];
            while (bits != 0u) {
                const int bpos = __ffs(bits) - 1;
                bits &= bits - 1u;
                if (at < (uint32_t)k) orow[at] = w * 32 + bpos;
                ++at;
            }
        }
    }
}

}  // namespace
}  // namespace sd

using namespace sd;

extern "C" size_t sd_topk_workspace_bytes(int rows, int N, int k) {
    (void)rows;
    (void)N;
    (void)k;
    return 0;
}

extern "C" sd_status sd_topk(const float* scores, int rows, int N, int k, int32_t* idx,
                             uint32_t* key_hist, void* workspace, size_t workspace_bytes,
                             void* stream) {
    (void)workspace;
    (void)workspace_bytes;
    clear_error();
    SD_REQUIRE(rows >= 0 && N >= 0, "sd_topk: negative size");
    SD_REQUIRE(k >= 0 && k <= N, "sd_topk: k (%d) must be in [0, N=%d]", k, N);
    if (rows == 0) return SD_OK;
    if (key_hist == nullptr && k == 0) return SD_OK;
    SD_REQUIRE(scores && (k == 0 || idx), "sd_topk: null pointer");
    cudaStream_t st = as_stream(stream);
    if (N <= kSmallN) {  // the row in registers, one CTA per row
        if (N <= kSmallWarps * 32 * 8)
            SD_CUDA_CHECK(launch_pdl(topk_small_kernel<8>, rows, kSmallThreads, 0, st, scores, N, k, idx, key_hist),
                          "sd_topk: launch");
        else
            SD_CUDA_CHECK(launch_pdl(topk_small_kernel<16>, rows, kSmallThreads, 0, st, scores, N, k, idx, key_hist),
                          "sd_topk: launch");
        return launch_status("sd_topk");
    }
    // few long rows: several CTAs per row in a thread-block cluster
    if (N >= kClusterMinN) {
        sd_status cs = SD_OK;
        if (topk_by_clusters(scores, rows, N, k, idx, key_hist, st, &cs)) return cs;
    }
    const size_t limit = (size_t)max_smem_optin();
    const size_t static_bytes = sizeof(TopkShared) + 1024;
    const size_t key_bytes = (size_t)N * sizeof(uint32_t);
    const size_t aux_bytes = (size_t)2 * kCandCap * sizeof(uint32_t) + (size_t)2 * ((N + 31) / 32) * sizeof(uint32_t);
    if (key_hist != nullptr && aux_bytes + static_bytes > limit) {
        // the bitmaps do not fit: plain select, and clear the histogram as promised
        SD_CUDA_CHECK(cudaMemsetAsync(key_hist, 0, (size_t)rows * kHistBins * sizeof(uint32_t), st),
                      "sd_topk: clearing key_hist");
        key_hist = nullptr;
        if (k == 0) return SD_OK;
    }
    if (key_hist != nullptr) {
        // more rows than SMs: 512-thread CTAs, two per SM, so the rows run in one wave
        const size_t dyn = aux_bytes;
        if (rows > num_sms()) {
            SD_CUDA_CHECK(cudaFuncSetAttribute(topk_hist_kernel<512>, cudaFuncAttributeMaxDynamicSharedMemorySize,
                                               (int)dyn),
                          "sd_topk: cudaFuncSetAttribute");
            SD_CUDA_CHECK(launch_pdl(topk_hist_kernel<512>, rows, 512, dyn, st, scores, N, k, idx, key_hist),
                          "sd_topk: launch");
        } else {
            SD_CUDA_CHECK(cudaFuncSetAttribute(topk_hist_kernel<kTkThreads>,
                                               cudaFuncAttributeMaxDynamicSharedMemorySize, (int)dyn),
                          "sd_topk: cudaFuncSetAttribute");
            SD_CUDA_CHECK(launch_pdl(topk_hist_kernel<kTkThreads>, rows, kTkThreads, dyn, st, scores, N, k, idx,
                                     key_hist),
                          "sd_topk: launch");
        }
    } else {
        const int cache = key_bytes + static_bytes <= limit ? 1 : 0;
        const size_t dyn = cache ? key_bytes : 0;
        SD_CUDA_CHECK(cudaFuncSetAttribute(topk_kernel, cudaFuncAttributeMaxDynamicSharedMemorySize, (int)dyn),
                      "sd_topk: cudaFuncSetAttribute");
        SD_CUDA_CHECK(launch_pdl(topk_kernel, rows, kTkThreads, dyn, st, scores, N, k, idx, cache, (int32_t*)nullptr),
                      "sd_topk: launch");
    }
    return launch_status("sd_topk");
}
