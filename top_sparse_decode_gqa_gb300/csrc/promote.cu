// promote.cu -- the HBM pool kept as a cache of host rows.
//
// "O Fim do Gargalo de Memoria: Como o Adaptive DHiSparse Revolutiona LLMs de Contexto
// Longo" (news page), "Metodologia e Eficiencia de Carga": the GPU keeps extra history
// while memory allows and fetches the rest; SparDA (gist.science summary), sec. 2 item 3:
// the needed rows are fetched ahead.  Reading taken, per sequence: the step's selected
// positions (union over the KV heads) that are not in the pool are promoted, in ascending
// position order, into the first slots of a FIFO ring (starting at the sequence's hand)
// that do not hold a position selected in the same step; a slot's old position leaves the
// pool.  A later step that selects the same rows reads them from HBM.  With a slot map per
// (sequence, KV head) every (b, KV head) is such a unit, holding only its own head's rows.
//
// Three launches:
//   mark   every selected position sets its bit in a per-sequence bitmap;
//   plan   one CTA per sequence: the misses (marked, slot -1) in ascending order by a block
//          scan over the bitmap, the victims (unpinned slots in ring order) by block scans
//          over the ring, the slot map, reverse map and hand updated, the bitmap cleared;
//   copy   a persistent grid copies each promoted position's K and V rows of every KV head
//          from the host cache (device mapping) into its pool slot; warps take tasks from a
//          counter that the last CTA resets.
//
// Staged mode (sd_promote_staged_rows, units of one KV head): the step's misses were already
// copied into the HBM stage by sd_stage_host_rows and read from there by the attention, so
// the promotion runs after the attention and copies each promoted row from the stage (the
// list row that selected it, recorded by the mark kernel) instead of crossing the host link
// a second time.  The pool state after the call is the same as in the host mode.
#include <algorithm>

#include "sd_common.cuh"
#include "sd_host.h"

namespace sd {
namespace {

constexpr int kPlanThreads = 1024;
constexpr int kCopyThreads = 256;

struct PromoteParams {
    const int32_t* idx;      // [B, groups, n_idx]
    int32_t* slot_map;       // [B, T]
    int32_t* pool_pos;       // [B, P]
    int32_t* hand;           // [B]
    const uint8_t* kh;       // mapped host cache [B, Hkv, T, d] (host mode)
    const uint8_t* vh;
    const uint8_t* ks;       // stage [units * groups * n_idx * block, d] (staged mode)
    const uint8_t* vs;
    int32_t* row_of;         // [B, T] staged mode: a list row that selected the position
    uint8_t* kp;             // pool [B, Hkv, P, d]
    uint8_t* vp;
    uint32_t* mark;          // [B, W32], zero between calls
    int2* tasks;             // [B, max_tasks] (position, slot)
    int32_t* ntask;          // [B]
    uint32_t* counter;       // [2], zero between calls
    int B, groups, n_idx, block, T, P, Hkv, row_bytes, W32, max_tasks;
    int32_t* err;
};

// Every selected position of every group sets its bit.
__global__ void __launch_bounds__(256) promote_mark_kernel(const PromoteParams p) {
    pdl_wait();  // idx comes from the preceding top-k
    pdl_launch_dependents();
    const long n_rows = (long)p.n_idx * p.block;
    const long total = (long)p.B * p.groups * n_rows;
    for (long e = blockIdx.x * (long)blockDim.x + threadIdx.x; e < total; e += (long)gridDim.x * blockDim.x) {
        const long gj = e / n_rows, j = e % n_rows;
        const int b = (int)(gj / p.groups);
        const long sel = p.idx[gj * p.n_idx + j / p.block];
        if (sel == -1) continue;
        const long pos = sel * p.block + j % p.block;
        if (sel < 0 || pos >= p.T) {
            report(p.err, SD_DEVERR_INDEX);
            continue;
        }
        atomicOr(&p.mark[(size_t)b * p.W32 + (pos >> 5)], 1u << (pos & 31));
        // several groups of a unit may select the same position: any one of their list rows
        // holds the row (one KV head per unit), so whichever store lands last is right
        if (p.row_of != nullptr) p.row_of[(size_t)b * p.T + pos] = (int)e;
    }
}

// Block-wide exclusive scan of one value per thread (kPlanThreads); also the total.
SD_DEVINL int plan_scan(int v, int* wsum, int& total) {
    const int lane = threadIdx.x & 31, warp = threadIdx.x >> 5;
    int x = v;
#pragma unroll
    for (int o = 1; o < 32; o <<= 1) {
        const int n = __shfl_up_sync(0xffffffffu, x, o);
        if (lane >= o) x += n;
    }
    if (lane == 31) wsum[warp] = x;
    __syncthreads();
    if (warp == 0) {
        int w = wsum[lane];
#pragma unroll
        for (int o = 1; o < 32; o <<= 1) {
            const int n = __shfl_up_sync(0xffffffffu, w, o);
            if (lane >= o) w += n;
        }
        wsum[lane] = w;
    }
    __syncthreads();
    total = wsum[31];
    const int excl = x - v + (warp > 0 ? wsum[warp - 1] : 0);
    __syncthreads();
    return excl;
}

// One CTA per sequence.
__global__ void __launch_bounds__(kPlanThreads) promote_plan_kernel(const PromoteParams p) {
    __shared__ int wsum[32];
    __shared__ int s_last;
    pdl_wait();
    pdl_launch_dependents();
    const int b = blockIdx.x, tid = threadIdx.x;
    const uint32_t* mk = p.mark + (size_t)b * p.W32;
    int32_t* sm = p.slot_map + (size_t)b * p.T;
    int32_t* pp = p.pool_pos + (size_t)b * p.P;
    int2* tk = p.tasks + (size_t)b * p.max_tasks;
    // ---- misses in ascending order: thread t owns words [t*Wp, t*Wp + Wp)
    const int Wp = (p.W32 + kPlanThreads - 1) / kPlanThreads;
    const int w0 = tid * Wp, w1 = min(p.W32, w0 + Wp);
    int cnt = 0;
    for (int w = w0; w < w1; ++w) {
        uint32_t bits = mk[w];
        while (bits != 0u) {
            const int pos = w * 32 + __ffs(bits) - 1;
            bits &= bits - 1u;
            if (sm[pos] == -1) ++cnt;
        }
    }
    int n_miss;
    int at = plan_scan(cnt, wsum, n_miss);
    for (int w = w0; w < w1; ++w) {
        uint32_t bits = mk[w];
        while (bits != 0u) {
            const int pos = w * 32 + __ffs(bits) - 1;
            bits &= bits - 1u;
            if (sm[pos] == -1) {
                if (at < p.max_tasks) tk[at].x = pos;
                ++at;
            }
        }
    }
    n_miss = min(n_miss, p.max_tasks);
    // ---- victims: the first n_miss unpinned slots in ring order from the hand
    const int h0 = (int)((((long)p.hand[b]) % p.P + p.P) % p.P);  // a hand outside [0, P) wraps
    if (tid == 0) s_last = -1;
    __syncthreads();
    int found = 0;
    for (int i0 = 0; i0 < p.P && found < n_miss; i0 += kPlanThreads) {
        const int i = i0 + tid;
        int s = -1, unpinned = 0;
        if (i < p.P) {
            s = (int)(((long)h0 + i) % p.P);
            const int t = pp[s];
            unpinned = (t < 0 || t >= p.T || ((mk[t >> 5] >> (t & 31)) & 1u) == 0u) ? 1 : 0;
        }
        int n_here;
        const int rank = found + plan_scan(unpinned, wsum, n_here);
        if (unpinned && rank < n_miss) {
            tk[rank].y = s;
            if (rank == n_miss - 1 || rank == found + n_here - 1) atomicMax(&s_last, i);
        }
        found += n_here;
    }
    const int take = min(found, n_miss);
    __syncthreads();
    // ---- apply: old positions leave, misses enter (all positions and slots distinct)
    for (int m = tid; m < take; m += kPlanThreads) {
        const int pos = tk[m].x, s = tk[m].y;
        const int old = pp[s];
        if (old >= 0 && old < p.T) sm[old] = -1;
        sm[pos] = s;
        pp[s] = pos;
    }
    if (tid == 0) {
        p.ntask[b] = take;
        if (take > 0) p.hand[b] = (int)(((long)h0 + s_last + 1) % p.P);
    }
    __syncthreads();
    // ---- the bitmap starts the next call at zero
    for (int w = tid; w < p.W32; w += kPlanThreads) p.mark[(size_t)b * p.W32 + w] = 0u;
}

// Warps take chunks of kTaskChunk tasks (a task: one promoted position of one unit) from the
// counter -- chunks past a unit's task count are skipped at once -- and copy each task's K
// and V rows of every KV head as 16-byte pieces, loads before stores.
constexpr int kTaskChunk = 32;

__global__ void __launch_bounds__(kCopyThreads) promote_copy_kernel(const PromoteParams p) {
    pdl_wait();
    pdl_launch_dependents();
    const int lane = threadIdx.x & 31;
    const int pieces = p.row_bytes / 16;       // per row
    const int per_task = 2 * p.Hkv * pieces;    // K and V of every head
    const int chunks_per_unit = (p.max_tasks + kTaskChunk - 1) / kTaskChunk;
    const long total = (long)p.B * chunks_per_unit;
    for (;;) {
        uint32_t c = 0;
        if (lane == 0) c = atomicAdd(&p.counter[0], 1u);
        c = __shfl_sync(0xffffffffu, c, 0);
        if ((long)c >= total) break;
        const int b = (int)(c / chunks_per_unit), m0 = (int)(c % chunks_per_unit) * kTaskChunk;
        const int m1 = min(p.ntask[b], m0 + kTaskChunk);
        for (int m = m0; m < m1; ++m) {
        const int2 t = p.tasks[(size_t)b * p.max_tasks + m];
        if (t.x < 0 || t.x >= p.T || t.y < 0 || t.y >= p.P) {  // never for a consistent plan
            if (lane == 0) report(p.err, SD_DEVERR_SLOT);
            continue;
        }
        // piece q: K (q < Hkv*pieces) or V, head h, 16 bytes at (q mod pieces) * 16
        for (int q0 = 0; q0 < per_task; q0 += 32 * 4) {
            uint4 v[4];
#pragma unroll
            for (int u = 0; u < 4; ++u) {
                const int q = q0 + u * 32 + lane;
                if (q >= per_task) continue;
                const int which = q / (p.Hkv * pieces), rem = q % (p.Hkv * pieces);
                const int h = rem / pieces, off = (rem % pieces) * 16;
                if (p.ks != nullptr) {  // staged mode: one KV head per unit
                    const size_t src = (size_t)p.row_of[(size_t)b * p.T + t.x] * p.row_bytes + off;
                    v[u] = __ldcs(reinterpret_cast<const uint4*>((which ? p.vs : p.ks) + src));
                } else {
                    const size_t src = (((size_t)b * p.Hkv + h) * p.T + t.x) * p.row_bytes + off;
                    v[u] = __ldcs(reinterpret_cast<const uint4*>((which ? p.vh : p.kh) + src));
                }
            }
#pragma unroll
            for (int u = 0; u < 4; ++u) {
                const int q = q0 + u * 32 + lane;
                if (q >= per_task) continue;
                const int which = q / (p.Hkv * pieces), rem = q % (p.Hkv * pieces);
                const int h = rem / pieces, off = (rem % pieces) * 16;
                const size_t dst = (((size_t)b * p.Hkv + h) * p.P + t.y) * p.row_bytes + off;
                *reinterpret_cast<uint4*>((which ? p.vp : p.kp) + dst) = v[u];
            }
        }
        }
    }
    __syncthreads();
    if (threadIdx.x == 0) {
        __threadfence();
        if (atomicAdd(&p.counter[1], 1u) == gridDim.x - 1) {
            p.counter[0] = 0u;
            p.counter[1] = 0u;
        }
    }
}

struct PromoteLayout {
    size_t mark, tasks, ntask, counter, row_of, bytes;
    int W32, max_tasks;
};

size_t al256(size_t x) { return (x + 255) & ~size_t(255); }

// The promotion's units.  With one slot map per sequence the unit is the sequence (its KV
// heads share a slot); with one per (sequence, KV head) every (b, KV head) is a unit of its
// own with a single KV head -- the same memory read as [B*Hkv, 1, ...] -- whose selection
// is its own row of idx (or the G query heads' rows with per-head selections).
struct PromoteUnits {
    int units, heads, groups;
};

PromoteUnits promote_units(const sd_attend_args* a) {
    const int G = a->Hq / a->Hkv;
    if (a->slot_per_head) return {a->B * a->Hkv, 1, a->per_head ? G : 1};
    return {a->B, a->Hkv, a->per_head ? a->Hq : a->Hkv};
}

PromoteLayout promote_layout(const sd_attend_args* a, bool staged) {
    PromoteLayout l{};
    const PromoteUnits u = promote_units(a);
    l.W32 = (a->T + 31) / 32;
    const long sel = (long)u.groups * a->n_idx * a->block;
    l.max_tasks = (int)std::min<long>((long)a->pool_rows, std::max<long>(1, sel));
    l.mark = 0;
    l.tasks = al256((size_t)u.units * l.W32 * 4);
    l.ntask = l.tasks + al256((size_t)u.units * l.max_tasks * sizeof(int2));
    l.counter = l.ntask + al256((size_t)u.units * 4);
    l.row_of = l.counter + 256;
    l.bytes = l.row_of + (staged ? al256((size_t)u.units * a->T * 4) : 0);
    return l;
}

}  // namespace
}  // namespace sd

using namespace sd;

namespace {

sd_status promote_impl(const sd_attend_args* a, int32_t* pool_pos, int32_t* hand, void* workspace,
                       size_t workspace_bytes, void* stream, bool staged, const char* who) {
    clear_error();
    sd_status vs = validate_attend_args(a, who);
    if (vs != SD_OK) return vs;
    SD_REQUIRE(a->idx != nullptr && a->slot_map != nullptr, "%s: needs idx and slot_map", who);
    SD_REQUIRE(a->pool_rows >= 1, "%s: needs a pool (pool_rows >= 1)", who);
    SD_REQUIRE(a->k_cache && a->v_cache && pool_pos && hand, "%s: needs the pool (k_cache, v_cache), pool_pos and hand",
               who);
    SD_REQUIRE(aligned16(a->k_cache) && aligned16(a->v_cache), "%s: pool pointers must be 16-byte aligned", who);
    if (staged) {
        SD_REQUIRE(a->slot_per_head == 1, "%s: needs a slot map per (sequence, KV head)", who);
        SD_REQUIRE(a->k_stage && a->v_stage && aligned16(a->k_stage) && aligned16(a->v_stage),
                   "%s: needs k_stage and v_stage (16-byte aligned)", who);
    } else {
        SD_REQUIRE(a->k_host && a->v_host, "%s: needs k_host and v_host", who);
        SD_REQUIRE(aligned16(a->k_host) && aligned16(a->v_host), "%s: host K/V must be 16-byte aligned", who);
    }
    SD_REQUIRE(a->B <= 65535, "%s: B must be <= 65535", who);
    if (a->B == 0 || a->n_idx == 0) return SD_OK;
    const PromoteLayout l = promote_layout(a, staged);
    SD_REQUIRE(workspace != nullptr && workspace_bytes >= l.bytes && aligned16(workspace),
               "%s: a 16-byte aligned workspace of %zu bytes is needed (got %zu)", who, l.bytes, workspace_bytes);
    PromoteParams p{};
    p.idx = a->idx;
    p.slot_map = const_cast<int32_t*>(a->slot_map);
    p.pool_pos = pool_pos;
    p.hand = hand;
    uint8_t* ws = static_cast<uint8_t*>(workspace);
    if (staged) {
        p.ks = static_cast<const uint8_t*>(a->k_stage);
        p.vs = static_cast<const uint8_t*>(a->v_stage);
        p.row_of = reinterpret_cast<int32_t*>(ws + l.row_of);
    } else {
        p.kh = mapped_host_ptr(a->k_host);
        p.vh = mapped_host_ptr(a->v_host);
        SD_REQUIRE(p.kh && p.vh, "%s: k_host/v_host must be pinned, mapped host memory", who);
    }
    p.kp = static_cast<uint8_t*>(const_cast<void*>(a->k_cache));
    p.vp = static_cast<uint8_t*>(const_cast<void*>(a->v_cache));
    p.mark = reinterpret_cast<uint32_t*>(ws + l.mark);
    p.tasks = reinterpret_cast<int2*>(ws + l.tasks);
    p.ntask = reinterpret_cast<int32_t*>(ws + l.ntask);
    p.counter = reinterpret_cast<uint32_t*>(ws + l.counter);
    const PromoteUnits u = promote_units(a);
    SD_REQUIRE(u.units <= 65535, "%s: %d units (sequences, or sequence x KV head) exceed 65535", who, u.units);
    p.B = u.units;
    p.groups = u.groups;
    p.n_idx = a->n_idx;
    p.block = a->block;
    p.T = a->T;
    p.P = a->pool_rows;
    p.Hkv = u.heads;
    p.row_bytes = a->d * dtype_bytes(a->dtype);
    p.W32 = l.W32;
    p.max_tasks = l.max_tasks;
    p.err = a->err_word;
    const long marks = (long)p.B * p.groups * a->n_idx * a->block;
    SD_REQUIRE(!staged || marks < (1L << 31), "%s: selected rows must be < 2^31", who);
    cudaStream_t st = as_stream(stream);
    const int mgrid = (int)std::min<long>((marks + 255) / 256, (long)num_sms() * 8);
    SD_CUDA_CHECK(launch_pdl(promote_mark_kernel, dim3((unsigned)mgrid), dim3(256), 0, st, p), who);
    SD_CUDA_CHECK(launch_pdl(promote_plan_kernel, dim3((unsigned)p.B), dim3(kPlanThreads), 0, st, p), who);
    SD_CUDA_CHECK(launch_pdl(promote_copy_kernel, dim3((unsigned)num_sms()), dim3(kCopyThreads), 0, st, p), who);
    return launch_status(who);
}

}  // namespace

extern "C" size_t sd_promote_rows_workspace_bytes(const sd_attend_args* a) {
    if (validate_attend_args(a, "sd_promote_rows") != SD_OK || a->pool_rows < 1) return 0;
    return promote_layout(a, false).bytes;
}

extern "C" sd_status sd_promote_rows(const sd_attend_args* a, int32_t* pool_pos, int32_t* hand, void* workspace,
                                     size_t workspace_bytes, void* stream) {
    return promote_impl(a, pool_pos, hand, workspace, workspace_bytes, stream, false, "sd_promote_rows");
}

extern "C" size_t sd_promote_staged_rows_workspace_bytes(const sd_attend_args* a) {
    if (validate_attend_args(a, "sd_promote_staged_rows") != SD_OK || a->pool_rows < 1) return 0;
    return promote_layout(a, true).bytes;
}

extern "C" sd_status sd_promote_staged_rows(const sd_attend_args* a, int32_t* pool_pos, int32_t* hand,
                                            void* workspace, size_t workspace_bytes, void* stream) {
    return promote_impl(a, pool_pos, hand, workspace, workspace_bytes, stream, true, "sd_promote_staged_rows");
}
