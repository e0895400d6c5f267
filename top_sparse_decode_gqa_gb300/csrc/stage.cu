// stage.cu -- the selected rows that live in host memory, copied into an HBM stage.
//
// "O Fim do Gargalo de Memoria: Como o Adaptive DHiSparse Revolutiona LLMs de Contexto
// Longo" (news page), "A Inovacao": the history stays in host memory and only the selected
// rows cross the link; "Metodologia e Eficiencia de Carga": the query rows of a group share
// the fetch of a missing row.  SparDA (gist.science summary), sec. 2 item 3: a kernel moves
// the needed rows from host memory through unified addressing ahead of the attention.
//
// Why a separate copy: when every (b, kvh) group fetches its own host rows inside the
// attention, each CTA waits on the link for its own share and the SMs the link serves last
// set the time.  Here every warp of a persistent grid takes the next chunk of rows from one
// counter, so the copy ends when the link has moved the bytes, whichever SMs asked; the
// attention then reads those rows from HBM.  A copy has no summation order, so dynamic
// scheduling changes no result.
#include "sd_common.cuh"
#include "sd_host.h"

namespace sd {
namespace {

constexpr int kStThreads = 256;
constexpr int kStPieces = 8;  // 16-byte pieces a lane moves per chunk (all loads before any store)
constexpr int kStTailShare = 4;  // the last 1/kStTailShare of the list rows go out as short tickets
constexpr int kStGrid = 64;      // CTAs of the copy (at most one per SM)

struct StageParams {
    const uint8_t* kh;  // mapped host cache [B, kv_heads, T, d]
    const uint8_t* vh;
    uint8_t* ks;        // stage [groups, n_rows, d]
    uint8_t* vs;
    const int32_t* slot_map;
    const int32_t* idx;
    int T, pool_rows, n_idx, block, n_rows;
    int groups_per_seq, kv_heads, heads_per_kv;
    int row_bytes, rows_per_chunk;  // rows_per_chunk: rows one copy batch moves
    int total_rows;
    int n_long, long_rows;  // tickets of 32 list rows first (n_long of them, long_rows rows), then of
                            // rows_per_chunk rows
    uint32_t* counter;  // [0] next chunk, [1] CTAs done; zero between calls
    int32_t* err;
    int slot_per_head;  // 1: slot_map is [B, kv_heads, T]
};

// Position of the n-th (from 0) set bit of `mask`, for n < popc(mask): the largest x with
// popc(mask & (2^x - 1)) <= n, by binary search over x.
SD_DEVINL int nth_set_bit(uint32_t mask, int n) {
    int x = 0;
#pragma unroll
    for (int step = 16; step > 0; step >>= 1)
        if (__popc(mask & ((1u << (x + step)) - 1u)) <= n) x += step;
    return x;
}

// A warp takes the next ticket of list rows from the counter (one row per lane), resolves
// each to its host row or to nothing (pooled or empty), and copies only the misses,
// rows_per_chunk rows (kStPieces 16-byte pieces per lane, all loads before any store) at a
// time; a piece's miss is found in the ballot of misses and its rows are shuffled from the
// lane that resolved it.  Tickets hold 32 rows (one resolving lane each: cheap when the pool
// serves most rows) except over the last 1/kStTailShare of the list, where they hold one copy
// batch: when most rows are misses a 32-row ticket takes four batches in a row, and the last
// such tickets would keep a few warps copying after the rest have finished.
// No shared memory, and registers capped at 80 (the bound's 3 CTAs; the grid has at most one per SM):
// the kernel runs beside the indexer, whose CTAs need most of an SM's shared memory, and
// beside the attention.
__global__ void __launch_bounds__(kStThreads, 3) stage_host_rows_kernel(const StageParams p) {
    pdl_wait();  // idx (and the slot map) may come from the preceding kernel
    pdl_launch_dependents();
    const int lane = threadIdx.x & 31;
    const int ppr = p.row_bytes / 16;  // pieces per K (or V) row
    const int C = p.rows_per_chunk;    // C * 2 * ppr == 32 * kStPieces
    const int nchunks = p.n_long + (p.total_rows - p.long_rows + C - 1) / C;
    for (;;) {
        uint32_t c = 0;
        if (lane == 0) c = atomicAdd(&p.counter[0], 1u);
        c = __shfl_sync(0xffffffffu, c, 0);
        if (c >= (uint32_t)nchunks) break;
        // the ticket's rows [base, base + cnt); lane r resolves list row f = base + r to its
        // host row, or -1 (nothing to copy)
        const bool lng = c < (uint32_t)p.n_long;
        const int base = lng ? (int)c * 32 : p.long_rows + ((int)c - p.n_long) * C;
        const int cnt = lng ? 32 : C;
        int host_row = -1;  // < 2^31 (checked on the host)
        const int f = base + lane;
        if (lane < cnt && f < p.total_rows) {
            const int g = f / p.n_rows, j = f % p.n_rows;
            const int b = g / p.groups_per_seq;
            const int kvsrc = b * p.kv_heads + (g % p.groups_per_seq) / p.heads_per_kv;
            long pos = j;
            bool ok = true;
            if (p.idx != nullptr) {
                const long sel = p.idx[(size_t)g * p.n_idx + j / p.block];
                pos = sel * p.block + j % p.block;
                if (sel == -1) {
                    ok = false;  // empty slot
                } else if (sel < 0 || pos >= p.T) {
                    report(p.err, SD_DEVERR_INDEX);
                    ok = false;
                }
            }
            if (ok) {
                const int slot = p.slot_map[(size_t)(p.slot_per_head ? kvsrc : b) * p.T + pos];
                if (slot == -1)
                    host_row = kvsrc * p.T + (int)pos;
                else if (slot < -1 || slot >= p.pool_rows)
                    report(p.err, SD_DEVERR_SLOT);
            }
        }
        const uint32_t miss = __ballot_sync(0xffffffffu, host_row >= 0);
        if (miss == 0u) continue;
        const int n_miss = __popc(miss);
        for (int m0 = 0; m0 < n_miss; m0 += C) {
            // piece q = lane + 32 i of the batch: miss m0 + q / (2 ppr) (resolved by the lane
            // holding the miss's bit), K for the first ppr pieces of a row and V for the rest,
            // 16 bytes at (q mod ppr) * 16
            uint4 v[kStPieces];
#pragma unroll
            for (int i = 0; i < kStPieces; ++i) {
                const int q = lane + 32 * i, m = m0 + q / (2 * ppr), w = q % (2 * ppr);
                const int hr = __shfl_sync(0xffffffffu, host_row, nth_set_bit(miss, m < n_miss ? m : 0));
                if (m < n_miss) {
                    const uint8_t* s_ = (w < ppr ? p.kh : p.vh) + (size_t)hr * p.row_bytes + (w % ppr) * 16;
                    v[i] = __ldcs(reinterpret_cast<const uint4*>(s_));
                }
            }
#pragma unroll
            for (int i = 0; i < kStPieces; ++i) {
                const int q = lane + 32 * i, m = m0 + q / (2 * ppr), w = q % (2 * ppr);
                const int fr = __shfl_sync(0xffffffffu, f, nth_set_bit(miss, m < n_miss ? m : 0));
                if (m < n_miss) {
                    uint8_t* dst = (w < ppr ? p.ks : p.vs) + (size_t)fr * p.row_bytes + (w % ppr) * 16;
                    *reinterpret_cast<uint4*>(dst) = v[i];
                }
            }
        }
    }
    // the last CTA to finish leaves the counter at zero for the next call
    __syncthreads();
    if (threadIdx.x == 0) {
        __threadfence();
        if (atomicAdd(&p.counter[1], 1u) == gridDim.x - 1) {
            p.counter[0] = 0u;
            p.counter[1] = 0u;
        }
    }
}

}  // namespace
}  // namespace sd

using namespace sd;

extern "C" sd_status sd_stage_host_rows(const sd_attend_args* a, uint32_t* counter, void* stream) {
    clear_error();
    sd_status vs = validate_attend_args(a, "sd_stage_host_rows");
    if (vs != SD_OK) return vs;
    SD_REQUIRE(a->slot_map != nullptr, "sd_stage_host_rows: needs slot_map");
    if (a->tier != nullptr) {
        set_error("sd_stage_host_rows: tiered rows read their host rows in sd_gather_attend");
        return SD_ERR_UNSUPPORTED;
    }
    SD_REQUIRE(a->k_host && a->v_host, "sd_stage_host_rows: needs k_host and v_host");
    SD_REQUIRE(a->k_stage && a->v_stage, "sd_stage_host_rows: needs k_stage and v_stage");
    SD_REQUIRE(aligned16(a->k_stage) && aligned16(a->v_stage),
               "sd_stage_host_rows: k_stage/v_stage must be 16-byte aligned");
    SD_REQUIRE(aligned16(a->k_host) && aligned16(a->v_host), "sd_stage_host_rows: host K/V must be 16-byte aligned");
    SD_REQUIRE(a->pool_rows >= 0, "sd_stage_host_rows: pool_rows must be >= 0");
    SD_REQUIRE(counter != nullptr && (reinterpret_cast<uintptr_t>(counter) & 3u) == 0,
               "sd_stage_host_rows: needs a 4-byte aligned device counter");
    StageParams p{};
    p.kh = mapped_host_ptr(a->k_host);
    p.vh = mapped_host_ptr(a->v_host);
    SD_REQUIRE(p.kh && p.vh, "sd_stage_host_rows: k_host/v_host must be pinned, mapped host memory");
    p.ks = static_cast<uint8_t*>(const_cast<void*>(a->k_stage));
    p.vs = static_cast<uint8_t*>(const_cast<void*>(a->v_stage));
    p.slot_map = a->slot_map;
    p.idx = a->idx;
    p.T = a->T;
    p.pool_rows = a->pool_rows;
    p.n_idx = a->n_idx;
    p.block = a->block;
    p.n_rows = a->n_idx * a->block;
    p.groups_per_seq = a->per_head ? a->Hq : a->Hkv;
    p.kv_heads = a->Hkv;
    p.heads_per_kv = a->per_head ? a->Hq / a->Hkv : 1;
    p.row_bytes = a->d * dtype_bytes(a->dtype);
    p.rows_per_chunk = 32 * kStPieces / (2 * (p.row_bytes / 16));
    const long total = (long)a->B * p.groups_per_seq * p.n_rows;
    SD_REQUIRE(total + 32 < (1L << 31) && (long)a->B * a->Hkv * a->T < (1L << 31),
               "sd_stage_host_rows: selected rows and host cache rows must be < 2^31");
    p.total_rows = (int)total;
    p.n_long = (int)(total - total / kStTailShare) / 32;
    p.long_rows = p.n_long * 32;
    p.counter = counter;
    p.err = a->err_word;
    p.slot_per_head = a->slot_per_head;
    if (p.total_rows == 0) return SD_OK;
    // 64 CTAs of 8 warps (2 MB of host reads in flight) keep the host link busy (~200 GB/s:
    // the same rate as one CTA per SM) and leave most SMs to the kernels running beside the
    // copy (the next layer's indexer, the current layer's attention); a grid of one CTA per
    // SM slowed those enough to cost ~10 % of a lookahead step, while fewer than ~32 CTAs
    // no longer fill the link and calls whose rows are mostly pooled lose to the longer
    // resolve per warp
    const int grid = num_sms() < kStGrid ? num_sms() : kStGrid;
    SD_CUDA_CHECK(launch_pdl(stage_host_rows_kernel, dim3((unsigned)grid), dim3(kStThreads), 0, as_stream(stream), p),
                  "sd_stage_host_rows: launch");
    return launch_status("sd_stage_host_rows");
}
