/*
 * sd.h -- C ABI of libsdgqa: top-k sparse decode attention with GQA on GB300 (sm_103a).
 *
 * The library is one hand-written CUDA kernel (or a short fixed sequence of them) per
 * call.  Every call is asynchronous on the CUDA stream passed as `stream` (a
 * cudaStream_t, given as void* so this header needs no CUDA include; NULL = the legacy
 * default stream).  Arguments are validated on the host before anything is launched; a
 * rejected call launches nothing and returns SD_ERR_INVALID_ARG or SD_ERR_UNSUPPORTED
 * (sd_last_error_message() tells why).  A failed launch returns SD_ERR_CUDA.
 *
 * Ownership: the caller owns every buffer.  The library allocates no device or host
 * memory on any call; calls that need scratch space take a caller-provided workspace
 * whose size is queried first.  Pointers are device pointers unless stated otherwise;
 * "pinned host" pointers must come from cudaHostAlloc / cudaHostRegister (page-locked
 * and mapped into the device address space).  All tensors are dense, row-major, with the
 * layouts given below; data pointers must be 16-byte aligned.
 *
 * Device-side faults: a selected row or pool slot outside its tensor is never read; the
 * kernel skips it and ORs a bit into *err_word (a caller-owned device int32, nullable:
 * NULL means such errors are not reported).  Every wait inside a kernel is bounded; a
 * wait that runs out sets SD_DEVERR_TIMEOUT and the kernel returns.  No kernel traps.
 *
 * Element types: SD_F32 = IEEE binary32, SD_BF16 = bfloat16 (upper half of a binary32),
 * SD_F16 = IEEE binary16 (only where a call says so: sd_block_pool's output and the
 * indexer's q and k together).  Arithmetic is fp32 (fp64 for the importance score)
 * whatever the storage type.
 *
 * Sources the operations follow (web pages, cited by title and section):
 *   [SparDA]    "SparDA: Atencao Esparsa Desacoplada para Inferencia Eficiente de LLMs de
 *               Longo Contexto" (gist.science technical summary), sec. 2.
 *   [Illusion]  "Esparsidade de Contexto no Tempo de Inferencia: Ilusao ou Oportunidade?"
 *               (gist.science technical summary), sec. 2 and 3C.
 *   [HBM]       "Nem Todos os Pensamentos Necessitam de HBM" (gist.science technical
 *               summary), Metodologia 1-4.
 *   [DHiSparse] "O Fim do Gargalo de Memoria: Como o Adaptive DHiSparse Revolutiona LLMs
 *               de Contexto Longo" (news page), "A Inovacao", "Metodologia e Eficiencia".
 */
#ifndef SDGQA_SD_H
#define SDGQA_SD_H

#include <stddef.h>
#include <stdint.h>

#ifdef __cplusplus
extern "C" {
#endif

typedef enum {
    SD_OK = 0,
    SD_ERR_INVALID_ARG = 1,   /* shape, pointer, alignment or workspace check failed */
    SD_ERR_UNSUPPORTED = 2,   /* valid request outside the compiled kernels (e.g. d) */
    SD_ERR_CUDA = 3,          /* a CUDA runtime call or launch failed */
    SD_ERR_DEVICE_BOUNDS = 4, /* reserved: reported through *err_word, see below */
    SD_ERR_TIMEOUT = 5        /* reserved: reported through *err_word, see below */
} sd_status;

typedef enum { SD_F32 = 0, SD_BF16 = 1, SD_F16 = 2 } sd_dtype;

/* Bits a kernel ORs into *err_word. */
#define SD_DEVERR_INDEX 0x1   /* a selected index outside [0, N) or [0, T) was skipped */
#define SD_DEVERR_SLOT 0x2    /* a slot_map entry outside [-1, pool_rows) was skipped */
#define SD_DEVERR_TIMEOUT 0x4 /* a bounded wait ran out; the kernel's outputs are invalid */

/* Library version: 100 * major + minor. */
int sd_version(void);

/* Static text for a status code. */
const char* sd_status_string(sd_status status);

/* Detail of the last failed call on this host thread ("" if none). */
const char* sd_last_error_message(void);

/*
 * sd_index_score -- compact indexer score of every cached token.
 * [SparDA] sec. 2 "Indexador de Previsao Compacto": one indexer head per GQA group
 * (= per KV head) scores each token with a plain dot product, with no softmax and no
 * loop over query heads.  With V > 1 query tokens sharing one selection (a speculative
 * verify batch whose tokens share the fetch of missing rows, [DHiSparse] "Metodologia")
 * the score is the maximum over the V queries:
 *     scores[b,h,t] = max_v  sum_j q_idx[b,h,v,j] * k_idx[b,h,t,j]
 * q_idx  [B,Hkv,V,d_idx] of q_dtype; k_idx [B,Hkv,N,d_idx] of k_dtype (token keys, or
 * the pooled block keys of sd_block_pool for block-granular selection, then N = blocks);
 * scores [B,Hkv,N] fp32 (written).  fp32 products and sums: integer-valued inputs with
 * |sum| < 2^24 give exact scores (likewise multiples of 2^-6, e.g. pooled block keys, with
 * |sum| < 2^18).  q_dtype and k_dtype are each F32 or BF16, or both F16 (q and k of one
 * 16-bit type run on the tensor cores).  Limits: d_idx in {64, 128}, 1 <= V <= 8, N >= 0.
 * key_hist: nullable [B*Hkv, SD_KEY_HIST_BINS] uint32 in/out.  When given, every score
 * written adds 1 to the bin of its top 11 order-key bits (the order key maps fp32 to
 * uint32 preserving order, -0.0 like +0.0).  Pass the same array to sd_topk for these
 * scores: it then skips its own first pass and leaves the array zeroed again.  The caller
 * zero-fills it once when it allocates it.
 * err_word: nullable device int32 (only SD_DEVERR_TIMEOUT can be set).
 */
#define SD_KEY_HIST_BINS 2048
sd_status sd_index_score(const void* q_idx, sd_dtype q_dtype, const void* k_idx,
                         sd_dtype k_dtype, int B, int Hkv, int V, int N, int d_idx,
                         float* scores, uint32_t* key_hist, int32_t* err_word, void* stream);

/*
 * sd_index_score_heads -- one score row per query row (no max over the V queries).
 * [Illusion] sec. 2 "Mecanismos de Esparsidade": Oracle Top-K selects per query head with the
 * attention query itself.  For every (b, kvh), query row v and token t:
 *     scores[b, kvh, v, t] = sum_j q[b, kvh, v, j] * k[b, kvh, t, j]
 * With the attention query [B, 1, Hq, d] seen as q [B, Hkv, G, d] (V = G) and the attention
 * keys k [B, Hkv, T, d], scores [B, Hkv, G, T] = [B, Hq, T] are every query head's unscaled
 * logits, the input of a per-head sd_topk (B*Hq rows).  Same dtypes and limits as
 * sd_index_score, except V <= 16 for bf16 q and k (tensor cores) and V <= 8 otherwise; the
 * sums are fp32 (exact for integer inputs; otherwise fp32 rounding in an order of the
 * kernel's choosing).  key_hist: nullable [B*Hkv*V, SD_KEY_HIST_BINS], one histogram per
 * score row, zero-filled by the caller.
 */
sd_status sd_index_score_heads(const void* q, sd_dtype q_dtype, const void* k, sd_dtype k_dtype, int B, int Hkv,
                               int V, int N, int d, float* scores, uint32_t* key_hist, int32_t* err_word,
                               void* stream);

/*
 * sd_block_pool -- block keys for block-granular selection (cache-build helper).
 * [SparDA] sec. 2 item 1 (top-k blocks) and "Estrategia de Treinamento" (pooling onto the
 * block grid).  Disjoint blocks of `block` tokens; the key of block n is the mean of its
 * tokens' indexer keys, computed in fp32 (exact for integer keys and power-of-two block):
 *     pooled[b,h,n,j] = (1/block) * sum_{t in [n*block, (n+1)*block)} k_idx[b,h,t,j]
 * k_idx [B,Hkv,T,d_idx] of k_dtype (F32 or BF16); pooled [B,Hkv,T/block,d_idx] of
 * pooled_dtype (written): F32, or F16 rounded to nearest even -- exact when the means are
 * multiples of 2^-14 below 2048 in magnitude with at most 11 significant bits, as for
 * integer keys in [-8, 8] and block <= 64 (half the key bytes, and with an F16 indexer
 * query the block scores run on the tensor cores).
 * T must be a multiple of block.  Limits: d_idx in {64, 128}, 1 <= block <= 4096.
 */
sd_status sd_block_pool(const void* k_idx, sd_dtype k_dtype, int B, int Hkv, int T, int d_idx,
                        int block, void* pooled, sd_dtype pooled_dtype, void* stream);

/*
 * sd_topk -- exact top-k per row.
 * [Illusion] sec. 2 "Mecanismos de Esparsidade" (Oracle Top-K: exact selection of the k
 * highest-scoring tokens); [SparDA] sec. 2 item 1 (top-k blocks).  Per row r, the k
 * entries first in the order (score descending, index ascending) -- ties go to the lower
 * index -- written in ascending index order.  -0.0 and +0.0 compare equal.
 * scores [rows,N] fp32 (NaN is outside the contract); idx [rows,k] int32 (written).
 * 0 <= k <= N.  key_hist: nullable [rows, SD_KEY_HIST_BINS] uint32, the histogram
 * sd_index_score accumulated for exactly these scores; when given, the select starts from
 * it (one pass over the scores instead of three) and the call zero-fills it again.
 * Uses no workspace in this version: sd_topk_workspace_bytes returns 0 and `workspace`
 * may be NULL.
 */
size_t sd_topk_workspace_bytes(int rows, int N, int k);
sd_status sd_topk(const float* scores, int rows, int N, int k, int32_t* idx, uint32_t* key_hist,
                  void* workspace, size_t workspace_bytes, void* stream);

/*
 * sd_gather_attend -- exact softmax attention over only the selected K/V rows.
 * [Illusion] sec. 2 (custom sparse decode kernels, irregular per token) and sec. 3C
 * (memory traffic O(k*d) instead of O(N*d)); [DHiSparse] "A Inovacao" (history in host
 * memory, only the selected rows fetched, fused with attention) and "Metodologia"
 * (queries share the fetch of missing rows); [HBM] Metodologia 3 (a row contributes the
 * same terms wherever it is stored).
 *
 * For query row (b, v, h) with kvh = h / (Hq/Hkv):
 *   rows_j = idx[b,kvh, j / block] * block + j % block, j < n_idx*block  (idx == NULL:
 *            dense, rows_j = j and n_idx*block must equal T; n_idx == 0 is an empty
 *            selection whatever idx is; an idx entry of -1 is an empty slot whose rows
 *            take no part, z_j = -inf, e.g. the padding of sd_window_union)
 *   z_j    = scale * q[b,v,h,:] . K[b,kvh,rows_j,:]
 *   out[b,v,h,:] = sum_j softmax(z)_j V[b,kvh,rows_j,:],  lse[b,v,h] = log sum_j exp(z_j)
 *   logits[b,v,h,j] = z_j (optional).  No rows: out = 0, lse = -inf.
 * Row source: with slot_map == NULL every row is read from k_cache/v_cache, which then
 * hold the whole cache [B,Hkv,T,d] (pool_rows == T).  With slot_map [B,T] int32, a row t
 * with slot_map[b,t] = s >= 0 is read from the HBM pool k_cache/v_cache [B,Hkv,pool_rows,d]
 * at slot s, and s == -1 reads it from pinned host memory k_host/v_host [B,Hkv,T,d]
 * through the device's mapping of that memory.  Each selected row is read once per
 * (b, kvh) and shared by all G*V query rows of the group.  The result does not depend on
 * where the rows were read from: bit-identical outputs for any slot_map.
 * Accumulation order depends only on (n_idx, block, splits), never on the data source.
 * Limits: d in {64, 128}; G*V <= 32; dtype F32 or BF16 for q, K and V alike.
 * The split-K partition over selected rows needs workspace (sd_gather_attend_workspace_bytes;
 * 0 when one split suffices): the splits' (m, l, o) partials, which a second kernel of the
 * call merges per (group, query row) in a fixed order.  The workspace needs no
 * initialisation and can be reused; calls sharing one workspace must not overlap on the
 * GPU.  splits = 0 picks one wave of CTAs for this GPU;
 * a requested split count is adjusted to at least one 64-row chunk per split and at most
 * 448 rows per split when rows are selected through idx or slot_map.
 * Draft ring ([DHiSparse] "Metodologia": the draft tokens' K/V live in a ring bounded by a
 * window; reading taken: the verify queries attend it causally): with ring_w > 0 the list
 * of every group is the n_idx*block selected rows followed by the ring_w slots of its KV
 * head's ring, and query token v of sequence b attends slot s only when
 * 0 <= ring_pos[b,s] <= qpos[b,v] (z = -inf otherwise); logits then have n_idx*block +
 * ring_w columns.  sd_ring_append fills the ring.
 * Residency per KV head: with slot_per_head = 1, slot_map is [B,Hkv,T] and the row of KV
 * head kvh at position t is in pool slot slot_map[b,kvh,t] (or host memory at -1), so the
 * KV heads of a sequence may keep different positions in the pool.
 * Staged host rows: with slot_map and k_stage/v_stage set, a row whose slot is -1 is read
 * from the stage at [group, j] (j = its position in the group's selection list, group =
 * b*Hkv + kvh, or b*Hq + h with per_head) instead of host memory; the stage must hold what
 * sd_stage_host_rows copied there for the same args.  Same values, so the same bits.
 * per_head = 1 ([Illusion] sec. 2: Oracle Top-K per query head): idx is [B,Hq,n_idx] and
 * query head h attends to its own selection idx[b,h,:], rows read from KV head
 * h / (Hq/Hkv) (all V query tokens of the head share it); the split plan and workspace then
 * count B*Hq groups of V query rows.  Needs idx.
 * Tiers ([HBM] Metodologia 1: T0 in HBM, T1 in host memory, T2 at 8 bits, T3 evicted;
 * Metodologia 3: a row contributes the same terms wherever it is stored): with tier set,
 * a row at a position whose tier is 3 takes no part (z = -inf, as an empty slot); a row
 * whose tier is 2 is read as K = k_int8 * k_scale, V = v_int8 * v_scale (its row of codes
 * and its per-row scale, as sd_quantize_rows_int8 writes them); rows of tiers 0 and 1 are
 * read as without tiers (from the pool, or host memory at slot -1, or the cache).  The
 * codes enter the tensor cores unchanged (small integers are exact in bf16) and the
 * scales multiply the row's logit and its softmax weight in fp32.  A call in which no
 * selected row has tier 2 or 3 gives the bits of the same call without tiers and with
 * row_loop = 1.  Limits: bf16, d = 128, not per_head, no ring, no
 * stage; T and pool_rows < 2^29.
 * Dense calls over a cache in HBM (idx, slot_map, tier, ring and stage all unset, not
 * per_head; bf16, d = 128, G*V <= 16) move each split's contiguous rows as whole 64-row
 * tiles (tiled TMA into a two-stage ring per CTA) through a tile that puts the keys on the
 * tensor cores' M side; their splits are ranges of whole tiles (never more than the
 * workspace holds).  Block-sparse calls over a cache in HBM (idx set, block a multiple of
 * 16, T a multiple of block, logits NULL, otherwise as dense calls) take the same tiles,
 * each 64-row stage made of four 16-row boxes at the selected blocks' rows (an empty or bad
 * index loads nothing and is masked; a bad one is reported as without tiles).  Same values
 * within rounding, in another summation order; row_loop = 1 makes such a call run the
 * general row loop instead, e.g. to compare its bits with a tiered, pooled or staged
 * call's.
 * The kernel is launched as a programmatic dependent of the preceding kernel in the
 * stream (it waits for that kernel's results before reading anything).
 */
typedef struct {
    const void* q;            /* [B,V,Hq,d] */
    const void* k_cache;      /* [B,Hkv,pool_rows,d]: HBM pool, or full cache if !slot_map */
    const void* v_cache;      /* same layout as k_cache */
    const void* k_host;       /* pinned host [B,Hkv,T,d], or NULL when slot_map == NULL */
    const void* v_host;       /* pinned host [B,Hkv,T,d], or NULL when slot_map == NULL */
    const int32_t* slot_map;  /* [B,T] slot or -1, or NULL */
    const int32_t* idx;       /* [B,Hkv,n_idx] selected tokens or blocks, or NULL (dense) */
    sd_dtype dtype;
    int B, V, Hq, Hkv, d, T, pool_rows, n_idx, block;
    float scale;              /* softmax scale, e.g. 1/sqrt(d) */
    float* out;               /* [B,V,Hq,d] fp32, written */
    float* lse;               /* [B,V,Hq] fp32 natural-log log-sum-exp, written */
    float* logits;            /* [B,V,Hq,n_idx*block] fp32, written if not NULL */
    int32_t* err_word;        /* nullable device int32 */
    void* workspace;          /* device scratch of workspace_bytes */
    size_t workspace_bytes;
    int splits;               /* 0 = automatic */
    int per_head;             /* 1: idx is [B,Hq,n_idx], one selection per query head */
    const void* k_stage;      /* nullable HBM stage [groups, n_idx*block, d] (sd_stage_host_rows) */
    const void* v_stage;      /* same layout as k_stage; both set or both NULL */
    const void* ring_k;       /* draft ring [B,Hkv,ring_w,d] (device, dtype), or NULL */
    const void* ring_v;       /* same layout as ring_k */
    const int32_t* ring_pos;  /* [B,ring_w] token position held by each slot, -1 = empty */
    const int32_t* qpos;      /* [B,V] token position of each query token */
    int ring_w;               /* ring slots; 0 = no ring */
    int slot_per_head;        /* 1: slot_map is [B,Hkv,T], one residency map per KV head */
    const uint8_t* tier;      /* nullable [B,T] tier of every position (sd_tier_classify) */
    const int8_t* k_int8;     /* [B,Hkv,T,d] int8 codes of the T2 rows of K (sd_quantize_rows_int8) */
    const int8_t* v_int8;     /* same layout, of V */
    const float* k_scale;     /* [B,Hkv,T] fp32 scales of the T2 rows of K */
    const float* v_scale;     /* [B,Hkv,T] fp32, of V */
    int row_loop;             /* 1: a dense or tiled block-sparse call runs the general row loop (see above) */
} sd_attend_args;

size_t sd_gather_attend_workspace_bytes(const sd_attend_args* args);
sd_status sd_gather_attend(const sd_attend_args* args, void* stream);

/*
 * sd_gather_attend_noalloc -- sd_gather_attend for callers that cannot allocate device
 * memory.  The source pages have no counterpart: this is a library convenience.
 * Some callers cannot provide the split-K scratch buffer: a plugin that only receives
 * input and output pointers from a framework owning all device memory, an engine that
 * fixes its memory budget at start-up, or a C caller with no allocator at hand.  This call
 * computes exactly what sd_gather_attend computes (same arguments, same split plan) but
 * ignores args->workspace / workspace_bytes and uses a 16 MiB array of device memory
 * compiled into the library, which every GPU that loads the library holds until exit.
 * It allocates nothing.  On the first call made on each device (with that device
 * current) the array's device address is looked up and the array is cleared once: make
 * that first call before any stream capture.  The address is kept for the life of the
 * process, so do not use this call on a device after cudaDeviceReset.  All calls share the array and it keeps the
 * last call's contents (nothing in it needs to start at zero), so calls whose kernels
 * overlap on the GPU race on the array.  A request
 * whose split-K partials need more than 16 MiB returns SD_ERR_INVALID_ARG without
 * launching (pass a smaller `splits`, or use sd_gather_attend with a workspace).
 */
sd_status sd_gather_attend_noalloc(const sd_attend_args* args, void* stream);

/*
 * sd_stage_host_rows -- copy the selected rows that live in host memory into an HBM stage.
 * [DHiSparse] "A Inovacao" (the history stays in host memory and only the selected rows
 * are fetched) and "Metodologia" (the query rows of a group share the fetch of a missing
 * row); [SparDA] sec. 2 item 3 (a kernel moves the needed rows from host memory through
 * unified addressing ahead of the attention).
 * With the same args as the sd_gather_attend call that follows (slot_map, k_host/v_host,
 * idx, n_idx, block, per_head and k_stage/v_stage must be set): for every group g (b*Hkv +
 * kvh, or b*Hq + h with per_head) and list row j < n_idx*block whose token
 * t = idx[g, j/block]*block + j%block has slot_map[b,t] == -1, copies K/V host row
 * [b, kvh, t, :] (kvh = h / (Hq/Hkv) with per_head) to k_stage/v_stage[g, j, :].  Other
 * stage rows are left as they are; empty slots (-1), pool rows and rows that
 * sd_gather_attend would reject (reported through err_word) are skipped.  The copy is
 * spread over every SM: warps take chunks of rows from counter[0], a caller-owned device
 * uint32[2] that must be zero-filled before the first call and is left at zero by every
 * call (calls sharing one counter must not overlap on the GPU).  The result does not depend
 * on which warp copied which row.  Launched as a programmatic dependent of the preceding
 * kernel; sd_gather_attend launched after it waits for it.  Limits as sd_gather_attend.
 */
sd_status sd_stage_host_rows(const sd_attend_args* args, uint32_t* counter, void* stream);

/*
 * sd_promote_rows -- keep the HBM pool as a cache of host rows.
 * [DHiSparse] "Metodologia" (the GPU keeps extra history while memory allows and fetches
 * the rest); [SparDA] sec. 2 item 3 (the needed rows are fetched ahead).  Reading taken,
 * per sequence b: the step's selected positions (the union over the groups of args->idx,
 * block-expanded, -1 entries empty) whose slot_map is -1 are the misses; in ascending
 * position order they go to the first slots of a ring of pool_rows slots, taken in order
 * from hand[b], that do not hold a position selected in this step.  A slot's old position
 * leaves the pool (slot_map = -1); the miss's K and V rows of every KV head are copied from
 * k_host/v_host into the pool (args->k_cache/v_cache, which this call writes), slot_map[b,
 * miss] = slot, pool_pos[b, slot] = miss, and hand[b] moves past the last slot taken.
 * Misses beyond the free slots stay in host memory.  A following sd_gather_attend reads the
 * promoted rows from HBM, with the same bits (the values are the same).  With
 * slot_per_head = 1 every (b, KV head) is such a unit of its own (its selection, its slot
 * map row, its pool slots; one row per miss): pool_pos is then [B*Hkv, pool_rows] and hand
 * [B*Hkv].
 * pool_pos [B, pool_rows] int32 (slot -> position, -1 empty) and hand [B] int32 are the
 * caller's device state, kept consistent with slot_map between calls.  The workspace
 * (sd_promote_rows_workspace_bytes) must be zero-filled before the first call; every call
 * leaves it ready for the next.  Three launches (mark, plan, copy), each a programmatic
 * dependent of the one before.  Limits as sd_gather_attend; needs idx, slot_map, the pool
 * and the host cache.
 */
size_t sd_promote_rows_workspace_bytes(const sd_attend_args* args);
sd_status sd_promote_rows(const sd_attend_args* args, int32_t* pool_pos, int32_t* hand, void* workspace,
                          size_t workspace_bytes, void* stream);

/*
 * sd_promote_staged_rows -- sd_promote_rows with the promoted rows taken from the HBM stage.
 * [DHiSparse] "Metodologia" and [SparDA] sec. 2 item 3, as sd_promote_rows; the order of the
 * calls is a reading: the step's misses cross the host link once, into the stage
 * (sd_stage_host_rows), the attention reads them there, and only then are they promoted, so
 * the promotion can run beside the next step's selection.
 * Leaves slot_map, pool_pos, hand and the pool exactly as sd_promote_rows would with the same
 * arguments and state.  Contract: slot_per_head = 1 (a unit is one (b, KV head), so each
 * promoted row is the one its own head staged), and args->k_stage/v_stage hold what
 * sd_stage_host_rows copied for these args with slot_map as it is now (no promotion in
 * between); the host cache is not read.  A stage not filled that way gives wrong pool rows
 * but no out-of-bounds access.  The workspace (sd_promote_staged_rows_workspace_bytes, a
 * [B*Hkv, T] int32 map beyond sd_promote_rows' layout) is zero-filled before the first call
 * and left ready for the next.  Errors as sd_promote_rows; SD_ERR_INVALID_ARG without
 * slot_per_head or the stage, or with B*Hkv*groups*n_idx*block >= 2^31.
 */
size_t sd_promote_staged_rows_workspace_bytes(const sd_attend_args* args);
sd_status sd_promote_staged_rows(const sd_attend_args* args, int32_t* pool_pos, int32_t* hand, void* workspace,
                                 size_t workspace_bytes, void* stream);

/*
 * sd_ring_append -- write new tokens' K/V into the window-bounded draft ring.
 * [DHiSparse] "Metodologia" (the draft tokens' K/V live in a ring bounded by a window).
 * Token i < n of sequence b, at position pos0[b] + i, goes to slot (pos0[b] + i) mod W:
 * ring_k/ring_v[b, h, slot, :] = k_new/v_new[b, h, i, :] for every KV head h, and
 * ring_pos[b, slot] = pos0[b] + i.  k_new, v_new [B,Hkv,n,d] and ring_k, ring_v
 * [B,Hkv,W,d] of `dtype`; ring_pos [B,W] int32; pos0 [B] int32 (device, >= 0).  Limits:
 * 1 <= n <= W (no slot is written twice in one call), d in {64, 128}.
 */
sd_status sd_ring_append(const void* k_new, const void* v_new, sd_dtype dtype, int B, int Hkv, int n, int d,
                         void* ring_k, void* ring_v, int32_t* ring_pos, const int32_t* pos0, int W, void* stream);

/*
 * sd_select_attend -- sd_topk and sd_gather_attend fused in one launch.
 * [Illusion] sec. 2 "Mecanismos de Esparsidade" (Oracle Top-K feeding a sparse decode
 * kernel) and sec. 3C; [SparDA] sec. 2 item 1 (top-k blocks); [DHiSparse] "Metodologia"
 * (the query rows of a group share each fetched row).
 * Computes what sd_topk(scores, B*Hkv, N, n_idx, idx, key_hist) followed by
 * sd_gather_attend(args with idx) computes: idx [B,Hkv,n_idx] int32 (written, ascending,
 * bit-identical to sd_topk), out, lse and optional logits as sd_gather_attend defines
 * them, with the selection list of every (b, kvh) taken from idx.  args->idx, workspace,
 * workspace_bytes, k_stage and v_stage are ignored; k = args->n_idx; a draft ring
 * (ring_w > 0) is not supported here (SD_ERR_UNSUPPORTED: use the separate calls).  scores [B*Hkv, N] fp32 with
 * N * args->block == args->T (one score per token, or per block of `block` tokens).
 * key_hist: nullable, as in sd_topk (the indexer's histogram of exactly these scores;
 * zero-filled again by the call).  args->splits: CTAs per (b, kvh), 0 = automatic, at most
 * 8; they form one thread-block cluster that exchanges the selection threshold and merges
 * the attention partials through distributed shared memory, so no workspace is needed.
 * The summation order of the attention depends on (N, n_idx, block, splits) and on which
 * part of the row each selected entry falls in, never on where the rows are stored.
 * Limits: bf16 q/K/V, d in {64, 128}, G*V <= 32 (other inputs: SD_ERR_UNSUPPORTED, use the
 * two separate calls).  Launched as a programmatic dependent of the preceding kernel.
 */
sd_status sd_select_attend(const float* scores, int N, uint32_t* key_hist, int32_t* idx,
                           const sd_attend_args* args, void* stream);

/*
 * sd_decode_step -- one whole decode step in one launch: sd_index_score, sd_topk and
 * sd_gather_attend fused in a persistent kernel for K/V resident in HBM.
 * [SparDA] sec. 2 "Indexador de Previsao Compacto" (one indexer head per KV group, no softmax)
 * and item 1 (top-k blocks); [Illusion] sec. 2 "Mecanismos de Esparsidade" (exact top-k feeding
 * a sparse decode kernel) and sec. 3C (traffic O(k*d)); [DHiSparse] "Metodologia" (the query
 * rows of a group share every fetched row).
 * Computes, with N = T / block:
 *   scores [B,Hkv,N] = sd_index_score(q_idx, keys)   (max over the V queries; bit-identical)
 *   idx [B,Hkv,n_idx] = sd_topk(scores, n_idx)       (ascending, ties to the lower index;
 *                                                     bit-identical)
 *   out [B,V,Hq,d], lse [B,V,Hq] = sd_gather_attend over the selected rows of k_cache/v_cache
 *                                  (entry e covers rows e*block .. e*block + block - 1), with
 *                                  the same definition; the summation order is the call's own
 *                                  and depends only on (T, block, n_idx), not on the data.
 * q_idx [B,Hkv,V,d_idx] and keys [B,Hkv,N,d_idx] both of key_dtype (SD_BF16, or SD_F16 e.g. for
 * the pooled block keys of sd_block_pool): products and sums are fp32, exact for the
 * integer-valued (or multiple-of-2^-6) indexer inputs sd_index_score describes.  q [B,V,Hq,d],
 * k_cache and v_cache [B,Hkv,T,d] bf16; scores, idx, out and lse are written.
 * Limits: d = d_idx = 128, 1 <= V <= 8, (Hq/Hkv)*V <= 16, N <= 65536, 0 <= n_idx <= N,
 * B*Hkv*T < 2^31 (SD_ERR_UNSUPPORTED outside the first three; use the separate calls).
 * Workspace (sd_decode_step_workspace_bytes; 256-byte aligned): task counters, per-group
 * counters and histograms, and the attention partials.  Zero-fill it once before the first
 * call; every call leaves it ready for the next (its counters and histograms back at zero).
 * Calls sharing one workspace must not overlap on the GPU.  After a call that reported
 * SD_DEVERR_TIMEOUT the workspace must be zero-filled again before the next call.
 * lag: the scoring of group g + lag is scheduled before the attention of group g (0 =
 * automatic); wait_limit_ns: the bound of every wait inside the kernel (0 = 1 s).
 * The launch is a programmatic dependent of the preceding kernel in the stream (it waits for
 * that kernel's results before reading anything).
 */
typedef struct {
    const void* q_idx;        /* [B,Hkv,V,d_idx] of key_dtype */
    const void* keys;         /* [B,Hkv,T/block,d_idx] of key_dtype */
    sd_dtype key_dtype;       /* SD_BF16 or SD_F16 */
    const void* q;            /* [B,V,Hq,d] bf16 */
    const void* k_cache;      /* [B,Hkv,T,d] bf16, HBM */
    const void* v_cache;      /* same layout as k_cache */
    int B, V, Hq, Hkv, d, d_idx, T, block, n_idx;
    float scale;              /* softmax scale, e.g. 1/sqrt(d) */
    float* scores;            /* [B,Hkv,T/block] fp32, written (16-byte aligned) */
    int32_t* idx;             /* [B,Hkv,n_idx] int32, written (may be NULL when n_idx == 0) */
    float* out;               /* [B,V,Hq,d] fp32, written */
    float* lse;               /* [B,V,Hq] fp32, written */
    int32_t* err_word;        /* nullable device int32 */
    void* workspace;          /* device scratch of workspace_bytes, zero-filled before first use */
    size_t workspace_bytes;
    int lag;                  /* 0 = automatic */
    long long wait_limit_ns;  /* 0 = 1 s */
} sd_decode_step_args;

size_t sd_decode_step_workspace_bytes(const sd_decode_step_args* args);
sd_status sd_decode_step(const sd_decode_step_args* args, void* stream);

/*
 * sd_window_max -- block scores on overlapping compression windows.
 * [SparDA] "Estrategia de Treinamento": the inference block grid is a compression window of
 * `kernel` tokens moved by `stride` (32, 16), and finer scores are max-pooled onto it.
 * Reading taken: window n's score is the maximum of the token scores it covers,
 *     wscores[r, n] = max over t in [n*stride, min(n*stride + kernel, N)) of scores[r, t],
 * n < NW = sd_window_count(N, kernel, stride) = 1 + ceil((N - kernel) / stride) (1 when
 * N <= kernel, 0 when N == 0).  scores [rows, N] fp32 (as written by sd_index_score);
 * wscores [rows, NW] fp32 (written).  key_hist: nullable [rows, SD_KEY_HIST_BINS] uint32,
 * zero-filled by the caller; the call adds the histogram sd_topk takes for these window
 * scores.  Limits: 1 <= stride <= kernel <= 1024.
 */
int sd_window_count(int N, int kernel, int stride);
sd_status sd_window_max(const float* scores, int rows, int N, int kernel, int stride, float* wscores,
                        uint32_t* key_hist, void* stream);

/*
 * sd_window_union -- the tokens of the selected windows, each once.
 * Windows overlap, so a token can lie in two selected windows; attention must see it once.
 * With kernel a multiple of stride and N a multiple of stride, the tokens are whole segments
 * of `stride` tokens: window n covers segments n .. n + kernel/stride - 1 (those below
 * N/stride).  Per row r: the union of the segments of the windows in widx[r, 0..k),
 * ascending, written to segs[r, 0..), padded with -1 (empty slots) to max_segs entries;
 * segs feeds sd_gather_attend with block = stride and n_idx = max_segs.
 * widx [rows, k] int32 window indices in [0, NW) (others are skipped and set
 * SD_DEVERR_INDEX in *err_word); segs [rows, max_segs] int32 (written);
 * max_segs >= k * kernel/stride.  Limit: N/stride <= 65536 segments per row.
 */
sd_status sd_window_union(const int32_t* widx, int rows, int k, int N, int kernel, int stride, int32_t* segs,
                          int max_segs, int32_t* err_word, void* stream);

/*
 * sd_score_accumulate -- one layer's term of the cumulative attention-importance score.
 * [HBM] Metodologia 2:  s_i(t) = s_i(t-1) + (1/|L|) sum_l (1/H) sum_h alpha_{l,h}(t)[i].
 * Adds, for every query row (b, v, h) and selected row j (expanded as in
 * sd_gather_attend, kvh = h / (Hq/Hkv)):
 *     s[b, rows_j] += weight * exp(logits[b,v,h,j] - lse[b,v,h])
 * so calling it once per layer with weight = 1/(|L| * Hq) applies the equation.
 * logits [B,V,Hq,n_idx*block] and lse [B,V,Hq] fp32 as written by sd_gather_attend;
 * idx [B,Hkv,n_idx] or NULL (dense); s [B,T] fp64, updated in place.
 * Rows not selected, and the rows of empty slots (-1), receive nothing.  Order of
 * additions into one s entry is not fixed
 * when several KV groups select it (fp64 atomics); the result varies only by rounding.
 */
sd_status sd_score_accumulate(const float* logits, const float* lse, const int32_t* idx, int B,
                              int V, int Hq, int Hkv, int n_idx, int block, int T, double weight,
                              double* s, int32_t* err_word, void* stream);

/*
 * sd_tier_classify -- four-tier residency classes from the importance score.
 * [HBM] Metodologia 1: T0 (HBM) = protected tokens (prompt/sinks = the first n_sink
 * positions, recent window = the last n_recent) and the most important; T1 (host DDR,
 * full precision); T2 (8-bit); T3 (evicted, the least important tail).  Metodologia 4:
 * the caller re-runs it every Delta = 64 decode steps.
 * Per sequence: protected positions rank first (in index order), then the others by
 * (s descending, index ascending).  With c_m = floor(cum_frac[m] * T):
 *   rank < c_0 -> 0, < c_1 -> 1, < c_2 -> 2, else 3; protected positions are always 0.
 * s [B,T] fp64; tier [B,T] uint8 and counts [B,4] int32 (written).
 * cum_frac must be nondecreasing within [0, 1].  Workspace: sd_tier_classify_workspace_bytes.
 */
size_t sd_tier_classify_workspace_bytes(int B, int T);
sd_status sd_tier_classify(const double* s, int B, int T, const double cum_frac[3], int n_sink,
                           int n_recent, uint8_t* tier, int32_t* counts, void* workspace,
                           size_t workspace_bytes, void* stream);

/*
 * sd_quantize_rows_int8 -- 8-bit storage of the T2 rows of one K or V cache.
 * [HBM] Metodologia 1 (T2 keeps low-importance tokens at reduced precision, "e.g. 8-bit").
 * The pages give no scheme; this is symmetric per-row absmax: a = max_j |x_j| (fp32);
 * a == 0 gives scale 0 and zero codes; else scale = a/127 and
 * code_j = clamp(rint(x_j * (127/a)), -127, 127), each division and the product a
 * correctly rounded fp32 operation, rint = round half to even.
 * x [B,Hkv,T,d] of dtype; tier [B,T] uint8; only rows with tier == 2 are written:
 * codes [B,Hkv,T,d] int8, scales [B,Hkv,T] fp32.  Limits: d in {64, 128}.
 */
sd_status sd_quantize_rows_int8(const void* x, sd_dtype dtype, const uint8_t* tier, int B,
                                int Hkv, int T, int d, int8_t* codes, float* scales,
                                void* stream);

#ifdef __cplusplus
}
#endif

#endif /* SDGQA_SD_H */
