/*
 * oracle.c -- plain, slow CPU oracle for top-k sparse decode attention with GQA.
 *
 * TEST INFRASTRUCTURE ONLY.  Nothing on the product path may call, link or load this
 * file: only the tests, the package's smoke check and the benchmark's CPU-baseline leg
 * use it.  It shares no code, header, table or constant with the CUDA library.
 *
 * Every function is the textbook definition of one step, written as loops in fp64
 * (fp32 where noted, for the one step whose output is an integer code decided by a
 * floating-point product).  No blocking, fusion or reordering: the loops follow the
 * definition so a reader can check them by eye.  Each function names the passage of
 * the source pages it restates.
 *
 * Sources (web pages, cited by title and section):
 *   [SparDA]   "SparDA: Atencao Esparsa Desacoplada ..." (gist.science summary),
 *              sec. 2 "Indexador de Previsao Compacto" and "Estrategia de Treinamento".
 *   [Illusion] "Esparsidade de Contexto no Tempo de Inferencia: Ilusao ou Oportunidade?"
 *              (gist.science summary), sec. 2 "Mecanismos de Esparsidade", sec. 3C.
 *   [HBM]      "Nem Todos os Pensamentos Necessitam de HBM" (gist.science summary),
 *              Metodologia 1 (four tiers), 2 (importance score equation), 3 (Prop. 1), 4.
 *   [DHiSparse] "O Fim do Gargalo de Memoria: Como o Adaptive DHiSparse ..." (news page),
 *              "A Inovacao" and "Metodologia e Eficiencia de Carga".
 *
 * Parity pins: every function here is pinned by the not-gpu tests against closed forms,
 * brute force or library routines (see tests/test_oracle_*.py); none is "parity unpinned".
 *
 * Element types: dtype 0 = IEEE fp32, dtype 1 = bfloat16 given as its raw 16 bits.
 * A bfloat16 value is the fp32 value whose upper 16 bits are those bits, so the
 * conversion below is exact.
 */
#include <math.h>
#include <stdint.h>
#include <stdlib.h>
#include <string.h>

#define ORC_F32 0
#define ORC_BF16 1

/* Return codes. */
#define ORC_OK 0
#define ORC_BAD_ARG (-1)
#define ORC_BAD_INDEX (-2)

static double orc_elem(const void* base, int dtype, size_t i) {
    if (dtype == ORC_F32) return (double)((const float*)base)[i];
    uint32_t bits = ((uint32_t)((const uint16_t*)base)[i]) << 16;
    float f;
    memcpy(&f, &bits, sizeof f);
    return (double)f;
}

static void orc_load_row(const void* base, int dtype, size_t offset, int n, double* dst) {
    for (int j = 0; j < n; ++j) dst[j] = orc_elem(base, dtype, offset + (size_t)j);
}

int oracle_num_threads(void) {
#ifdef _OPENMP
    extern int omp_get_max_threads(void);
    return omp_get_max_threads();
#else
    return 1;
#endif
}

/*
 * Step 1 -- compact indexer score.  [SparDA] sec. 2 "Indexador de Previsao Compacto":
 * one indexer head per GQA group (= per KV head) scores each cached token with a
 * plain dot product, with no softmax and no loop over query heads.
 *
 *   scores[b,h,t] = max over v of  sum_j  q_idx[b,h,v,j] * k_idx[b,h,t,j]
 *
 * The max over v (V > 1) is the reading used for a speculative-verify batch whose V
 * query tokens share one selection ([DHiSparse] "Metodologia": queries share the
 * retrieval of missing rows).  With V = 1 it is the plain score.
 * Layouts: q_idx [B,Hkv,V,dI], k_idx [B,Hkv,N,dI], scores [B,Hkv,N].
 */
int oracle_index_score(const void* q_idx, int q_dtype, const void* k_idx, int k_dtype,
                       int B, int Hkv, int V, int N, int dI, double* scores) {
    if (B < 0 || Hkv < 0 || V < 1 || N < 0 || dI < 1) return ORC_BAD_ARG;
#pragma omp parallel for collapse(2) schedule(dynamic)
    for (int b = 0; b < B; ++b) {
        for (int h = 0; h < Hkv; ++h) {
            double* q = (double*)malloc(sizeof(double) * (size_t)V * dI);
            double* k = (double*)malloc(sizeof(double) * (size_t)dI);
            for (int v = 0; v < V; ++v)
                orc_load_row(q_idx, q_dtype, (((size_t)b * Hkv + h) * V + v) * dI, dI, q + (size_t)v * dI);
            for (int t = 0; t < N; ++t) {
                orc_load_row(k_idx, k_dtype, (((size_t)b * Hkv + h) * N + t) * dI, dI, k);
                double best = -INFINITY;
                for (int v = 0; v < V; ++v) {
                    double dot = 0.0;
                    for (int j = 0; j < dI; ++j) dot += q[(size_t)v * dI + j] * k[j];
                    if (dot > best) best = dot;
                }
                scores[((size_t)b * Hkv + h) * N + t] = best;
            }
            free(q);
            free(k);
        }
    }
    return ORC_OK;
}

/*
 * Step 1, per query -- [Illusion] sec. 2 "Mecanismos de Esparsidade": Oracle Top-K selects
 * per query head with the attention query itself, so every query row keeps its own scores:
 *
 *   scores[b,h,v,t] = sum_j  q[b,h,v,j] * k[b,h,t,j]      (no max over v)
 *
 * With the attention query [B,1,Hq,d] read as [B,Hkv,G,d] (V = G) these are every query
 * head's unscaled logits.  Layouts: q [B,Hkv,V,dI], k [B,Hkv,N,dI], scores [B,Hkv,V,N].
 */
int oracle_index_score_heads(const void* q_in, int q_dtype, const void* k_in, int k_dtype, int B, int Hkv, int V,
                             int N, int dI, double* scores) {
    if (B < 0 || Hkv < 0 || V < 1 || N < 0 || dI < 1) return ORC_BAD_ARG;
#pragma omp parallel for collapse(2) schedule(dynamic)
    for (int b = 0; b < B; ++b) {
        for (int h = 0; h < Hkv; ++h) {
            double* q = (double*)malloc(sizeof(double) * (size_t)V * dI);
            double* k = (double*)malloc(sizeof(double) * (size_t)dI);
            for (int v = 0; v < V; ++v)
                orc_load_row(q_in, q_dtype, (((size_t)b * Hkv + h) * V + v) * dI, dI, q + (size_t)v * dI);
            for (int t = 0; t < N; ++t) {
                orc_load_row(k_in, k_dtype, (((size_t)b * Hkv + h) * N + t) * dI, dI, k);
                for (int v = 0; v < V; ++v) {
                    double dot = 0.0;
                    for (int j = 0; j < dI; ++j) dot += q[(size_t)v * dI + j] * k[j];
                    scores[(((size_t)b * Hkv + h) * V + v) * N + t] = dot;
                }
            }
            free(q);
            free(k);
        }
    }
    return ORC_OK;
}

/*
 * Step 1' -- block key for block-granular selection.  [SparDA] sec. 2 item 1 selects
 * top-k *blocks*, and "Estrategia de Treinamento" pools finer scores onto a block grid.
 * Reading taken: disjoint blocks of `block` tokens; the block key is the mean of the
 * block's indexer keys.  T must be a multiple of block.
 *
 *   pooled[b,h,n,j] = (1/block) * sum over t in [n*block, (n+1)*block) of k_idx[b,h,t,j]
 */
int oracle_block_pool(const void* k_idx, int k_dtype, int B, int Hkv, int T, int dI, int block,
                      double* pooled) {
    if (block < 1 || T % block != 0 || dI < 1) return ORC_BAD_ARG;
    int NB = T / block;
#pragma omp parallel for collapse(2) schedule(static)
    for (int b = 0; b < B; ++b)
        for (int h = 0; h < Hkv; ++h)
            for (int n = 0; n < NB; ++n)
                for (int j = 0; j < dI; ++j) {
                    double sum = 0.0;
                    for (int t = n * block; t < (n + 1) * block; ++t)
                        sum += orc_elem(k_idx, k_dtype, (((size_t)b * Hkv + h) * T + t) * dI + j);
                    pooled[(((size_t)b * Hkv + h) * NB + n) * dI + j] = sum / (double)block;
                }
    return ORC_OK;
}

/* (score, index) pair ordered by score descending, then index ascending. */
typedef struct {
    double s;
    int32_t i;
} orc_pair;

static int orc_pair_cmp(const void* pa, const void* pb) {
    const orc_pair* a = (const orc_pair*)pa;
    const orc_pair* b = (const orc_pair*)pb;
    if (a->s > b->s) return -1;
    if (a->s < b->s) return 1;
    return (a->i < b->i) ? -1 : (a->i > b->i) ? 1 : 0;
}

static int orc_int_cmp(const void* pa, const void* pb) {
    int32_t a = *(const int32_t*)pa, b = *(const int32_t*)pb;
    return (a < b) ? -1 : (a > b) ? 1 : 0;
}

/*
 * Step 2 -- exact top-k.  [Illusion] sec. 2 "Mecanismos de Esparsidade" ("Oracle Top-K":
 * exact selection of the k highest-scoring tokens); [SparDA] sec. 2 item 1 (top-k blocks).
 * Ties, on which the pages are silent, go to the lower index.  The chosen set is emitted
 * in ascending index order.
 *
 * Per row: sort all indices by (score descending, index ascending) -- a total order, so
 * the result is unique -- keep the first k, then sort those k ascending.
 * scores [rows, N] -> idx [rows, k].
 */
int oracle_topk(const double* scores, int rows, int N, int k, int32_t* idx) {
    if (rows < 0 || N < 0 || k < 0 || k > N) return ORC_BAD_ARG;
#pragma omp parallel for schedule(dynamic)
    for (int r = 0; r < rows; ++r) {
        orc_pair* p = (orc_pair*)malloc(sizeof(orc_pair) * (size_t)(N > 0 ? N : 1));
        for (int t = 0; t < N; ++t) {
            p[t].s = scores[(size_t)r * N + t];
            p[t].i = t;
        }
        qsort(p, (size_t)N, sizeof(orc_pair), orc_pair_cmp);
        int32_t* out = idx + (size_t)r * k;
        for (int j = 0; j < k; ++j) out[j] = p[j].i;
        qsort(out, (size_t)k, sizeof(int32_t), orc_int_cmp);
        free(p);
    }
    return ORC_OK;
}

/*
 * Step 3 -- exact attention over only the selected rows.  [Illusion] sec. 2 (custom
 * sparse decode kernels, irregular per token) and sec. 3C (traffic O(k*d) instead of
 * O(N*d)); [HBM] Metodologia 3 (a row contributes the same terms wherever it was
 * stored, so this function has no notion of where a row lives).
 *
 * For each query row (b, v, h), with kvh = h / (Hq/Hkv):
 *   rows_j = idx[b,kvh, j / block] * block + (j % block),  j = 0 .. n_idx*block - 1
 *            (identity rows_j = j when idx is NULL: dense attention over all T rows)
 *   z_j    = scale * sum_c q[b,v,h,c] * K[b,kvh,rows_j,c]
 *   m      = max_j z_j,  w_j = exp(z_j - m),  l = sum_j w_j
 *   out    = sum_j w_j * Vv[b,kvh,rows_j,:] / l,   lse = m + log(l)
 *   logits[b,v,h,j] = z_j  (if logits != NULL)
 * per_head = 1 ([Illusion] sec. 2, Oracle Top-K per query head): idx is [B,Hq,n_idx] and
 * query head h takes its rows from idx[b,h,:] (still from KV head kvh = h / G).
 * An idx entry of -1 is an empty slot: its rows take no part (z_j = -infinity, weight 0);
 * reading taken for selections of varying size padded to a fixed length (the union of
 * overlapping windows).  An empty selection gives out = 0 and lse = -infinity.
 * Layouts: q [B,V,Hq,d]; K, Vv [B,Hkv,T,d]; idx [B,Hkv,n_idx]; out [B,V,Hq,d];
 * lse [B,V,Hq]; logits [B,V,Hq,n_idx*block].  Returns ORC_BAD_INDEX if a row is
 * outside [0, T).
 */
int oracle_gather_attend(const void* q, const void* K, const void* Vv, int dtype,
                         const int32_t* idx, int B, int V, int Hq, int Hkv, int d, int T,
                         int n_idx, int block, double scale, double* out, double* lse,
                         double* logits, int per_head) {
    if (Hkv < 1 || Hq % Hkv != 0 || d < 1 || block < 1 || n_idx < 0) return ORC_BAD_ARG;
    if (idx == NULL && n_idx * block != T) return ORC_BAD_ARG;
    const int G = Hq / Hkv;
    const long n_rows = (long)n_idx * block;
    int bad = 0;
#pragma omp parallel for collapse(3) schedule(dynamic) reduction(| : bad)
    for (int b = 0; b < B; ++b)
        for (int v = 0; v < V; ++v)
            for (int h = 0; h < Hq; ++h) {
                const int kvh = h / G;
                const size_t qrow = (((size_t)b * V + v) * Hq + h);
                double* qv = (double*)malloc(sizeof(double) * (size_t)d);
                double* kr = (double*)malloc(sizeof(double) * (size_t)d);
                double* acc = (double*)malloc(sizeof(double) * (size_t)d);
                double* z = (double*)malloc(sizeof(double) * (size_t)(n_rows > 0 ? n_rows : 1));
                long* rows = (long*)malloc(sizeof(long) * (size_t)(n_rows > 0 ? n_rows : 1));
                orc_load_row(q, dtype, qrow * d, d, qv);
                for (long j = 0; j < n_rows; ++j) {
                    long row = j;
                    if (idx != NULL) {
                        const size_t irow = per_head ? (size_t)b * Hq + h : (size_t)b * Hkv + kvh;
                        const long sel = idx[irow * n_idx + j / block];
                        row = sel == -1 ? -1 : sel * block + j % block;
                        if (sel != -1 && (sel < 0 || row >= T)) {
                            bad = 1;
                            row = -1;
                        }
                    }
                    rows[j] = row;
                }
                double m = -INFINITY;
                long n_valid = 0;
                for (long j = 0; j < n_rows; ++j) {
                    if (rows[j] < 0) {
                        z[j] = -INFINITY;
                        continue;
                    }
                    ++n_valid;
                    orc_load_row(K, dtype, (((size_t)b * Hkv + kvh) * T + rows[j]) * d, d, kr);
                    double dot = 0.0;
                    for (int c = 0; c < d; ++c) dot += qv[c] * kr[c];
                    z[j] = scale * dot;
                    if (z[j] > m) m = z[j];
                }
                /* w_j = exp(z_j - m), evaluated once per row; every column sums its terms
                   in ascending j. */
                double l = 0.0;
                for (int c = 0; c < d; ++c) acc[c] = 0.0;
                for (long j = 0; j < n_rows; ++j) {
                    if (rows[j] < 0) continue;
                    const double wj = exp(z[j] - m);
                    l += wj;
                    orc_load_row(Vv, dtype, (((size_t)b * Hkv + kvh) * T + rows[j]) * d, d, kr);
                    for (int c = 0; c < d; ++c) acc[c] += wj * kr[c];
                }
                for (int c = 0; c < d; ++c) out[qrow * d + c] = (n_valid > 0) ? acc[c] / l : 0.0;
                lse[qrow] = (n_valid > 0) ? m + log(l) : -INFINITY;
                if (logits != NULL)
                    for (long j = 0; j < n_rows; ++j) logits[qrow * n_rows + j] = z[j];
                free(qv);
                free(kr);
                free(acc);
                free(z);
                free(rows);
            }
    return bad ? ORC_BAD_INDEX : ORC_OK;
}

/*
 * Verify attention with the draft tokens' window-bounded ring.  Adaptive DHiSparse (news
 * page), "Metodologia e Eficiencia de Carga": the verify queries share the fetch of the
 * selected history rows, and the draft tokens' K/V live in a ring bounded by a window.
 * Reading taken: the ring holds W slots per (b, kvh); ring_pos[b,s] is the token position
 * slot s holds (-1 = empty); query token v of sequence b sits at position qpos[b,v].  Query
 * row (b,v,h) attends the selected history rows (as oracle_gather_attend) and every ring
 * slot s with 0 <= ring_pos[b,s] <= qpos[b,v] (causal among the drafts; the window bound
 * is the ring's size).  List order: the n_idx*block history rows, then the W slots;
 * logits [B,V,Hq,n_idx*block + W] with -inf where a row takes no part.
 */
int oracle_gather_attend_ring(const void* q, const void* K, const void* Vv, int dtype, const int32_t* idx, int B,
                              int V, int Hq, int Hkv, int d, int T, int n_idx, int block, double scale,
                              const void* ring_k, const void* ring_v, const int32_t* ring_pos,
                              const int32_t* qpos, int W, double* out, double* lse, double* logits) {
    if (Hkv < 1 || Hq % Hkv != 0 || d < 1 || block < 1 || n_idx < 0 || W < 0) return ORC_BAD_ARG;
    if (idx == NULL && n_idx * block != T) return ORC_BAD_ARG;
    const int G = Hq / Hkv;
    const long n_rows = (long)n_idx * block, n_all = n_rows + W;
    int bad = 0;
#pragma omp parallel for collapse(3) schedule(dynamic) reduction(| : bad)
    for (int b = 0; b < B; ++b)
        for (int v = 0; v < V; ++v)
            for (int h = 0; h < Hq; ++h) {
                const int kvh = h / G;
                const size_t qrow = (((size_t)b * V + v) * Hq + h);
                double* qv = (double*)malloc(sizeof(double) * (size_t)d);
                double* kr = (double*)malloc(sizeof(double) * (size_t)d);
                double* acc = (double*)malloc(sizeof(double) * (size_t)d);
                double* z = (double*)malloc(sizeof(double) * (size_t)(n_all > 0 ? n_all : 1));
                orc_load_row(q, dtype, qrow * d, d, qv);
                /* z_j for every list row: history row, or ring slot j - n_rows */
                double m = -INFINITY;
                long n_valid = 0;
                for (long j = 0; j < n_all; ++j) {
                    z[j] = -INFINITY;
                    if (j < n_rows) {
                        long row = j;
                        if (idx != NULL) {
                            const long sel = idx[((size_t)b * Hkv + kvh) * n_idx + j / block];
                            if (sel == -1) continue;
                            row = sel * block + j % block;
                            if (sel < 0 || row >= T) {
                                bad = 1;
                                continue;
                            }
                        }
                        orc_load_row(K, dtype, (((size_t)b * Hkv + kvh) * T + row) * d, d, kr);
                    } else {
                        const long slot = j - n_rows;
                        const long tpos = ring_pos[(size_t)b * W + slot];
                        if (tpos < 0 || tpos > qpos[(size_t)b * V + v]) continue;
                        orc_load_row(ring_k, dtype, (((size_t)b * Hkv + kvh) * W + slot) * d, d, kr);
                    }
                    double dot = 0.0;
                    for (int c = 0; c < d; ++c) dot += qv[c] * kr[c];
                    z[j] = scale * dot;
                    if (z[j] > m) m = z[j];
                    ++n_valid;
                }
                double l = 0.0;
                for (int c = 0; c < d; ++c) acc[c] = 0.0;
                for (long j = 0; j < n_all; ++j) {
                    if (z[j] == -INFINITY) continue;
                    const double wj = exp(z[j] - m);
                    l += wj;
                    if (j < n_rows) {
                        const long row = idx != NULL ? (long)idx[((size_t)b * Hkv + kvh) * n_idx + j / block] * block +
                                                           j % block
                                                     : j;
                        orc_load_row(Vv, dtype, (((size_t)b * Hkv + kvh) * T + row) * d, d, kr);
                    } else {
                        orc_load_row(ring_v, dtype, (((size_t)b * Hkv + kvh) * W + (j - n_rows)) * d, d, kr);
                    }
                    for (int c = 0; c < d; ++c) acc[c] += wj * kr[c];
                }
                for (int c = 0; c < d; ++c) out[qrow * d + c] = (n_valid > 0) ? acc[c] / l : 0.0;
                lse[qrow] = (n_valid > 0) ? m + log(l) : -INFINITY;
                if (logits != NULL)
                    for (long j = 0; j < n_all; ++j) logits[qrow * n_all + j] = z[j];
                free(qv);
                free(kr);
                free(acc);
                free(z);
            }
    return bad ? ORC_BAD_INDEX : ORC_OK;
}

/*
 * Step 4 -- cumulative attention-importance score.  [HBM] Metodologia 2, the equation
 *   s_i(t) = s_i(t-1) + (1/|L|) sum over layers l of (1/H) sum over heads h of alpha_{l,h}(t)[i].
 * One call adds one layer's term with weight = 1/(|L| * H):
 *   alpha_{v,h}[j] = exp(logits[b,v,h,j] - lse[b,v,h])   (softmax weight of selected row j)
 *   s[b, rows_j] += weight * alpha_{v,h}[j]   for every v, h and selected row j
 * where rows_j expands idx exactly as in step 3 (rows not selected, and the rows of empty
 * slots -1, receive nothing).
 * With V > 1 verify tokens, every query token's weights are summed (reading: each
 * query token is one decode step's worth of attention).
 * Layouts: logits [B,V,Hq,n_idx*block], lse [B,V,Hq], idx [B,Hkv,n_idx] (NULL: dense),
 * s [B,T] (accumulated in place).
 */
int oracle_score_accumulate(const double* logits, const double* lse, const int32_t* idx, int B,
                            int V, int Hq, int Hkv, int n_idx, int block, int T, double weight,
                            double* s) {
    if (Hkv < 1 || Hq % Hkv != 0 || block < 1 || n_idx < 0) return ORC_BAD_ARG;
    if (idx == NULL && n_idx * block != T) return ORC_BAD_ARG;
    const int G = Hq / Hkv;
    const long n_rows = (long)n_idx * block;
    int bad = 0;
#pragma omp parallel for schedule(static) reduction(| : bad)
    for (int b = 0; b < B; ++b)
        for (int v = 0; v < V; ++v)
            for (int h = 0; h < Hq; ++h) {
                const int kvh = h / G;
                const size_t qrow = (((size_t)b * V + v) * Hq + h);
                for (long j = 0; j < n_rows; ++j) {
                    long row = j;
                    if (idx != NULL) {
                        const long sel = idx[((size_t)b * Hkv + kvh) * n_idx + j / block];
                        if (sel == -1) continue;
                        row = sel * block + j % block;
                    }
                    if (row < 0 || row >= T) {
                        bad = 1;
                        continue;
                    }
                    double alpha = exp(logits[qrow * n_rows + j] - lse[qrow]);
                    s[(size_t)b * T + row] += weight * alpha;
                }
            }
    return bad ? ORC_BAD_INDEX : ORC_OK;
}

/*
 * Step 2' -- block scores on overlapping compression windows.  [SparDA] "Estrategia de
 * Treinamento": the inference block grid is a compression window of `kernel` tokens moved by
 * `stride` (32, 16), and finer scores are max-pooled onto that grid.  Reading taken: the
 * score of window n is the maximum of the token scores it covers,
 *   w[r, n] = max over t in [n*stride, min(n*stride + kernel, N)) of scores[r, t],
 * for n = 0 .. NW-1 with NW = 1 + ceil((N - kernel) / stride) windows (one clipped window
 * when N < kernel; none when N = 0).  scores [rows, N] -> w [rows, NW].
 */
int oracle_window_count(int N, int kernel, int stride) {
    if (N <= 0) return 0;
    if (N <= kernel) return 1;
    return 1 + (N - kernel + stride - 1) / stride;
}

int oracle_window_max(const double* scores, int rows, int N, int kernel, int stride, double* w) {
    if (rows < 0 || N < 0 || kernel < 1 || stride < 1) return ORC_BAD_ARG;
    const int NW = oracle_window_count(N, kernel, stride);
    for (int r = 0; r < rows; ++r)
        for (int n = 0; n < NW; ++n) {
            const long t0 = (long)n * stride;
            const long t1 = t0 + kernel < N ? t0 + kernel : N;
            double m = -INFINITY;
            for (long t = t0; t < t1; ++t)
                if (scores[(size_t)r * N + t] > m) m = scores[(size_t)r * N + t];
            w[(size_t)r * NW + n] = m;
        }
    return ORC_OK;
}

/*
 * Step 2'' -- the tokens of the selected windows.  Windows overlap, so a token may lie in
 * two selected windows; attention must see it once.  With kernel a multiple of stride and
 * N a multiple of stride, the tokens are whole segments of `stride` tokens: window n covers
 * segments n .. n + kernel/stride - 1 (those below N/stride).  Per row the union of the
 * selected windows' segments, ascending, padded to max_segs entries with -1 (empty slots).
 * widx [rows, k] window indices -> segs [rows, max_segs]; max_segs >= k * kernel/stride.
 */
int oracle_window_union(const int32_t* widx, int rows, int k, int N, int kernel, int stride, int32_t* segs,
                        int max_segs) {
    if (rows < 0 || k < 0 || N < 0 || kernel < 1 || stride < 1) return ORC_BAD_ARG;
    if (kernel % stride != 0 || N % stride != 0) return ORC_BAD_ARG;
    const int per = kernel / stride, NS = N / stride, NW = oracle_window_count(N, kernel, stride);
    if ((long)max_segs < (long)k * per) return ORC_BAD_ARG;
    unsigned char* in = (unsigned char*)malloc((size_t)(NS > 0 ? NS : 1));
    int bad = 0;
    for (int r = 0; r < rows; ++r) {
        memset(in, 0, (size_t)(NS > 0 ? NS : 1));
        for (int j = 0; j < k; ++j) {
            const int n = widx[(size_t)r * k + j];
            if (n < 0 || n >= NW) {
                bad = 1;
                continue;
            }
            for (int q = 0; q < per; ++q)
                if (n + q < NS) in[n + q] = 1;
        }
        int at = 0;
        for (int g = 0; g < NS; ++g)
            if (in[g]) segs[(size_t)r * max_segs + at++] = g;
        for (; at < max_segs; ++at) segs[(size_t)r * max_segs + at] = -1;
    }
    free(in);
    return bad ? ORC_BAD_INDEX : ORC_OK;
}

/*
 * Step 5 -- four-tier classification.  [HBM] Metodologia 1: T0 (HBM) holds the protected
 * tokens (prompt, attention sinks, recent window) and the highest-importance tokens; T1
 * (DDR) the medium ones; T2 (8-bit) the low ones; T3 (evicted) only the lowest tail.
 * Metodologia 4: re-run every Delta = 64 decode steps (the caller's schedule).
 *
 * Per sequence b: order = protected positions (t < n_sink or t >= T - n_recent) in index
 * order, then the others by (s descending, index ascending).  With c_m = floor(f_m * T)
 * for the cumulative fractions f = cum_frac[0..2]:
 *   rank < c_0 -> T0,  c_0 <= rank < c_1 -> T1,  c_1 <= rank < c_2 -> T2,  else T3,
 * and protected positions are T0 whatever their rank.
 * s [B,T] -> tier [B,T] (0..3), counts [B,4].
 */
int oracle_tier_classify(const double* s, int B, int T, const double cum_frac[3], int n_sink,
                         int n_recent, uint8_t* tier, int32_t* counts) {
    if (T < 0 || n_sink < 0 || n_recent < 0) return ORC_BAD_ARG;
    for (int m = 0; m < 3; ++m) {
        if (!(cum_frac[m] >= 0.0 && cum_frac[m] <= 1.0)) return ORC_BAD_ARG;
        if (m > 0 && cum_frac[m] < cum_frac[m - 1]) return ORC_BAD_ARG;
    }
    long c[3];
    for (int m = 0; m < 3; ++m) c[m] = (long)floor(cum_frac[m] * (double)T);
#pragma omp parallel for schedule(dynamic)
    for (int b = 0; b < B; ++b) {
        orc_pair* p = (orc_pair*)malloc(sizeof(orc_pair) * (size_t)(T > 0 ? T : 1));
        int n_prot = 0, n_free = 0;
        for (int t = 0; t < T; ++t)
            if (t < n_sink || t >= T - n_recent) n_prot++;
        for (int t = 0; t < T; ++t) {
            int prot = (t < n_sink || t >= T - n_recent);
            if (!prot) {
                p[n_free].s = s[(size_t)b * T + t];
                p[n_free].i = t;
                n_free++;
            }
        }
        qsort(p, (size_t)n_free, sizeof(orc_pair), orc_pair_cmp);
        for (int m = 0; m < 4; ++m) counts[(size_t)b * 4 + m] = 0;
        for (int t = 0; t < T; ++t)
            if (t < n_sink || t >= T - n_recent) {
                tier[(size_t)b * T + t] = 0;
                counts[(size_t)b * 4 + 0]++;
            }
        for (int r = 0; r < n_free; ++r) {
            long rank = (long)n_prot + r;
            int tr = (rank < c[0]) ? 0 : (rank < c[1]) ? 1 : (rank < c[2]) ? 2 : 3;
            tier[(size_t)b * T + p[r].i] = (uint8_t)tr;
            counts[(size_t)b * 4 + tr]++;
        }
        free(p);
    }
    return ORC_OK;
}

/*
 * Step 6 -- 8-bit storage of T2 rows.  [HBM] Metodologia 1 (T2 stores low-importance
 * tokens at reduced precision, "e.g. 8-bit") and "Sensibilidade a Precisao".  The pages
 * give no scheme; the reading taken is symmetric per-row absmax:
 *   a = max_j |x_j|;  a == 0 -> scale = 0 and every code 0;
 *   else scale = a / 127 and code_j = clamp(round_half_even(x_j * (127 / a)), -127, 127).
 * The code is an integer decided by a floating-point product, so this step runs in fp32
 * (each division and the product one correctly rounded fp32 operation), the precision
 * the GPU kernel decides it in.  Only rows whose tier is 2 are written.
 * Layouts: x [B,Hkv,T,d]; tier [B,T]; codes [B,Hkv,T,d]; scales [B,Hkv,T].
 */
int oracle_quantize_rows_int8(const void* x, int dtype, const uint8_t* tier, int B, int Hkv,
                              int T, int d, int8_t* codes, float* scales) {
    if (B < 0 || Hkv < 0 || T < 0 || d < 1) return ORC_BAD_ARG;
#pragma omp parallel for collapse(2) schedule(static)
    for (int b = 0; b < B; ++b)
        for (int h = 0; h < Hkv; ++h)
            for (int t = 0; t < T; ++t) {
                if (tier[(size_t)b * T + t] != 2) continue;
                const size_t row = ((size_t)b * Hkv + h) * T + t;
                volatile float a = 0.0f;
                for (int j = 0; j < d; ++j) {
                    float xj = (float)orc_elem(x, dtype, row * d + j);
                    float mag = fabsf(xj);
                    if (mag > a) a = mag;
                }
                if (a == 0.0f) {
                    scales[row] = 0.0f;
                    for (int j = 0; j < d; ++j) codes[row * d + j] = 0;
                    continue;
                }
                volatile float scale = a / 127.0f;
                volatile float inv = 127.0f / a;
                scales[row] = scale;
                for (int j = 0; j < d; ++j) {
                    float xj = (float)orc_elem(x, dtype, row * d + j);
                    volatile float y = xj * inv;
                    float r = rintf(y);
                    if (r > 127.0f) r = 127.0f;
                    if (r < -127.0f) r = -127.0f;
                    codes[row * d + j] = (int8_t)r;
                }
            }
    return ORC_OK;
}
