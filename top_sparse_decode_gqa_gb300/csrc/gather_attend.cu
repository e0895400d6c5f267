// gather_attend.cu -- exact softmax attention over only the selected K/V rows.
//
// "Esparsidade de Contexto no Tempo de Inferencia" (gist.science summary), sec. 2: sparse
// decode kernels with irregular per-token selection; sec. 3C: memory traffic falls from
// O(N*d) to O(k*d).  Adaptive DHiSparse (news page), "A Inovacao" / "Metodologia": the
// history lives in host memory, only selected rows are fetched, fused with attention,
// and queries share the fetch of missing rows.  "Nem Todos os Pensamentos Necessitam de
// HBM" (gist.science summary), Metodologia 3: a row fetched from host memory at full
// precision contributes exactly the terms it would from HBM.
//
// Grid (split, kvh, b).  One CTA owns a contiguous range of the (b, kvh) selection list and
// computes all R = G*V query rows of the group over it, so every selected row is read from
// memory once and shared by the whole GQA group / verify batch.  Rows are staged 64 at a
// time into shared memory with 16-byte cp.async (double-buffered), from the HBM pool or,
// for slot -1, from pinned host memory through the device mapping; the staged bytes are
// the same either way, so the result does not depend on the source.  fp32 online softmax
// in base 2 per query row; with several splits each CTA writes (m, l, o) partials and a
// merge kernel combines them in split order (deterministic).
#include <algorithm>

#include "attend_mma.cuh"
#include "sd_common.cuh"
#include "sd_host.h"

namespace sd {
namespace {

constexpr int kAttThreads = 128;
constexpr int kCH = 64;             // rows per staged chunk
constexpr int kMaxSplitRows = 448;  // rows whose sources a CTA resolves up front
constexpr float kLn2 = 0.69314718055994530942f;
constexpr float kLog2e = 1.44269504088896340736f;

struct AttendParams {
    const void* q;
    const uint8_t* kc;
    const uint8_t* vc;
    const uint8_t* kh;
    const uint8_t* vh;
    const int32_t* slot_map;
    const int32_t* idx;
    int B, V, Hq, Hkv, G, R, T, pool_rows, n_idx, block, n_rows, rows_per_split, splits;
    int kv_heads, heads_per_kv;  // KV heads of the cache; groups per KV head (per-head mode: G)
    int dtype;
    int resolve;  // 1: sources resolved up front (idx or slot_map given)
    int staged;   // 1: kh/vh are the HBM stage [groups, n_hist, d], host rows by list position
    int slot_per_head;  // 1: slot_map is [B, kv_heads, T] (residency per (b, KV head))
    int n_hist;   // selected (history) list rows; list rows [n_hist, n_rows) are the draft ring's slots
    int ring_w;   // draft ring slots (0: none)
    const uint8_t* rk;        // draft ring [B, kv_heads, ring_w, d]
    const uint8_t* rv;
    const int32_t* ring_pos;  // [B, ring_w] token position per slot, -1 empty
    const int32_t* qpos;      // [B, V] position of each query token
    float scale_log2;
    float* out;
    float* lse;
    float* logits;
    int32_t* err;
    float* ws_o;
    float* ws_m;
    float* ws_l;
    const uint8_t* tier;  // [B, T] or null: 3 skipped, 2 read from the int8 rows
    const int8_t* ki8;    // [B, kv_heads, T, d] int8 codes
    const int8_t* vi8;
    const float* ksc;     // [B, kv_heads, T] scales
    const float* vsc;
};

template <typename ST, int D, int RP>
struct AttLayout {
    static constexpr int kPadE = 16 / (int)sizeof(ST);  // 16-byte row pad for K
    static constexpr int kKRow = (D + kPadE) * (int)sizeof(ST);
    static constexpr int kVRow = D * (int)sizeof(ST);
    static constexpr int kPRow = RP + 4;  // floats per p row
    static constexpr int kSRow = kCH + 4;  // floats per s row
    static constexpr int oQ = 0;
    static constexpr int oK = oQ + RP * D * 4;
    static constexpr int oV = oK + 2 * kCH * kKRow;
    static constexpr int oP = oV + 2 * kCH * kVRow;
    static constexpr int oS = oP + kCH * kPRow * 4;
    static constexpr int oSrc = oS + RP * kSRow * 4;
    static constexpr int oAlpha = oSrc + kMaxSplitRows * 4;
    static constexpr int oM = oAlpha + RP * 4;
    static constexpr int oL = oM + RP * 4;
    static constexpr int oFlag = oL + RP * 4;
    static constexpr int kBytes = oFlag + 16;
    static_assert(oV % 16 == 0 && oP % 16 == 0 && oS % 16 == 0 && oSrc % 16 == 0, "align");
    static_assert((RP == 4 ? 4 : 1) * RP * D * 4 <= 2 * kCH * kKRow, "reduction buffer must fit in K");
};

// Shared-memory CTAs per SM for a layout (228 KB per SM, 1 KB reserved per CTA), at most 3.
int att_ctas_per_sm(int bytes) {
    const int per = 233472 / (bytes + 1024);
    return per < 1 ? 1 : (per > 3 ? 3 : per);
}

constexpr int kMergeThreads = 128;
constexpr int kMergeWarps = kMergeThreads / 32;

// Block-wide max / sum of one value per thread (kMergeThreads), the same in every thread.
SD_DEVINL float merge_block_max(float v, float* red) {
    for (int o = 16; o > 0; o >>= 1) v = fmaxf(v, __shfl_xor_sync(0xffffffffu, v, o));
    __syncthreads();
    if ((threadIdx.x & 31) == 0) red[threadIdx.x >> 5] = v;
    __syncthreads();
    float r = red[0];
    for (int w = 1; w < kMergeWarps; ++w) r = fmaxf(r, red[w]);
    return r;
}
SD_DEVINL float merge_block_sum(float v, float* red) {
    for (int o = 16; o > 0; o >>= 1) v += __shfl_xor_sync(0xffffffffu, v, o);
    __syncthreads();
    if ((threadIdx.x & 31) == 0) red[threadIdx.x >> 5] = v;
    __syncthreads();
    float r = red[0];
    for (int w = 1; w < kMergeWarps; ++w) r += red[w];
    return r;
}

// The split-K merge, after every split wrote its (m, l, o) partial: grid (groups, R), one
// CTA per (group, query row).  M = max over the splits of m, L = sum of l * 2^(m - M), and
// o = sum over the splits of o_s * 2^(m_s - M) / L, each split's terms in a fixed order
// (warp w takes splits w, w + 4, ...; the warps' sums are added in warp order), so the
// result is the same on every run.  lse = (M + log2 L) ln 2.
template <int D>
__global__ void __launch_bounds__(kMergeThreads, 8) attend_merge_kernel(const AttendParams p, int RP) {
    __shared__ float red[kMergeWarps];
    __shared__ __align__(16) float part[kMergeWarps][D];
    pdl_wait();  // every split's partial is written
    pdl_launch_dependents();
    constexpr int CPL = D / 32;  // columns per lane
    const int bk = blockIdx.x, r = blockIdx.y;
    const int b = bk / p.Hkv, kvh = bk % p.Hkv;
    const int tid = threadIdx.x, lane = tid & 31, warp = tid >> 5;
    const int S = p.splits;
    const size_t base = (size_t)bk * S * RP + r;  // partial row of split s: base + s * RP
    // (m, l) of every split in one pass: this thread's running maximum and sum, then the
    // block's maximum and the sums rescaled to it
    float m = -INFINITY, l = 0.f;
    for (int s = tid; s < S; s += kMergeThreads) {
        const float ms = __ldcg(p.ws_m + base + (size_t)s * RP);
        const float ls = __ldcg(p.ws_l + base + (size_t)s * RP);
        if (ms == -INFINITY) continue;
        if (ms > m) {
            l = (m == -INFINITY) ? ls : fmaf(l, exp2f(m - ms), ls);
            m = ms;
        } else {
            l = fmaf(ls, exp2f(ms - m), l);
        }
    }
    const float M = merge_block_max(m, red);
    const float L = merge_block_sum(m == -INFINITY ? 0.f : l * exp2f(m - M), red);
    float o[CPL];
#pragma unroll
    for (int c = 0; c < CPL; ++c) o[c] = 0.f;
    constexpr int U = 8;  // splits a warp requests before using any (8 CTAs per SM fit: one wave)
    for (int s0 = warp; s0 < S; s0 += U * kMergeWarps) {
        float ms[U], x[U][CPL];
#pragma unroll
        for (int u = 0; u < U; ++u) {
            const int s = s0 + u * kMergeWarps;
            ms[u] = s < S ? __ldcg(p.ws_m + base + (size_t)s * RP) : -INFINITY;
            const float* orow = p.ws_o + (base + (size_t)(s < S ? s : 0) * RP) * D + lane * CPL;
#pragma unroll
            for (int c = 0; c < CPL; ++c) x[u][c] = s < S ? __ldcg(orow + c) : 0.f;
        }
#pragma unroll
        for (int u = 0; u < U; ++u) {
            const float w = (L > 0.f && ms[u] != -INFINITY) ? exp2f(ms[u] - M) / L : 0.f;
#pragma unroll
            for (int c = 0; c < CPL; ++c) o[c] = fmaf(w, x[u][c], o[c]);
        }
    }
#pragma unroll
    for (int c = 0; c < CPL; ++c) part[warp][lane * CPL + c] = o[c];
    __syncthreads();
    const int v = r / p.G, g = r % p.G;
    const size_t qrow = ((size_t)b * p.V + v) * p.Hq + kvh * p.G + g;
    for (int col = tid; col < D; col += kMergeThreads) {
        float x = part[0][col];
        for (int w = 1; w < kMergeWarps; ++w) x += part[w][col];
        p.out[qrow * D + col] = x;
    }
    if (tid == 0) p.lse[qrow] = L > 0.f ? (M + log2f(L)) * kLn2 : -INFINITY;
}

template <typename ST, int D, int RP>
__global__ void __launch_bounds__(kAttThreads) attend_kernel(const AttendParams p) {
    using L = AttLayout<ST, D, RP>;
    using U = Unpack16<ST>;
    constexpr int EPC = U::kElems;               // elements per 16 bytes
    constexpr int PPR = L::kVRow / 16;           // 16-byte pieces per row
    constexpr int CPL = D / 32;                  // PV columns per lane
    constexpr bool kKeySplit = (RP == 4);        // PV: warps split keys (else query rows)
    constexpr int QW = kKeySplit ? RP : RP / 4;  // PV query rows per warp

    extern __shared__ __align__(128) uint8_t sm[];
    float* qs = reinterpret_cast<float*>(sm + L::oQ);
    float* ps = reinterpret_cast<float*>(sm + L::oP);
    float* ss = reinterpret_cast<float*>(sm + L::oS);
    int32_t* src = reinterpret_cast<int32_t*>(sm + L::oSrc);  // per row of the split
    float* alpha_s = reinterpret_cast<float*>(sm + L::oAlpha);
    float* m_s = reinterpret_cast<float*>(sm + L::oM);
    float* l_s = reinterpret_cast<float*>(sm + L::oL);

    const int tid = threadIdx.x, lane = tid & 31, warp = tid >> 5;
    const int split = blockIdx.x, kvh = blockIdx.y, b = blockIdx.z;
    const int bk = b * p.Hkv + kvh;
    const int kvsrc = b * p.kv_heads + kvh / p.heads_per_kv;  // the (b, KV head) slab the rows come from
    // host rows: the (b, KV head) slab of the host cache, or this group's rows of the stage
    const size_t host_row0 = p.staged ? (size_t)bk * p.n_hist : (size_t)kvsrc * p.T;
    const size_t esz = sizeof(ST);

    pdl_wait();  // everything below may read what the preceding kernel wrote

    // ---- query rows r = v*G + g (head h = kvh*G + g), pre-scaled by scale*log2(e)
    for (int e = tid; e < RP * D; e += kAttThreads) {
        const int r = e / D, c = e % D;
        float x = 0.f;
        if (r < p.R) {
            const int v = r / p.G, g = r % p.G;
            x = load_elem(p.q, p.dtype, (((size_t)b * p.V + v) * p.Hq + kvh * p.G + g) * D + c) *
                p.scale_log2;
        }
        qs[e] = x;
    }

    const int j0 = split * p.rows_per_split;
    const int j1 = min(p.n_rows, j0 + p.rows_per_split);
    const int nrows = max(0, j1 - j0);
    const int nch = (nrows + kCH - 1) / kCH;

    // ---- resolve every row's source once: >= 0 device row (pool slot, or cache
    // position without a slot map), < 0 host row -1 - position, kNoRow skipped
    auto resolve_row = [&](int jg) -> int32_t {
        if (jg >= p.n_hist) {  // draft ring slot: skipped when empty
            const int slot = jg - p.n_hist;
            return p.ring_pos[(size_t)b * p.ring_w + slot] < 0 ? kNoRow : kRingBase + slot;
        }
        long pos = jg;
        if (p.idx != nullptr) {
            const long sel = p.idx[(size_t)bk * p.n_idx + jg / p.block];
            if (sel == -1) return kNoRow;  // empty slot
            pos = sel * p.block + jg % p.block;
            if (sel < 0 || pos >= p.T) {
                report(p.err, SD_DEVERR_INDEX);
                return kNoRow;
            }
        }
        if (p.slot_map == nullptr) return (int32_t)pos;
        const int slot = p.slot_map[(size_t)(p.slot_per_head ? kvsrc : b) * p.T + pos];
        if (slot >= 0 && slot < p.pool_rows) return slot;
        if (slot == -1) return (int32_t)(-1 - (p.staged ? (long)jg : pos));
        report(p.err, SD_DEVERR_SLOT);
        return kNoRow;
    };
    if (p.resolve)
        for (int j = tid; j < nrows; j += kAttThreads) src[j] = resolve_row(j0 + j);
    __syncthreads();
    auto row_code = [&](int j) -> int32_t { return p.resolve ? src[j] : (int32_t)(j0 + j); };
    // a draft-ring row is visible to query row r (token v = r / G) up to its own position
    auto visible = [&](int r, int j) -> bool {
        if (p.ring_w == 0) return true;
        const int32_t code = row_code(j);
        if (code < kRingBase || r >= p.R) return true;
        return p.ring_pos[(size_t)b * p.ring_w + (code - kRingBase)] <= p.qpos[(size_t)b * p.V + r / p.G];
    };

    auto issue = [&](int c, int bf) {
        uint8_t* kdst = sm + L::oK + bf * kCH * L::kKRow;
        uint8_t* vdst = sm + L::oV + bf * kCH * L::kVRow;
        const int rows_here = min(kCH, nrows - c * kCH);
        for (int pc = tid; pc < 2 * kCH * PPR; pc += kAttThreads) {
            const int which = pc / (kCH * PPR);
            const int rem = pc - which * (kCH * PPR);
            const int j = rem / PPR, part = rem % PPR;
            uint8_t* dst = which ? vdst + j * L::kVRow + part * 16 : kdst + j * L::kKRow + part * 16;
            const int32_t code = j < rows_here ? row_code(c * kCH + j) : kNoRow;
            if (code == kNoRow) {
                *reinterpret_cast<uint4*>(dst) = make_uint4(0u, 0u, 0u, 0u);
                continue;
            }
            const uint8_t* base;
            size_t row;
            if (code >= kRingBase) {
                base = which ? p.rv : p.rk;
                row = (size_t)kvsrc * p.ring_w + (code - kRingBase);
            } else if (code >= 0) {
                base = which ? p.vc : p.kc;
                row = (size_t)kvsrc * p.pool_rows + code;
            } else {
                base = which ? p.vh : p.kh;
                row = host_row0 + (size_t)(-1 - (long)code);
            }
            cp_async16(dst, base + row * L::kVRow + part * 16);
        }
        cp_async_commit();
    };

    float m_reg[RP / 4], l_reg[RP / 4];
#pragma unroll
    for (int i = 0; i < RP / 4; ++i) {
        m_reg[i] = -INFINITY;
        l_reg[i] = 0.f;
    }
    float acc[QW][CPL];
#pragma unroll
    for (int i = 0; i < QW; ++i)
#pragma unroll
        for (int c = 0; c < CPL; ++c) acc[i][c] = 0.f;

    if (nch > 0) issue(0, 0);
    if (nch > 1) issue(1, 1);
    for (int c = 0; c < nch; ++c) {
        const int bf = c & 1;
        if (c + 1 < nch)
            cp_async_wait<1>();
        else
            cp_async_wait<0>();
        __syncthreads();

        // ---- QK: thread -> key j, half hf of the query rows
        {
            const int j = tid & (kCH - 1), hf = tid / kCH;
            const uint8_t* krow = sm + L::oK + (bf * kCH + j) * L::kKRow;
            const bool valid = c * kCH + j < nrows && row_code(c * kCH + j) != kNoRow;
            float s[RP / 2];
#pragma unroll
            for (int r = 0; r < RP / 2; ++r) s[r] = 0.f;
#pragma unroll 4
            for (int e0 = 0; e0 < D; e0 += EPC) {
                float x[EPC];
                U::run(lds128(krow + e0 * esz), x);
#pragma unroll
                for (int r = 0; r < RP / 2; ++r) {
                    const float* qr = qs + (hf * (RP / 2) + r) * D + e0;
#pragma unroll
                    for (int e = 0; e < EPC; ++e) s[r] = fmaf(x[e], qr[e], s[r]);
                }
            }
#pragma unroll
            for (int r = 0; r < RP / 2; ++r)
                ss[(hf * (RP / 2) + r) * L::kSRow + j] = valid && visible(hf * (RP / 2) + r, c * kCH + j) ? s[r] : -INFINITY;
        }
        __syncthreads();

        // ---- online softmax (base 2) per query row
#pragma unroll
        for (int i = 0; i < RP / 4; ++i) {
            const int r = warp + 4 * i;
            const float s0 = ss[r * L::kSRow + lane], s1 = ss[r * L::kSRow + lane + 32];
            const float cm = warp_max(fmaxf(s0, s1));
            const float mo = m_reg[i];
            const float mn = fmaxf(mo, cm);
            const float alpha = (mn == -INFINITY) ? 1.f : exp2f(mo - mn);
            const float p0 = (s0 == -INFINITY) ? 0.f : exp2f(s0 - mn);
            const float p1 = (s1 == -INFINITY) ? 0.f : exp2f(s1 - mn);
            l_reg[i] = l_reg[i] * alpha + warp_sum(p0 + p1);
            m_reg[i] = mn;
            ps[lane * L::kPRow + r] = p0;
            ps[(lane + 32) * L::kPRow + r] = p1;
            if (lane == 0) alpha_s[r] = alpha;
            if (p.logits != nullptr && r < p.R) {
                const int v = r / p.G, g = r % p.G;
                float* lrow = p.logits + (((size_t)b * p.V + v) * p.Hq + kvh * p.G + g) * p.n_rows;
                const int jg = j0 + c * kCH + lane;
                if (jg < j1) lrow[jg] = s0 * kLn2;
                if (jg + 32 < j1) lrow[jg + 32] = s1 * kLn2;
            }
        }
        __syncthreads();

        // ---- PV
        {
            const uint8_t* vbuf = sm + L::oV + bf * kCH * L::kVRow;
            const int q0 = kKeySplit ? 0 : warp * QW;
#pragma unroll
            for (int i = 0; i < QW; ++i) {
                const float a = alpha_s[q0 + i];
#pragma unroll
                for (int cc = 0; cc < CPL; ++cc) acc[i][cc] *= a;
            }
            const int jb = kKeySplit ? warp * (kCH / 4) : 0;
            const int je = kKeySplit ? jb + kCH / 4 : kCH;
#pragma unroll 4
            for (int j = jb; j < je; ++j) {
                float vx[CPL];
                const uint8_t* vp = vbuf + j * L::kVRow + lane * CPL * esz;
                if constexpr (sizeof(ST) == 2) {
                    if constexpr (CPL == 4) {
                        const uint2 w = *reinterpret_cast<const uint2*>(vp);
                        vx[0] = bf16lo(w.x); vx[1] = bf16hi(w.x); vx[2] = bf16lo(w.y); vx[3] = bf16hi(w.y);
                    } else {
                        const uint32_t w = *reinterpret_cast<const uint32_t*>(vp);
                        vx[0] = bf16lo(w); vx[1] = bf16hi(w);
                    }
                } else {
#pragma unroll
                    for (int cc = 0; cc < CPL; ++cc) vx[cc] = reinterpret_cast<const float*>(vp)[cc];
                }
                const float* pr = ps + j * L::kPRow + q0;
#pragma unroll
                for (int i = 0; i < QW; ++i) {
                    const float pj = pr[i];
#pragma unroll
                    for (int cc = 0; cc < CPL; ++cc) acc[i][cc] = fmaf(pj, vx[cc], acc[i][cc]);
                }
            }
        }
        __syncthreads();  // buffer bf is refilled next
        if (c + 2 < nch) issue(c + 2, bf);
    }

    // ---- publish m, l; combine the warps' partial sums
#pragma unroll
    for (int i = 0; i < RP / 4; ++i)
        if (lane == 0) {
            m_s[warp + 4 * i] = m_reg[i];
            l_s[warp + 4 * i] = l_reg[i];
        }
    __syncthreads();
    float* red = reinterpret_cast<float*>(sm + L::oK);  // K buffers are free now
    if constexpr (kKeySplit) {
#pragma unroll
        for (int i = 0; i < QW; ++i)
#pragma unroll
            for (int cc = 0; cc < CPL; ++cc) red[(warp * RP + i) * D + lane * CPL + cc] = acc[i][cc];
    } else {
#pragma unroll
        for (int i = 0; i < QW; ++i)
#pragma unroll
            for (int cc = 0; cc < CPL; ++cc) red[(warp * QW + i) * D + lane * CPL + cc] = acc[i][cc];
    }
    __syncthreads();
    for (int e = tid; e < RP * D; e += kAttThreads) {
        const int r = e / D, col = e % D;
        if (r >= p.R) continue;
        float o = red[e];
        if constexpr (kKeySplit) o += red[RP * D + e] + red[2 * RP * D + e] + red[3 * RP * D + e];
        if (p.splits == 1) {
            const int v = r / p.G, g = r % p.G;
            const size_t qrow = ((size_t)b * p.V + v) * p.Hq + kvh * p.G + g;
            const float l = l_s[r];
            p.out[qrow * D + col] = l > 0.f ? o / l : 0.f;
            if (col == 0) p.lse[qrow] = l > 0.f ? (m_s[r] + log2f(l)) * kLn2 : -INFINITY;
        } else {
            const size_t prow = ((size_t)bk * p.splits + split) * RP + r;
            p.ws_o[prow * D + col] = o;
            if (col == 0) {
                p.ws_m[prow] = m_s[r];
                p.ws_l[prow] = l_s[r];
            }
        }
    }
}

// ------------------------------------------------------------------ bf16 path (warp MMA)

template <int D, int RP>
struct MmaLayout {
    using Rows = MmaRows<D>;
    static constexpr int oQ = 0;
    static constexpr int oStage = ((RP * Rows::kRowB + 127) / 128) * 128;
    static constexpr int oSrc = oStage + Rows::kStagesBytes;
    static constexpr int oML = oSrc + kMaxSplitRows * 4;   // [4 warps][RP] m, then l
    static constexpr int oRow = oML + 2 * kMmaWarps * RP * 4;  // [RP] row max, sum; [4][RP] factors
    static constexpr int oFlag = oRow + 6 * RP * 4;
    static constexpr int kBytes = oFlag + 16;
    static_assert(kMmaWarps * RP * D * 4 <= Rows::kStagesBytes, "warp outputs must fit in the stages");
};

// Grid (split, kvh, b), 4 warps.  The split's rows are resolved to their sources up front,
// then attend_mma.cuh's per-warp loop runs over them; the 4 warps' (m, l, O) are combined
// into the CTA's split partial (or, with one split, into out and lse); attend_merge_kernel
// then merges the splits.  RING: the list ends with draft-ring slots, masked per query row.
// I8: positions of tier 3 are skipped and those of tier 2 read from the int8 rows.
template <int D, int RP, bool RING, bool I8 = false>
__global__ void __launch_bounds__(kAttThreads) attend_mma_kernel(const AttendParams p) {
    using L = MmaLayout<D, RP>;
    using Rows = MmaRows<D>;
    constexpr int PPR = D * 2 / 16;  // 16-byte pieces per row
    extern __shared__ __align__(128) uint8_t sm[];
    int32_t* src = reinterpret_cast<int32_t*>(sm + L::oSrc);
    float* mlw = reinterpret_cast<float*>(sm + L::oML);
    float* rowv = reinterpret_cast<float*>(sm + L::oRow);

    const int tid = threadIdx.x, warp = tid >> 5;
    const int split = blockIdx.x, kvh = blockIdx.y, b = blockIdx.z;
    const int bk = b * p.Hkv + kvh;

    pdl_wait();

    // ---- prologue: query rows (cp.async, zero beyond R) and the rows' sources, together
    for (int e = tid; e < RP * PPR; e += kAttThreads) {
        const int r = e / PPR, part = e % PPR;
        uint8_t* dst = sm + L::oQ + r * Rows::kRowB + part * 16;
        if (r < p.R) {
            const int v = r / p.G, gg = r % p.G;
            const uint8_t* qrow = static_cast<const uint8_t*>(p.q) +
                                  ((((size_t)b * p.V + v) * p.Hq + kvh * p.G + gg) * D) * 2;
            cp_async16(dst, qrow + part * 16);
        } else {
            *reinterpret_cast<uint4*>(dst) = make_uint4(0u, 0u, 0u, 0u);
        }
    }
    cp_async_commit();
    const int j0 = split * p.rows_per_split;
    const int j1 = min(p.n_rows, j0 + p.rows_per_split);
    const int nrows = max(0, j1 - j0);
    const int kvsrc = b * p.kv_heads + kvh / p.heads_per_kv;  // the (b, KV head) slab the rows come from
    const int32_t* srow_map = p.slot_map != nullptr ? p.slot_map + (size_t)(p.slot_per_head ? kvsrc : b) * p.T : nullptr;
    if (p.resolve) {
        for (int j = tid; j < nrows; j += kAttThreads) {
            const int jg = j0 + j;
            if (jg >= p.n_hist) {  // draft ring slot: skipped when empty
                const int slot = jg - p.n_hist;
                src[j] = p.ring_pos[(size_t)b * p.ring_w + slot] < 0 ? kNoRow : kRingBase + slot;
                continue;
            }
            long pos = jg;
            int32_t code;
            bool ok = true;
            if (p.idx != nullptr) {
                const long sel = p.idx[(size_t)bk * p.n_idx + jg / p.block];
                pos = sel * p.block + jg % p.block;
                if (sel == -1) {  // empty slot
                    ok = false;
                } else if (sel < 0 || pos >= p.T) {
                    report(p.err, SD_DEVERR_INDEX);
                    ok = false;
                }
            }
            int tr = 0;
            if constexpr (I8) {
                if (ok) tr = p.tier[(size_t)b * p.T + pos];
            }
            if (!ok || tr == 3) {
                code = kNoRow;
            } else if (tr == 2) {
                code = kI8Base + (int32_t)pos;
            } else if (p.slot_map == nullptr) {
                code = (int32_t)pos;
            } else {
                const int slot = srow_map[pos];
                if (slot >= 0 && slot < p.pool_rows) {
                    code = slot;
                } else if (slot == -1) {
                    code = (int32_t)(-1 - (p.staged ? (long)jg : pos));
                } else {
                    report(p.err, SD_DEVERR_SLOT);
                    code = kNoRow;
                }
            }
            src[j] = code;
        }
    }
    cp_async_wait<0>();
    __syncthreads();

    RowSource rs;
    rs.k_pool = p.kc + (size_t)kvsrc * p.pool_rows * (D * 2);
    rs.v_pool = p.vc + (size_t)kvsrc * p.pool_rows * (D * 2);
    const size_t host_row0 = p.staged ? (size_t)bk * p.n_hist : (size_t)kvsrc * p.T;
    rs.k_host = p.kh + host_row0 * (D * 2);
    rs.v_host = p.vh + host_row0 * (D * 2);
    if (p.ring_w > 0) {
        rs.k_ring = p.rk + (size_t)kvsrc * p.ring_w * (D * 2);
        rs.v_ring = p.rv + (size_t)kvsrc * p.ring_w * (D * 2);
    }
    if constexpr (I8) {
        rs.k_i8 = p.ki8 + (size_t)kvsrc * p.T * D;
        rs.v_i8 = p.vi8 + (size_t)kvsrc * p.T * D;
        rs.k_scl = p.ksc + (size_t)kvsrc * p.T;
        rs.v_scl = p.vsc + (size_t)kvsrc * p.T;
    }
    auto row_code = [&](int j) -> int32_t {
        if (p.resolve) return src[j];
        const int32_t pos = j0 + j;
        if constexpr (I8) {  // dense over the cache: the position's tier decides, read as needed
            const uint8_t t = __ldg(p.tier + (size_t)b * p.T + pos);
            return t == 3 ? kNoRow : t == 2 ? kI8Base + pos : pos;
        }
        return pos;
    };
    float* lbase = nullptr;  // logits of query row 0 of this group, at list row j0
    if (p.logits != nullptr) lbase = p.logits + ((size_t)b * p.V * p.Hq + kvh * p.G) * p.n_rows + j0;
    auto logit = [&](int r, int j, float x) {
        if (lbase != nullptr && r < p.R) {
            const int v = r / p.G, gg = r % p.G;
            lbase[((size_t)v * p.Hq + gg) * p.n_rows + j] = x * kLn2;
        }
    };
    // a draft-ring row is visible to query row r (token v = r / G) up to its own position
    auto visible = [&](int r, int j) -> bool {
        if constexpr (!RING) {
            return true;
        } else {
            const int32_t code = row_code(j);
            if (code < kRingBase || r >= p.R) return true;
            return p.ring_pos[(size_t)b * p.ring_w + (code - kRingBase)] <= p.qpos[(size_t)b * p.V + r / p.G];
        }
    };
    WarpAcc<D, RP> acc;
    acc.init();
    if constexpr (I8) {
        mma_attend_warp<D, RP>(acc, sm + L::oStage + warp * Rows::kWarpBytes, smem_addr(sm + L::oQ), warp, nrows,
                               p.R, rs, p.scale_log2, row_code, logit, visible, Int8Rows{});
    } else {
        mma_attend_warp<D, RP>(acc, sm + L::oStage + warp * Rows::kWarpBytes, smem_addr(sm + L::oQ), warp, nrows,
                               p.R, rs, p.scale_log2, row_code, logit, visible);
    }

    float* ow = reinterpret_cast<float*>(sm + L::oStage);  // [4][RP][D]
    mma_combine_warps<D, RP>(acc, mlw, rowv, ow, p.R);
    const float* rowM = rowv;
    const float* rowL = rowv + RP;
    for (int e = tid; e < p.R * (D / 4); e += kAttThreads) {
        const int r = e / (D / 4), col = (e % (D / 4)) * 4;
        const float Ls = rowL[r];
        const float4 o = mma_cta_row4<D, RP>(ow, r, col);
        if (p.splits == 1) {
            const int v = r / p.G, gg = r % p.G;
            const size_t qrow = ((size_t)b * p.V + v) * p.Hq + kvh * p.G + gg;
            const float inv = Ls > 0.f ? 1.f / Ls : 0.f;
            *reinterpret_cast<float4*>(p.out + qrow * D + col) = make_float4(o.x * inv, o.y * inv, o.z * inv, o.w * inv);
            if (col == 0) p.lse[qrow] = Ls > 0.f ? (rowM[r] + log2f(Ls)) * kLn2 : -INFINITY;
        } else {
            const size_t prow = ((size_t)bk * p.splits + split) * RP + r;
            *reinterpret_cast<float4*>(p.ws_o + prow * D + col) = o;
            if (col == 0) {
                p.ws_m[prow] = rowM[r];
                p.ws_l[prow] = Ls;
            }
        }
    }
}

int padded_rows(int R) { return R <= 4 ? 4 : R <= 8 ? 8 : R <= 16 ? 16 : R <= 32 ? 32 : -1; }

// Query rows per CTA as the kernel lays them out: 16 or 32 on the bf16 (tensor-core) path,
// 4 / 8 / 16 / 32 on the fp32 path; -1 if G*V is beyond 32.
int kernel_rows(int dtype, int R) {
    if (R > 32 || R < 1) return -1;
    if (dtype == SD_BF16) return R <= 16 ? 16 : 32;
    return padded_rows(R);
}

int layout_bytes(int dtype, int d, int RP) {
    if (dtype == SD_BF16) {
        if (d == 128) return RP <= 16 ? MmaLayout<128, 16>::kBytes : MmaLayout<128, 32>::kBytes;
        return RP <= 16 ? MmaLayout<64, 16>::kBytes : MmaLayout<64, 32>::kBytes;
    }
    switch ((d == 128 ? 0 : 4) + (RP <= 4 ? 0 : RP <= 8 ? 1 : RP <= 16 ? 2 : 3)) {
        case 0: return AttLayout<float, 128, 4>::kBytes;
        case 1: return AttLayout<float, 128, 8>::kBytes;
        case 2: return AttLayout<float, 128, 16>::kBytes;
        case 3: return AttLayout<float, 128, 32>::kBytes;
        case 4: return AttLayout<float, 64, 4>::kBytes;
        case 5: return AttLayout<float, 64, 8>::kBytes;
        case 6: return AttLayout<float, 64, 16>::kBytes;
        default: return AttLayout<float, 64, 32>::kBytes;
    }
}

struct SplitPlan {
    int splits, rows_per_split, RP;
    size_t ws_bytes;
};

size_t align16(size_t x) { return (x + 15) & ~size_t(15); }

// Split-K plan: one wave of CTAs over the GPU (unless the caller asks for a split count),
// at least one chunk per split, and at most kMaxSplitRows rows per split when the rows'
// sources are resolved up front.  Workspace: partials o [bk][split][RP][d], then m, l.
SplitPlan plan_splits(const sd_attend_args* a) {
    SplitPlan sp{};
    const long n_rows = (long)a->n_idx * a->block + a->ring_w;
    const long bk = (long)a->B * (a->per_head ? a->Hq : a->Hkv);
    sp.RP = kernel_rows(a->dtype, a->per_head ? a->V : (a->Hkv > 0 ? (a->Hq / a->Hkv) * a->V : 0));
    const long chunks = (n_rows + kCH - 1) / kCH;
    const bool resolve = a->idx != nullptr || a->slot_map != nullptr || a->ring_w > 0;
    const bool tiled = dense_tma_eligible(a);
    long splits;
    if (a->splits > 0) {
        splits = a->splits;
    } else {
        // one wave of the kernel that will run (the tiled path has its own occupancy)
        const int per_sm = tiled ? dense_tma_ctas_per_sm(a) : att_ctas_per_sm(layout_bytes(a->dtype, a->d, sp.RP));
        const long slots = (long)num_sms() * per_sm;
        splits = bk > 0 ? slots / bk : 1;
    }
    splits = std::max(1L, std::min(splits, std::max(1L, chunks)));
    long rps = n_rows > 0 ? (n_rows + splits - 1) / splits : 1;
    // rows whose sources a CTA resolves up front: the row loop's list, or the tiled path's
    // table of 16-row sub-tiles
    const long max_rps = tiled ? dense_tma_max_split_rows() : kMaxSplitRows;
    if (resolve && rps > max_rps) rps = max_rps;
    splits = n_rows > 0 ? (n_rows + rps - 1) / rps : 1;
    sp.splits = (int)splits;
    sp.rows_per_split = (int)rps;
    if (splits > 1) {
        const size_t np = (size_t)bk * splits * sp.RP;
        sp.ws_bytes = align16(np * (a->d + 2) * sizeof(float));
    }
    return sp;
}

template <typename ST, int D, int RP>
sd_status launch_attend(const AttendParams& p, cudaStream_t st) {
    using L = AttLayout<ST, D, RP>;
    auto kern = attend_kernel<ST, D, RP>;
    SD_CUDA_CHECK(cudaFuncSetAttribute(kern, cudaFuncAttributeMaxDynamicSharedMemorySize, L::kBytes),
                  "sd_gather_attend: cudaFuncSetAttribute");
    SD_CUDA_CHECK(launch_pdl(kern, dim3(p.splits, p.Hkv, p.B), dim3(kAttThreads), L::kBytes, st, p),
                  "sd_gather_attend: launch");
    return launch_status("sd_gather_attend");
}

template <int D, int RP>
sd_status launch_attend_mma(const AttendParams& p, cudaStream_t st) {
    if constexpr (D == 128) {
        if (p.tier != nullptr) {  // int8 rows (validated: no ring)
            using L = MmaLayout<D, RP>;
            auto kern = attend_mma_kernel<D, RP, false, true>;
            SD_CUDA_CHECK(cudaFuncSetAttribute(kern, cudaFuncAttributeMaxDynamicSharedMemorySize, L::kBytes),
                          "sd_gather_attend: cudaFuncSetAttribute");
            SD_CUDA_CHECK(launch_pdl(kern, dim3(p.splits, p.Hkv, p.B), dim3(kAttThreads), L::kBytes, st, p),
                          "sd_gather_attend: launch");
            return launch_status("sd_gather_attend");
        }
    }
    using L = MmaLayout<D, RP>;
    auto kern = p.ring_w > 0 ? attend_mma_kernel<D, RP, true> : attend_mma_kernel<D, RP, false>;
    SD_CUDA_CHECK(cudaFuncSetAttribute(kern, cudaFuncAttributeMaxDynamicSharedMemorySize, L::kBytes),
                  "sd_gather_attend: cudaFuncSetAttribute");
    SD_CUDA_CHECK(launch_pdl(kern, dim3(p.splits, p.Hkv, p.B), dim3(kAttThreads), L::kBytes, st, p),
                  "sd_gather_attend: launch");
    return launch_status("sd_gather_attend");
}

template <int D>
sd_status dispatch_rp(const AttendParams& p, int dtype, int RP, cudaStream_t st) {
    if (dtype == SD_BF16) return RP <= 16 ? launch_attend_mma<D, 16>(p, st) : launch_attend_mma<D, 32>(p, st);
    switch (RP) {
        case 4: return launch_attend<float, D, 4>(p, st);
        case 8: return launch_attend<float, D, 8>(p, st);
        case 16: return launch_attend<float, D, 16>(p, st);
        default: return launch_attend<float, D, 32>(p, st);
    }
}

}  // namespace
}  // namespace sd

using namespace sd;

sd_status sd::validate_attend_args(const sd_attend_args* a, const char* who) {
    SD_REQUIRE(a != nullptr, "%s: null args", who);
    SD_REQUIRE(a->B >= 0 && a->V >= 1 && a->Hq >= 1 && a->Hkv >= 1 && a->T >= 0,
               "%s: bad sizes (B=%d V=%d Hq=%d Hkv=%d T=%d)", who, a->B, a->V, a->Hq, a->Hkv, a->T);
    SD_REQUIRE(a->Hq % a->Hkv == 0, "%s: Hq must be a multiple of Hkv", who);
    SD_REQUIRE(valid_dtype(a->dtype), "%s: bad dtype", who);
    SD_REQUIRE(a->block >= 1 && a->n_idx >= 0, "%s: bad block / n_idx", who);
    SD_REQUIRE((long)a->n_idx * a->block <= (1L << 30), "%s: selection too large", who);
    if (a->idx == nullptr && a->n_idx > 0)
        SD_REQUIRE((long)a->n_idx * a->block == a->T, "%s: dense mode needs n_idx*block == T", who);
    if (a->d != 64 && a->d != 128) {
        set_error("%s: d must be 64 or 128 (got %d)", who, a->d);
        return SD_ERR_UNSUPPORTED;
    }
    const int rows_per_group = a->per_head ? a->V : (a->Hq / a->Hkv) * a->V;
    if (kernel_rows(a->dtype, rows_per_group) < 0) {
        set_error("%s: %d query rows per group exceed 32", who, rows_per_group);
        return SD_ERR_UNSUPPORTED;
    }
    SD_REQUIRE(a->B <= 65535 && a->Hq <= 65535, "%s: B and Hq must be <= 65535", who);
    SD_REQUIRE(a->per_head == 0 || a->per_head == 1, "%s: per_head must be 0 or 1", who);
    SD_REQUIRE(!a->per_head || a->idx != nullptr || a->n_idx == 0, "%s: per_head needs idx", who);
    SD_REQUIRE(a->ring_w >= 0 && a->ring_w <= (1 << 20), "%s: ring_w must be in [0, 2^20]", who);
    if (a->ring_w > 0) {
        SD_REQUIRE(a->ring_k && a->ring_v && a->ring_pos && a->qpos, "%s: a ring needs ring_k, ring_v, ring_pos and qpos",
                   who);
        SD_REQUIRE(aligned16(a->ring_k) && aligned16(a->ring_v), "%s: ring_k/ring_v must be 16-byte aligned", who);
    }
    SD_REQUIRE(a->T < kRingBase && a->pool_rows < kRingBase, "%s: T and pool_rows must be < 2^30", who);
    SD_REQUIRE(a->slot_per_head == 0 || a->slot_per_head == 1, "%s: slot_per_head must be 0 or 1", who);
    if (a->tier != nullptr) {
        if (a->dtype != SD_BF16 || a->d != 128 || a->per_head || a->ring_w > 0 || a->k_stage != nullptr) {
            set_error("%s: tiered rows need bf16, d = 128, no per_head, no ring and no stage", who);
            return SD_ERR_UNSUPPORTED;
        }
        SD_REQUIRE(a->k_int8 && a->v_int8 && a->k_scale && a->v_scale,
                   "%s: tier needs k_int8, v_int8, k_scale and v_scale", who);
        SD_REQUIRE(aligned16(a->k_int8) && aligned16(a->v_int8), "%s: k_int8/v_int8 must be 16-byte aligned", who);
        SD_REQUIRE(a->T < kI8Base && a->pool_rows < kI8Base, "%s: with tiers, T and pool_rows must be < 2^29", who);
    }
    return SD_OK;
}

extern "C" size_t sd_gather_attend_workspace_bytes(const sd_attend_args* a) {
    if (validate_attend_args(a, "sd_gather_attend") != SD_OK) return 0;
    return plan_splits(a).ws_bytes;
}

extern "C" sd_status sd_gather_attend(const sd_attend_args* a, void* stream) {
    clear_error();
    sd_status vs = validate_attend_args(a, "sd_gather_attend");
    if (vs != SD_OK) return vs;
    if (a->B == 0) return SD_OK;
    SD_REQUIRE(a->q && a->out && a->lse, "sd_gather_attend: null q/out/lse");
    SD_REQUIRE(aligned16(a->q) && aligned16(a->out), "sd_gather_attend: q and out must be 16-byte aligned");
    SplitPlan sp = plan_splits(a);
    AttendParams p{};
    p.q = a->q;
    p.kc = static_cast<const uint8_t*>(a->k_cache);
    p.vc = static_cast<const uint8_t*>(a->v_cache);
    p.slot_map = a->slot_map;
    p.idx = a->idx;
    p.B = a->B;
    p.V = a->V;
    p.Hq = a->Hq;
    p.kv_heads = a->Hkv;
    if (a->per_head) {  // one group per query head: G = 1, rows from KV head h / (Hq/Hkv)
        p.Hkv = a->Hq;
        p.G = 1;
        p.heads_per_kv = a->Hq / a->Hkv;
    } else {
        p.Hkv = a->Hkv;
        p.G = a->Hq / a->Hkv;
        p.heads_per_kv = 1;
    }
    p.R = p.G * a->V;
    p.T = a->T;
    p.n_idx = a->n_idx;
    p.block = a->block;
    p.n_hist = a->n_idx * a->block;
    p.n_rows = p.n_hist + a->ring_w;
    p.ring_w = a->ring_w;
    if (a->ring_w > 0) {
        p.rk = static_cast<const uint8_t*>(a->ring_k);
        p.rv = static_cast<const uint8_t*>(a->ring_v);
        p.ring_pos = a->ring_pos;
        p.qpos = a->qpos;
    }
    p.dtype = a->dtype;
    p.scale_log2 = a->scale * kLog2e;
    p.out = a->out;
    p.lse = a->lse;
    p.logits = a->logits;
    p.err = a->err_word;
    p.splits = sp.splits;
    p.rows_per_split = sp.rows_per_split;
    if (a->slot_map != nullptr) {
        SD_REQUIRE(a->pool_rows >= 0, "sd_gather_attend: pool_rows must be >= 0");
        SD_REQUIRE(a->k_host && a->v_host, "sd_gather_attend: slot_map needs k_host and v_host");
        SD_REQUIRE((a->k_stage == nullptr) == (a->v_stage == nullptr),
                   "sd_gather_attend: k_stage and v_stage go together");
        p.kh = mapped_host_ptr(a->k_host);
        p.vh = mapped_host_ptr(a->v_host);
        SD_REQUIRE(p.kh && p.vh, "sd_gather_attend: k_host/v_host must be pinned, mapped host memory");
        SD_REQUIRE(aligned16(a->k_host) && aligned16(a->v_host), "sd_gather_attend: host K/V must be 16-byte aligned");
        p.pool_rows = a->pool_rows;
        if (a->k_stage != nullptr) {  // host rows come from the HBM stage
            SD_REQUIRE(aligned16(a->k_stage) && aligned16(a->v_stage),
                       "sd_gather_attend: k_stage/v_stage must be 16-byte aligned");
            p.kh = static_cast<const uint8_t*>(a->k_stage);
            p.vh = static_cast<const uint8_t*>(a->v_stage);
            p.staged = 1;
        }
        p.slot_per_head = a->slot_per_head;
    } else {
        p.pool_rows = a->T;
    }
    if (p.n_rows > 0 && (a->slot_map == nullptr || a->pool_rows > 0)) {
        SD_REQUIRE(a->k_cache && a->v_cache, "sd_gather_attend: null k_cache/v_cache");
        SD_REQUIRE(aligned16(a->k_cache) && aligned16(a->v_cache),
                   "sd_gather_attend: k_cache/v_cache must be 16-byte aligned");
    }
    if (sp.splits > 1) {
        SD_REQUIRE(a->workspace != nullptr && a->workspace_bytes >= sp.ws_bytes,
                   "sd_gather_attend: workspace of %zu bytes needed (got %zu)", sp.ws_bytes,
                   a->workspace_bytes);
        SD_REQUIRE(aligned16(a->workspace), "sd_gather_attend: workspace must be 16-byte aligned");
        const size_t np = (size_t)a->B * p.Hkv * sp.splits * sp.RP;
        p.ws_o = static_cast<float*>(a->workspace);
        p.ws_m = p.ws_o + np * a->d;
        p.ws_l = p.ws_m + np;
    }
    if (a->tier != nullptr) {
        p.tier = a->tier;
        p.ki8 = a->k_int8;
        p.vi8 = a->v_int8;
        p.ksc = a->k_scale;
        p.vsc = a->v_scale;
    }
    // tiers alone (dense over the cache) need no resolving: a row's code follows from its tier
    p.resolve = (a->idx != nullptr || a->slot_map != nullptr || a->ring_w > 0) ? 1 : 0;
    cudaStream_t st = as_stream(stream);
    SD_REQUIRE(a->row_loop == 0 || a->row_loop == 1, "sd_gather_attend: row_loop must be 0 or 1");
    sd_status s1;
    if (dense_tma_eligible(a)) {
        // whole 64-row tiles of a cache in HBM (dense, or blocks of 16 or more rows); its
        // split count, at most the plan's, is the merge's
        int used = 1;
        s1 = dense_tma_launch(a, sp.splits, sp.RP, p.ws_o, p.ws_m, p.ws_l, &used, st);
        p.splits = used;
        sp.splits = used;
    } else {
        s1 = a->d == 128 ? dispatch_rp<128>(p, a->dtype, sp.RP, st) : dispatch_rp<64>(p, a->dtype, sp.RP, st);
    }
    if (s1 != SD_OK || sp.splits == 1) return s1;
    // the splits' partials merged by (group, query row), all in parallel
    const dim3 mgrid((unsigned)((long)a->B * p.Hkv), (unsigned)p.R);
    if (a->d == 128)
        SD_CUDA_CHECK(launch_pdl(attend_merge_kernel<128>, mgrid, dim3(kMergeThreads), 0, st, p, sp.RP),
                      "sd_gather_attend: merge launch");
    else
        SD_CUDA_CHECK(launch_pdl(attend_merge_kernel<64>, mgrid, dim3(kMergeThreads), 0, st, p, sp.RP),
                      "sd_gather_attend: merge launch");
    return launch_status("sd_gather_attend (merge)");
}
