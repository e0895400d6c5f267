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

#include "sd_common.cuh"
#include "sd_host.h"

namespace sd {
namespace {

constexpr int kAttThreads = 128;
constexpr int kCH = 64;  // rows per staged chunk
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
    int dtype;
    float scale_log2;
    float* out;
    float* lse;
    float* logits;
    int32_t* err;
    float* ws_o;
    float* ws_m;
    float* ws_l;
};

template <typename ST, int D, int RP>
struct AttLayout {
    static constexpr int kPadE = 16 / (int)sizeof(ST);      // 16-byte row pad for K
    static constexpr int kKRow = (D + kPadE) * (int)sizeof(ST);
    static constexpr int kVRow = D * (int)sizeof(ST);
    static constexpr int kPRow = RP + 4;                    // floats per p row
    static constexpr int kSRow = kCH + 4;                   // floats per s row
    static constexpr int oQ = 0;
    static constexpr int oK = oQ + RP * D * 4;
    static constexpr int oV = oK + 2 * kCH * kKRow;
    static constexpr int oP = oV + 2 * kCH * kVRow;
    static constexpr int oS = oP + kCH * kPRow * 4;
    static constexpr int oSrc = oS + RP * kSRow * 4;
    static constexpr int oAlpha = oSrc + 2 * 2 * kCH * 8;
    static constexpr int oM = oAlpha + RP * 4;
    static constexpr int oL = oM + RP * 4;
    static constexpr int kBytes = oL + RP * 4;
    static_assert(oV % 16 == 0 && oP % 16 == 0 && oS % 16 == 0 && oSrc % 16 == 0, "align");
    static_assert((RP == 4 ? 4 : 1) * RP * D * 4 <= 2 * kCH * kKRow, "reduction buffer must fit in K");
};

template <typename ST, int D, int RP>
__global__ void __launch_bounds__(kAttThreads) attend_kernel(const AttendParams p) {
    using L = AttLayout<ST, D, RP>;
    using U = Unpack16<ST>;
    constexpr int EPC = U::kElems;         // elements per 16 bytes
    constexpr int PPR = L::kVRow / 16;     // 16-byte pieces per row
    constexpr int CPL = D / 32;            // PV columns per lane
    constexpr bool kKeySplit = (RP == 4);  // PV: warps split keys (else query rows)
    constexpr int QW = kKeySplit ? RP : RP / 4;  // PV query rows per warp

    extern __shared__ __align__(128) uint8_t sm[];
    float* qs = reinterpret_cast<float*>(sm + L::oQ);
    float* ps = reinterpret_cast<float*>(sm + L::oP);
    float* ss = reinterpret_cast<float*>(sm + L::oS);
    const uint8_t** srcs = reinterpret_cast<const uint8_t**>(sm + L::oSrc);  // [2 bufs][K,V][kCH]
    float* alpha_s = reinterpret_cast<float*>(sm + L::oAlpha);
    float* m_s = reinterpret_cast<float*>(sm + L::oM);
    float* l_s = reinterpret_cast<float*>(sm + L::oL);

    const int tid = threadIdx.x, lane = tid & 31, warp = tid >> 5;
    const int split = blockIdx.x, kvh = blockIdx.y, b = blockIdx.z;
    const int bk = b * p.Hkv + kvh;
    const size_t esz = sizeof(ST);

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
    const int nch = j1 > j0 ? (j1 - j0 + kCH - 1) / kCH : 0;

    auto compute_src = [&](int c, int bf) {
        if (tid < kCH) {
            const int jg = j0 + c * kCH + tid;
            const uint8_t* sk = nullptr;
            const uint8_t* sv = nullptr;
            if (jg < j1) {
                long pos = jg;
                bool ok = true;
                if (p.idx != nullptr) {
                    const long sel = p.idx[(size_t)bk * p.n_idx + jg / p.block];
                    pos = sel * p.block + jg % p.block;
                    if (sel < 0 || pos >= p.T) {
                        report(p.err, SD_DEVERR_INDEX);
                        ok = false;
                    }
                }
                if (ok) {
                    if (p.slot_map != nullptr) {
                        const int slot = p.slot_map[(size_t)b * p.T + pos];
                        if (slot >= 0 && slot < p.pool_rows) {
                            const size_t row = (size_t)bk * p.pool_rows + slot;
                            sk = p.kc + row * L::kVRow;
                            sv = p.vc + row * L::kVRow;
                        } else if (slot == -1) {
                            const size_t row = (size_t)bk * p.T + pos;
                            sk = p.kh + row * L::kVRow;
                            sv = p.vh + row * L::kVRow;
                        } else {
                            report(p.err, SD_DEVERR_SLOT);
                        }
                    } else {
                        const size_t row = (size_t)bk * p.T + pos;
                        sk = p.kc + row * L::kVRow;
                        sv = p.vc + row * L::kVRow;
                    }
                }
            }
            srcs[(bf * 2 + 0) * kCH + tid] = sk;
            srcs[(bf * 2 + 1) * kCH + tid] = sv;
        }
    };
    auto issue = [&](int bf) {
        uint8_t* kdst = sm + L::oK + bf * kCH * L::kKRow;
        uint8_t* vdst = sm + L::oV + bf * kCH * L::kVRow;
        for (int pc = tid; pc < 2 * kCH * PPR; pc += kAttThreads) {
            const int which = pc / (kCH * PPR);
            const int rem = pc - which * (kCH * PPR);
            const int j = rem / PPR, part = rem % PPR;
            const uint8_t* src = srcs[(bf * 2 + which) * kCH + j];
            uint8_t* dst = which ? vdst + j * L::kVRow + part * 16 : kdst + j * L::kKRow + part * 16;
            if (src != nullptr)
                cp_async16(dst, src + part * 16);
            else
                *reinterpret_cast<uint4*>(dst) = make_uint4(0u, 0u, 0u, 0u);
        }
        cp_async_commit();
    };

    // softmax state: warp w owns query rows r = w + 4*i
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

    if (nch > 0) {
        compute_src(0, 0);
        __syncthreads();
        issue(0);
    }
    for (int c = 0; c < nch; ++c) {
        const int bf = c & 1;
        if (c + 1 < nch) {
            compute_src(c + 1, bf ^ 1);
            __syncthreads();
            issue(bf ^ 1);
            cp_async_wait<1>();
        } else {
            cp_async_wait<0>();
        }
        __syncthreads();

        // ---- QK: thread -> key j, half hf of the query rows
        {
            const int j = tid & (kCH - 1), hf = tid / kCH;
            const uint8_t* krow = sm + L::oK + (bf * kCH + j) * L::kKRow;
            const bool valid = srcs[(bf * 2) * kCH + j] != nullptr;
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
            for (int r = 0; r < RP / 2; ++r) ss[(hf * (RP / 2) + r) * L::kSRow + j] = valid ? s[r] : -INFINITY;
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
    }

    // ---- publish m, l; reduce the key-split partial sums
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

// Combines the split partials of one (b, kvh) in split order.
template <int D>
__global__ void attend_merge_kernel(const AttendParams p, int RP) {
    const int bk = blockIdx.x;
    const int b = bk / p.Hkv, kvh = bk % p.Hkv;
    for (int e = threadIdx.x; e < p.R * D; e += blockDim.x) {
        const int r = e / D, col = e % D;
        const size_t base = (size_t)bk * p.splits * RP + r;
        float M = -INFINITY;
        for (int s = 0; s < p.splits; ++s) M = fmaxf(M, p.ws_m[base + (size_t)s * RP]);
        float Lsum = 0.f, acc = 0.f;
        if (M != -INFINITY) {
            for (int s = 0; s < p.splits; ++s) {
                const float m = p.ws_m[base + (size_t)s * RP];
                if (m == -INFINITY) continue;
                const float w = exp2f(m - M);
                Lsum = fmaf(p.ws_l[base + (size_t)s * RP], w, Lsum);
                acc = fmaf(p.ws_o[(base + (size_t)s * RP) * D + col], w, acc);
            }
        }
        const int v = r / p.G, g = r % p.G;
        const size_t qrow = ((size_t)b * p.V + v) * p.Hq + kvh * p.G + g;
        p.out[qrow * D + col] = Lsum > 0.f ? acc / Lsum : 0.f;
        if (col == 0) p.lse[qrow] = Lsum > 0.f ? (M + log2f(Lsum)) * kLn2 : -INFINITY;
    }
}

int padded_rows(int R) { return R <= 4 ? 4 : R <= 8 ? 8 : R <= 16 ? 16 : R <= 32 ? 32 : -1; }

struct SplitPlan {
    int splits, rows_per_split, RP;
    size_t ws_bytes;
};

SplitPlan plan_splits(const sd_attend_args* a) {
    SplitPlan sp{};
    const long n_rows = (long)a->n_idx * a->block;
    const long bk = (long)a->B * a->Hkv;
    sp.RP = padded_rows(a->Hkv > 0 ? (a->Hq / a->Hkv) * a->V : 0);
    const long chunks = (n_rows + kCH - 1) / kCH;
    long splits;
    if (a->splits > 0) {
        splits = a->splits;
    } else {
        const long target = (long)num_sms() * 6;  // ~2 waves of 3 CTAs per SM
        splits = bk > 0 ? (target + bk - 1) / bk : 1;
    }
    splits = std::max(1L, std::min(splits, std::max(1L, chunks)));
    long rps = chunks > 0 ? ((chunks + splits - 1) / splits) * kCH : kCH;
    splits = n_rows > 0 ? (n_rows + rps - 1) / rps : 1;
    sp.splits = (int)splits;
    sp.rows_per_split = (int)rps;
    sp.ws_bytes = splits > 1 ? (size_t)bk * splits * sp.RP * (a->d + 2) * sizeof(float) : 0;
    return sp;
}

template <typename ST, int D, int RP>
sd_status launch_attend(const AttendParams& p, cudaStream_t st) {
    using L = AttLayout<ST, D, RP>;
    auto kern = attend_kernel<ST, D, RP>;
    SD_CUDA_CHECK(cudaFuncSetAttribute(kern, cudaFuncAttributeMaxDynamicSharedMemorySize, L::kBytes),
                  "sd_gather_attend: cudaFuncSetAttribute");
    dim3 grid(p.splits, p.Hkv, p.B);
    kern<<<grid, kAttThreads, L::kBytes, st>>>(p);
    sd_status s = launch_status("sd_gather_attend");
    if (s != SD_OK || p.splits == 1) return s;
    attend_merge_kernel<D><<<p.B * p.Hkv, 256, 0, st>>>(p, RP);
    return launch_status("sd_gather_attend (merge)");
}

template <typename ST, int D>
sd_status dispatch_rp(const AttendParams& p, int RP, cudaStream_t st) {
    switch (RP) {
        case 4: return launch_attend<ST, D, 4>(p, st);
        case 8: return launch_attend<ST, D, 8>(p, st);
        case 16: return launch_attend<ST, D, 16>(p, st);
        default: return launch_attend<ST, D, 32>(p, st);
    }
}

// Device address of pinned host memory (NULL if it is not mapped pinned memory).
const uint8_t* host_dev_ptr(const void* h) {
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

static sd_status validate_attend(const sd_attend_args* a) {
    SD_REQUIRE(a != nullptr, "sd_gather_attend: null args");
    SD_REQUIRE(a->B >= 0 && a->V >= 1 && a->Hq >= 1 && a->Hkv >= 1 && a->T >= 0,
               "sd_gather_attend: bad sizes (B=%d V=%d Hq=%d Hkv=%d T=%d)", a->B, a->V, a->Hq, a->Hkv, a->T);
    SD_REQUIRE(a->Hq % a->Hkv == 0, "sd_gather_attend: Hq must be a multiple of Hkv");
    SD_REQUIRE(valid_dtype(a->dtype), "sd_gather_attend: bad dtype");
    SD_REQUIRE(a->block >= 1 && a->n_idx >= 0, "sd_gather_attend: bad block / n_idx");
    SD_REQUIRE((long)a->n_idx * a->block <= (1L << 30), "sd_gather_attend: selection too large");
    if (a->idx == nullptr && a->n_idx > 0)
        SD_REQUIRE((long)a->n_idx * a->block == a->T, "sd_gather_attend: dense mode needs n_idx*block == T");
    if (a->d != 64 && a->d != 128) {
        set_error("sd_gather_attend: d must be 64 or 128 (got %d)", a->d);
        return SD_ERR_UNSUPPORTED;
    }
    if (padded_rows((a->Hq / a->Hkv) * a->V) < 0) {
        set_error("sd_gather_attend: G*V = %d exceeds 32", (a->Hq / a->Hkv) * a->V);
        return SD_ERR_UNSUPPORTED;
    }
    SD_REQUIRE(a->B <= 65535 && a->Hkv <= 65535, "sd_gather_attend: B and Hkv must be <= 65535");
    return SD_OK;
}

extern "C" size_t sd_gather_attend_workspace_bytes(const sd_attend_args* a) {
    if (validate_attend(a) != SD_OK) return 0;
    return plan_splits(a).ws_bytes;
}

extern "C" sd_status sd_gather_attend(const sd_attend_args* a, void* stream) {
    clear_error();
    sd_status vs = validate_attend(a);
    if (vs != SD_OK) return vs;
    if (a->B == 0) return SD_OK;
    SD_REQUIRE(a->q && a->out && a->lse, "sd_gather_attend: null q/out/lse");
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
    p.Hkv = a->Hkv;
    p.G = a->Hq / a->Hkv;
    p.R = p.G * a->V;
    p.T = a->T;
    p.n_idx = a->n_idx;
    p.block = a->block;
    p.n_rows = a->n_idx * a->block;
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
        p.kh = host_dev_ptr(a->k_host);
        p.vh = host_dev_ptr(a->v_host);
        SD_REQUIRE(p.kh && p.vh, "sd_gather_attend: k_host/v_host must be pinned, mapped host memory");
        SD_REQUIRE(aligned16(a->k_host) && aligned16(a->v_host), "sd_gather_attend: host K/V must be 16-byte aligned");
        p.pool_rows = a->pool_rows;
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
        const size_t np = (size_t)a->B * a->Hkv * sp.splits * sp.RP;
        p.ws_o = static_cast<float*>(a->workspace);
        p.ws_m = p.ws_o + np * a->d;
        p.ws_l = p.ws_m + np;
    }
    cudaStream_t st = as_stream(stream);
    if (a->dtype == SD_BF16)
        return a->d == 128 ? dispatch_rp<bf16_t, 128>(p, sp.RP, st) : dispatch_rp<bf16_t, 64>(p, sp.RP, st);
    return a->d == 128 ? dispatch_rp<float, 128>(p, sp.RP, st) : dispatch_rp<float, 64>(p, sp.RP, st);
}
