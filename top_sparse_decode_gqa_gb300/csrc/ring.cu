// ring.cu -- the draft tokens' K/V written into a window-bounded ring.
//
// "O Fim do Gargalo de Memoria: Como o Adaptive DHiSparse Revolutiona LLMs de Contexto
// Longo" (news page), "Metodologia e Eficiencia de Carga": the draft model's K/V lives in
// a ring bounded by a window.  Token position t lives in slot t mod W, so the ring always
// holds the last W tokens and a slot's position tells the attention whether a query may
// see it (sd_gather_attend's causal mask over the ring).
#include "sd_common.cuh"
#include "sd_host.h"

namespace sd {
namespace {

constexpr int kRingThreads = 128;

// Grid (n tokens, Hkv, B): one CTA copies one token's K and V rows of one KV head as 16-byte
// pieces; the (h == 0) CTA also records the slot's position.
__global__ void __launch_bounds__(kRingThreads)
    ring_append_kernel(const uint8_t* __restrict__ k_new, const uint8_t* __restrict__ v_new, int n, int row_bytes,
                       uint8_t* __restrict__ ring_k, uint8_t* __restrict__ ring_v, int32_t* __restrict__ ring_pos,
                       const int32_t* __restrict__ pos0, int W) {
    pdl_wait();  // the new rows may come from the preceding kernel
    pdl_launch_dependents();
    const int i = blockIdx.x, h = blockIdx.y, b = blockIdx.z, Hkv = gridDim.y;
    const int pos = pos0[b] + i;
    if (pos < 0) return;  // outside the contract (pos0 >= 0): nothing is written
    const int slot = pos % W;
    const size_t src = (((size_t)b * Hkv + h) * n + i) * row_bytes;
    const size_t dst = (((size_t)b * Hkv + h) * W + slot) * row_bytes;
    const int pieces = row_bytes / 16;
    for (int e = threadIdx.x; e < 2 * pieces; e += kRingThreads) {
        const int which = e / pieces, off = (e % pieces) * 16;
        const uint4 x = *reinterpret_cast<const uint4*>((which ? v_new : k_new) + src + off);
        *reinterpret_cast<uint4*>((which ? ring_v : ring_k) + dst + off) = x;
    }
    if (h == 0 && threadIdx.x == 0) ring_pos[(size_t)b * W + slot] = pos;
}

}  // namespace
}  // namespace sd

using namespace sd;

extern "C" sd_status sd_ring_append(const void* k_new, const void* v_new, sd_dtype dtype, int B, int Hkv, int n, int d,
                                    void* ring_k, void* ring_v, int32_t* ring_pos, const int32_t* pos0, int W,
                                    void* stream) {
    clear_error();
    SD_REQUIRE(valid_dtype(dtype), "sd_ring_append: bad dtype");
    SD_REQUIRE(B >= 0 && Hkv >= 1 && W >= 1, "sd_ring_append: bad sizes (B=%d Hkv=%d W=%d)", B, Hkv, W);
    SD_REQUIRE(n >= 1 && n <= W, "sd_ring_append: n (%d) must be in [1, W=%d]", n, W);
    SD_REQUIRE(B <= 65535 && Hkv <= 65535, "sd_ring_append: B and Hkv must be <= 65535");
    if (d != 64 && d != 128) {
        set_error("sd_ring_append: d must be 64 or 128 (got %d)", d);
        return SD_ERR_UNSUPPORTED;
    }
    if (B == 0) return SD_OK;
    SD_REQUIRE(k_new && v_new && ring_k && ring_v && ring_pos && pos0, "sd_ring_append: null pointer");
    SD_REQUIRE(aligned16(k_new) && aligned16(v_new) && aligned16(ring_k) && aligned16(ring_v),
               "sd_ring_append: K/V pointers must be 16-byte aligned");
    SD_CUDA_CHECK(launch_pdl(ring_append_kernel, dim3((unsigned)n, (unsigned)Hkv, (unsigned)B), dim3(kRingThreads), 0,
                             as_stream(stream), static_cast<const uint8_t*>(k_new), static_cast<const uint8_t*>(v_new),
                             n, d * dtype_bytes(dtype), static_cast<uint8_t*>(ring_k), static_cast<uint8_t*>(ring_v),
                             ring_pos, pos0, W),
                  "sd_ring_append: launch");
    return launch_status("sd_ring_append");
}
