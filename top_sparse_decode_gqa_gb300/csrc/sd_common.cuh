// sd_common.cuh -- device helpers shared by the libsdgqa kernels (sm_103a).
//
// Inline PTX for the Blackwell data-movement primitives the kernels use: mbarrier
// (init / expect-tx / bounded try_wait), 1-D bulk copies global -> shared completed on an
// mbarrier (the TMA unit's untiled path), and 16-byte cp.async.  Every wait is bounded by
// a wall-clock deadline read from %globaltimer; a wait that runs out reports
// SD_DEVERR_TIMEOUT instead of hanging.
#pragma once

#include <cuda_runtime.h>
#include <stdint.h>

#include "../../include/sd.h"

#define SD_DEVINL __device__ __forceinline__

namespace sd {

// Deadline for any single bounded wait: 1 s of wall-clock time.
constexpr uint64_t kWaitDeadlineNs = 1000000000ull;

SD_DEVINL uint64_t globaltimer_ns() {
    uint64_t t;
    asm volatile("mov.u64 %0, %%globaltimer;" : "=l"(t));
    return t;
}

SD_DEVINL void report(int32_t* err_word, int bits) {
    if (err_word != nullptr) atomicOr(reinterpret_cast<int*>(err_word), bits);
}

SD_DEVINL uint32_t smem_addr(const void* p) {
    return static_cast<uint32_t>(__cvta_generic_to_shared(p));
}

// ---------------------------------------------------------------- mbarrier

SD_DEVINL void mbar_init(uint64_t* bar, uint32_t count) {
    asm volatile("mbarrier.init.shared::cta.b64 [%0], %1;" ::"r"(smem_addr(bar)), "r"(count)
                 : "memory");
}

SD_DEVINL void fence_mbarrier_init() {
    asm volatile("fence.mbarrier_init.release.cluster;" ::: "memory");
}

// Order this thread's earlier generic-proxy shared-memory accesses before later
// async-proxy (bulk copy) accesses to the same memory.
SD_DEVINL void fence_proxy_async_shared() {
    asm volatile("fence.proxy.async.shared::cta;" ::: "memory");
}

SD_DEVINL void mbar_arrive_expect_tx(uint64_t* bar, uint32_t bytes) {
    asm volatile("mbarrier.arrive.expect_tx.shared::cta.b64 _, [%0], %1;" ::"r"(smem_addr(bar)),
                 "r"(bytes)
                 : "memory");
}

SD_DEVINL bool mbar_try_wait(uint64_t* bar, uint32_t parity) {
    uint32_t ok;
    asm volatile(
        "{\n\t.reg .pred p;\n\t"
        "mbarrier.try_wait.parity.shared::cta.b64 p, [%1], %2;\n\t"
        "selp.u32 %0, 1, 0, p;\n\t}"
        : "=r"(ok)
        : "r"(smem_addr(bar)), "r"(parity)
        : "memory");
    return ok != 0;
}

// try_wait that may suspend the thread for up to `hint_ns` (it resumes as soon as the phase
// completes): a waiting warp then takes no issue slots from the warps that work.
SD_DEVINL bool mbar_try_wait_sleep(uint64_t* bar, uint32_t parity, uint32_t hint_ns) {
    uint32_t ok;
    asm volatile(
        "{\n\t.reg .pred p;\n\t"
        "mbarrier.try_wait.parity.shared::cta.b64 p, [%1], %2, %3;\n\t"
        "selp.u32 %0, 1, 0, p;\n\t}"
        : "=r"(ok)
        : "r"(smem_addr(bar)), "r"(parity), "r"(hint_ns)
        : "memory");
    return ok != 0;
}

// Bounded wait for the phase with the given parity to complete.  Returns false when the
// deadline (limit_ns of wall-clock time, 1 s by default) passed first.
SD_DEVINL bool mbar_wait(uint64_t* bar, uint32_t parity, uint64_t limit_ns = kWaitDeadlineNs) {
    if (mbar_try_wait(bar, parity)) return true;
    const uint64_t t0 = globaltimer_ns();
    for (uint32_t i = 1;; ++i) {
        if (mbar_try_wait(bar, parity)) return true;
        if ((i & 63u) == 0 && globaltimer_ns() - t0 > limit_ns) return false;
    }
}

// Adds `bytes` to the transaction count the current phase waits for, without arriving.
SD_DEVINL void mbar_expect_tx(uint64_t* bar, uint32_t bytes) {
    asm volatile("mbarrier.expect_tx.relaxed.cta.shared::cta.b64 [%0], %1;" ::"r"(smem_addr(bar)), "r"(bytes)
                 : "memory");
}

// 1-D bulk copy (TMA, untiled) of `bytes` (multiple of 16, both addresses 16-byte
// aligned) from global to this CTA's shared memory, completing on `bar`.
SD_DEVINL void bulk_g2s(void* dst_smem, const void* src_gmem, uint32_t bytes, uint64_t* bar) {
    asm volatile(
        "cp.async.bulk.shared::cluster.global.mbarrier::complete_tx::bytes [%0], [%1], %2, [%3];" ::"r"(
            smem_addr(dst_smem)),
        "l"(src_gmem), "r"(bytes), "r"(smem_addr(bar))
        : "memory");
}

// ---------------------------------------------------------------- programmatic launch

// Wait until the grids this launch depends on have completed and their writes are
// visible (a no-op when the kernel was not launched as a programmatic dependent).
SD_DEVINL void pdl_wait() { asm volatile("griddepcontrol.wait;" ::: "memory"); }

// Allow the next kernel in the stream, if launched as a programmatic dependent, to be
// scheduled now; it still waits (pdl_wait) for this grid to finish before reading.
SD_DEVINL void pdl_launch_dependents() { asm volatile("griddepcontrol.launch_dependents;" ::: "memory"); }

// ---------------------------------------------------------------- L2 policies

// A cache policy that marks the lines a load brings into L2 as first to evict: for data
// streamed once (so that it does not push out data that is read again soon).
SD_DEVINL uint64_t l2_evict_first_policy() {
    uint64_t pol;
    asm volatile("createpolicy.fractional.L2::evict_first.b64 %0, 1.0;" : "=l"(pol));
    return pol;
}

// 1-D bulk copy with an L2 cache policy (see bulk_g2s).
SD_DEVINL void bulk_g2s_hint(void* dst_smem, const void* src_gmem, uint32_t bytes, uint64_t* bar,
                             uint64_t policy) {
    asm volatile(
        "cp.async.bulk.shared::cluster.global.mbarrier::complete_tx::bytes.L2::cache_hint [%0], [%1], %2, [%3], %4;" ::"r"(
            smem_addr(dst_smem)),
        "l"(src_gmem), "r"(bytes), "r"(smem_addr(bar)), "l"(policy)
        : "memory");
}

// 2^x with the hardware approximation (relative error about 2^-22), flushing denormals.
SD_DEVINL float fast_exp2(float x) {
    float y;
    asm("ex2.approx.ftz.f32 %0, %1;" : "=f"(y) : "f"(x));
    return y;
}

// ---------------------------------------------------------------- cp.async (16 B)

SD_DEVINL void cp_async16(void* dst_smem, const void* src) {
    asm volatile("cp.async.cg.shared.global [%0], [%1], 16;" ::"r"(smem_addr(dst_smem)), "l"(src)
                 : "memory");
}
// 4-byte cp.async (through L1); both addresses 4-byte aligned.
SD_DEVINL void cp_async4(void* dst_smem, const void* src) {
    asm volatile("cp.async.ca.shared.global [%0], [%1], 4;" ::"r"(smem_addr(dst_smem)), "l"(src) : "memory");
}
// 16-byte cp.async that copies src_size (0 or 16) bytes and fills the rest with zeros.
SD_DEVINL void cp_async16_zfill(void* dst_smem, const void* src, uint32_t src_size) {
    asm volatile("cp.async.cg.shared.global [%0], [%1], 16, %2;" ::"r"(smem_addr(dst_smem)), "l"(src),
                 "r"(src_size)
                 : "memory");
}
// One arrival on `bar` once every cp.async this thread issued before it has landed (the
// arrival is not added to the barrier's expected count: init the count to include it).
SD_DEVINL void cp_async_mbar_arrive_noinc(uint64_t* bar) {
    asm volatile("cp.async.mbarrier.arrive.noinc.shared::cta.b64 [%0];" ::"r"(smem_addr(bar)) : "memory");
}
// Like cp_async_mbar_arrive_noinc, but the arrival is counted at issue and taken back when the
// copies land (no change to the expected count; the phase cannot complete before they land).
SD_DEVINL void cp_async_mbar_arrive(uint64_t* bar) {
    asm volatile("cp.async.mbarrier.arrive.shared::cta.b64 [%0];" ::"r"(smem_addr(bar)) : "memory");
}
SD_DEVINL void cp_async_commit() { asm volatile("cp.async.commit_group;" ::: "memory"); }
template <int N>
SD_DEVINL void cp_async_wait() {
    asm volatile("cp.async.wait_group %0;" ::"n"(N) : "memory");
}

// ---------------------------------------------------------------- warp-level MMA (m16n8k16)

// Four 8x8 b16 matrices from shared memory; lane l gives the address of row (l & 7) of
// matrix (l >> 3).  The .trans form transposes each matrix.
SD_DEVINL void ldsm_x4(uint32_t addr, uint32_t& r0, uint32_t& r1, uint32_t& r2, uint32_t& r3) {
    asm volatile("ldmatrix.sync.aligned.m8n8.x4.shared.b16 {%0,%1,%2,%3}, [%4];"
                 : "=r"(r0), "=r"(r1), "=r"(r2), "=r"(r3)
                 : "r"(addr));
}
SD_DEVINL void ldsm_x4_t(uint32_t addr, uint32_t& r0, uint32_t& r1, uint32_t& r2, uint32_t& r3) {
    asm volatile("ldmatrix.sync.aligned.m8n8.x4.trans.shared.b16 {%0,%1,%2,%3}, [%4];"
                 : "=r"(r0), "=r"(r1), "=r"(r2), "=r"(r3)
                 : "r"(addr));
}

// Transpose of an 8x8 matrix of 16-bit elements held one 32-bit pair per lane (lane l: row
// l / 4, columns 2(l % 4) and 2(l % 4) + 1), returned in the same distribution.
SD_DEVINL uint32_t movmatrix_t(uint32_t a) {
    uint32_t d;
    asm volatile("movmatrix.sync.aligned.m8n8.trans.b16 %0, %1;" : "=r"(d) : "r"(a));
    return d;
}

// D (16x8 fp32) += A (16x16 bf16, row) * B (16x8 bf16, col).
SD_DEVINL void mma_bf16_16816(float (&d)[4], uint32_t a0, uint32_t a1, uint32_t a2, uint32_t a3,
                              uint32_t b0, uint32_t b1) {
    asm volatile(
        "mma.sync.aligned.m16n8k16.row.col.f32.bf16.bf16.f32 {%0,%1,%2,%3}, {%4,%5,%6,%7}, {%8,%9}, "
        "{%0,%1,%2,%3};"
        : "+f"(d[0]), "+f"(d[1]), "+f"(d[2]), "+f"(d[3])
        : "r"(a0), "r"(a1), "r"(a2), "r"(a3), "r"(b0), "r"(b1));
}

// D (16x8 fp32) += A (16x16 fp16, row) * B (16x8 fp16, col).
SD_DEVINL void mma_f16_16816(float (&d)[4], uint32_t a0, uint32_t a1, uint32_t a2, uint32_t a3, uint32_t b0,
                             uint32_t b1) {
    asm volatile(
        "mma.sync.aligned.m16n8k16.row.col.f32.f16.f16.f32 {%0,%1,%2,%3}, {%4,%5,%6,%7}, {%8,%9}, "
        "{%0,%1,%2,%3};"
        : "+f"(d[0]), "+f"(d[1]), "+f"(d[2]), "+f"(d[3])
        : "r"(a0), "r"(a1), "r"(a2), "r"(a3), "r"(b0), "r"(b1));
}

// ---------------------------------------------------------------- device-scope flags

SD_DEVINL uint32_t ld_acquire_gpu(const uint32_t* p) {
    uint32_t v;
    asm volatile("ld.acquire.gpu.global.u32 %0, [%1];" : "=r"(v) : "l"(p) : "memory");
    return v;
}
SD_DEVINL void st_release_gpu(uint32_t* p, uint32_t v) {
    asm volatile("st.release.gpu.global.u32 [%0], %1;" ::"l"(p), "r"(v) : "memory");
}
SD_DEVINL uint32_t atom_add_acq_rel_gpu(uint32_t* p, uint32_t v) {
    uint32_t old;
    asm volatile("atom.acq_rel.gpu.global.add.u32 %0, [%1], %2;" : "=r"(old) : "l"(p), "r"(v) : "memory");
    return old;
}
SD_DEVINL void fence_acq_rel_gpu() { asm volatile("fence.acq_rel.gpu;" ::: "memory"); }
// Fire-and-forget device-scope add with release semantics (no value comes back, so the issuing
// thread does not wait for it).
SD_DEVINL void red_add_release_gpu(uint32_t* p, uint32_t v) {
    asm volatile("red.release.gpu.global.add.u32 [%0], %1;" ::"l"(p), "r"(v) : "memory");
}

// Two fp32 -> packed bf16x2 (round to nearest even), first value in the low half.
SD_DEVINL uint32_t pack_bf16x2(float lo, float hi) {
    uint32_t d;
    asm("cvt.rn.bf16x2.f32 %0, %1, %2;" : "=r"(d) : "f"(hi), "f"(lo));
    return d;
}

// x = hi + lo with hi = bf16(x) and lo = bf16(x - hi): 16 significant bits in two bf16.
SD_DEVINL void split_bf16x2(float x0, float x1, uint32_t& hi, uint32_t& lo) {
    hi = pack_bf16x2(x0, x1);
    const float h0 = __uint_as_float(hi << 16), h1 = __uint_as_float(hi & 0xffff0000u);
    lo = pack_bf16x2(x0 - h0, x1 - h1);
}

// ---------------------------------------------------------------- element access

// Two bfloat16 packed in a 32-bit word -> two fp32 (exact).
SD_DEVINL float bf16lo(uint32_t w) { return __uint_as_float(w << 16); }
SD_DEVINL float bf16hi(uint32_t w) { return __uint_as_float(w & 0xffff0000u); }

SD_DEVINL float load_elem(const void* base, int dtype, size_t i) {
    if (dtype == SD_F32) return reinterpret_cast<const float*>(base)[i];
    const uint16_t b = reinterpret_cast<const uint16_t*>(base)[i];
    return __uint_as_float(static_cast<uint32_t>(b) << 16);
}

// 16 bytes of storage -> fp32 values (8 for bf16, 4 for fp32).
template <typename T>
struct Unpack16;
template <>
struct Unpack16<float> {
    static constexpr int kElems = 4;
    SD_DEVINL static void run(const uint4& r, float* x) {
        x[0] = __uint_as_float(r.x);
        x[1] = __uint_as_float(r.y);
        x[2] = __uint_as_float(r.z);
        x[3] = __uint_as_float(r.w);
    }
};
struct bf16_t {
    uint16_t bits;
};
template <>
struct Unpack16<bf16_t> {
    static constexpr int kElems = 8;
    SD_DEVINL static void run(const uint4& r, float* x) {
        x[0] = bf16lo(r.x);
        x[1] = bf16hi(r.x);
        x[2] = bf16lo(r.y);
        x[3] = bf16hi(r.y);
        x[4] = bf16lo(r.z);
        x[5] = bf16hi(r.z);
        x[6] = bf16lo(r.w);
        x[7] = bf16hi(r.w);
    }
};

SD_DEVINL uint4 lds128(const void* p) { return *reinterpret_cast<const uint4*>(p); }

// ---------------------------------------------------------------- warp reductions

SD_DEVINL float warp_max(float v) {
#pragma unroll
    for (int o = 16; o > 0; o >>= 1) v = fmaxf(v, __shfl_xor_sync(0xffffffffu, v, o));
    return v;
}
SD_DEVINL float warp_sum(float v) {
#pragma unroll
    for (int o = 16; o > 0; o >>= 1) v += __shfl_xor_sync(0xffffffffu, v, o);
    return v;
}

SD_DEVINL uint32_t lanemask_lt() {
    uint32_t m;
    asm("mov.u32 %0, %%lanemask_lt;" : "=r"(m));
    return m;
}

// Order-preserving map of fp32 to uint32 (a < b as floats <=> key(a) < key(b)), with
// -0.0 mapped like +0.0 so the two compare equal.
SD_DEVINL uint32_t float_key(float f) {
    uint32_t u = __float_as_uint(f);
    if ((u << 1) == 0u) u = 0u;
    return (u & 0x80000000u) ? ~u : (u | 0x80000000u);
}

// Same for fp64 -> uint64.
SD_DEVINL uint64_t double_key(double f) {
    uint64_t u = static_cast<uint64_t>(__double_as_longlong(f));
    if ((u << 1) == 0ull) u = 0ull;
    return (u & 0x8000000000000000ull) ? ~u : (u | 0x8000000000000000ull);
}

}  // namespace sd
