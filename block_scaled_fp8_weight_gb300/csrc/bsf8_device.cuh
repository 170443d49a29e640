// bsf8_device.cuh -- device helpers shared by the libbsf8 kernels (sm_103a).
//
// PTX wrappers for mbarriers, bulk copies, L2 prefetch, programmatic dependent launch,
// cluster barriers and the bf16 tensor-core MMA, plus the exact e4m3 -> bf16 rebuild
// used by the GEMM and by bsf8_dequant.
#pragma once

#include <cuda_runtime.h>
#include <stdint.h>

namespace bsf8 {

// Kernels record a bounded wait that ran out in the library's device status word
// (defined in bsf8_abi.cu; its address reaches the kernels as a parameter).
constexpr int kStatusTimeout = 7;  // == BSF8_ERR_TIMEOUT

__device__ __forceinline__ uint32_t smem_u32(const void *p) {
    return static_cast<uint32_t>(__cvta_generic_to_shared(p));
}

// ------------------------------------------------------------------ mbarrier

__device__ __forceinline__ void mbar_init(uint64_t *bar, uint32_t count) {
    asm volatile("mbarrier.init.shared::cta.b64 [%0], %1;" ::"r"(smem_u32(bar)), "r"(count)
                 : "memory");
}

__device__ __forceinline__ void fence_mbar_init() {
    asm volatile("fence.mbarrier_init.release.cluster;" ::: "memory");
}

__device__ __forceinline__ void mbar_arrive_expect_tx(uint64_t *bar, uint32_t bytes) {
    asm volatile("mbarrier.arrive.expect_tx.shared::cta.b64 _, [%0], %1;" ::"r"(smem_u32(bar)),
                 "r"(bytes)
                 : "memory");
}

__device__ __forceinline__ void mbar_arrive(uint64_t *bar) {
    asm volatile("mbarrier.arrive.shared::cta.b64 _, [%0];" ::"r"(smem_u32(bar)) : "memory");
}

__device__ __forceinline__ bool mbar_try_wait(uint64_t *bar, uint32_t parity) {
    uint32_t done;
    asm volatile(
        "{\n\t.reg .pred p;\n\t"
        "mbarrier.try_wait.parity.shared::cta.b64 p, [%1], %2;\n\t"
        "selp.u32 %0, 1, 0, p;\n\t}"
        : "=r"(done)
        : "r"(smem_u32(bar)), "r"(parity)
        : "memory");
    return done != 0;
}

// As mbar_try_wait, but the thread may be suspended (issuing nothing) until the phase
// completes or about hint_ns have passed, instead of returning at once.
__device__ __forceinline__ bool mbar_try_wait_suspend(uint64_t *bar, uint32_t parity,
                                                      uint32_t hint_ns) {
    uint32_t done;
    asm volatile(
        "{\n\t.reg .pred p;\n\t"
        "mbarrier.try_wait.parity.shared::cta.b64 p, [%1], %2, %3;\n\t"
        "selp.u32 %0, 1, 0, p;\n\t}"
        : "=r"(done)
        : "r"(smem_u32(bar)), "r"(parity), "r"(hint_ns)
        : "memory");
    return done != 0;
}

__device__ __forceinline__ uint64_t global_ns() {
    uint64_t t;
    asm volatile("mov.u64 %0, %%globaltimer;" : "=l"(t));
    return t;
}

// Waits for the phase of `bar` with the given parity to complete, for at most
// timeout_ns of wall time.  Returns false when the bound ran out.  While it waits the
// thread sleeps in the barrier (suspend hint) rather than spinning, so a waiting warp
// leaves the SM's issue slots to the warps that have work.
__device__ __forceinline__ bool mbar_wait_bounded(uint64_t *bar, uint32_t parity,
                                                  uint64_t timeout_ns) {
    if (mbar_try_wait(bar, parity)) return true;
    const uint64_t t0 = global_ns();
    while (true) {
        if (mbar_try_wait_suspend(bar, parity, 1000000u)) return true;
        if (global_ns() - t0 > timeout_ns) return false;
    }
}

__device__ __forceinline__ void report_timeout(int *status) { atomicExch(status, kStatusTimeout); }

// ------------------------------------------------------------- bulk copies (TMA)

// 1-D bulk copy global -> this CTA's shared memory; completes `bytes` of transaction
// count on `bar`.  dst, src 16-byte aligned; bytes a multiple of 16.
__device__ __forceinline__ void bulk_g2s(void *dst, const void *src, uint32_t bytes,
                                         uint64_t *bar) {
    asm volatile(
        "cp.async.bulk.shared::cluster.global.mbarrier::complete_tx::bytes [%0], [%1], %2, [%3];" ::
            "r"(smem_u32(dst)),
        "l"(src), "r"(bytes), "r"(smem_u32(bar))
        : "memory");
}

// Bulk prefetch of [src, src+bytes) into L2 (a hint; L2 is coherent, so it is safe to
// issue before the producing kernel has finished).  src 16-byte aligned, bytes % 16 == 0.
__device__ __forceinline__ void prefetch_l2(const void *src, uint32_t bytes) {
    asm volatile("cp.async.bulk.prefetch.L2.global [%0], %1;" ::"l"(src), "r"(bytes) : "memory");
}

// --------------------------------------------------- programmatic dependent launch

__device__ __forceinline__ void pdl_wait() { asm volatile("griddepcontrol.wait;" ::: "memory"); }
__device__ __forceinline__ void pdl_trigger() {
    asm volatile("griddepcontrol.launch_dependents;" ::: "memory");
}

// ------------------------------------------------------------------- clusters

__device__ __forceinline__ void cluster_sync() {
    asm volatile("barrier.cluster.arrive.release.aligned;\n\t"
                 "barrier.cluster.wait.acquire.aligned;" ::: "memory");
}

// Address of `p` (this CTA's shared memory) in the shared memory of cluster CTA `rank`.
__device__ __forceinline__ uint32_t map_to_rank(const void *p, uint32_t rank) {
    uint32_t r;
    asm volatile("mapa.shared::cluster.u32 %0, %1, %2;" : "=r"(r) : "r"(smem_u32(p)), "r"(rank));
    return r;
}

__device__ __forceinline__ float ld_cluster_f32(uint32_t addr) {
    float v;
    asm volatile("ld.shared::cluster.f32 %0, [%1];" : "=f"(v) : "r"(addr) : "memory");
    return v;
}

// ------------------------------------------------------------------- bf16 / MMA

__device__ __forceinline__ uint32_t bf16x2_mul(uint32_t a, uint32_t b) {
    uint32_t d;
    asm("mul.rn.bf16x2 %0, %1, %2;" : "=r"(d) : "r"(a), "r"(b));
    return d;
}

__device__ __forceinline__ uint16_t f32_to_bf16_rn(float f) {
    uint16_t h;
    asm("cvt.rn.bf16.f32 %0, %1;" : "=h"(h) : "f"(f));
    return h;
}

// D += A * B for one m16n8k16 tile: A bf16 16x16 (row), B bf16 16x8 (col), fp32 acc.
__device__ __forceinline__ void mma_bf16_16816(float (&c)[4], uint32_t a0, uint32_t a1,
                                               uint32_t a2, uint32_t a3, uint32_t b0,
                                               uint32_t b1) {
    asm volatile(
        "mma.sync.aligned.m16n8k16.row.col.f32.bf16.bf16.f32 "
        "{%0,%1,%2,%3}, {%4,%5,%6,%7}, {%8,%9}, {%0,%1,%2,%3};"
        : "+f"(c[0]), "+f"(c[1]), "+f"(c[2]), "+f"(c[3])
        : "r"(a0), "r"(a1), "r"(a2), "r"(a3), "r"(b0), "r"(b1));
}

// --------------------------------------------------- exact e4m3 -> bf16 rebuild
//
// For an e4m3 byte b = s.EEEE.MMM, the 16-bit pattern s.0000.EEEE.MMM.0000 read as
// bf16 is exactly e4m3(b) * 2^-120, subnormals included (bf16 has 8 exponent bits, so
// the e4m3 exponent field lands in its low four bits, and an e4m3 subnormal becomes a
// bf16 subnormal with the same mantissa).  One bf16 multiply by 2^(e-7) then gives
// bf16(e4m3(b) * 2^(e-127)) with a single rounding -- exactly the rule
// bf16(float(q) * 2^(e-127)) -- as long as 2^(e-7) is a bf16 number, i.e. e <= 134.
// Above that the value e4m3(b) is first restored exactly (times 2^120) and then scaled
// by 2^(e-127) (byte 255: the +inf pattern 0x7F80, as 2^128 overflows), which can
// only round at overflow.  The byte pattern 0x7F/0xFF (e4m3 NaN) is patched to NaN.

struct Scale {
    uint32_t s1;  // first bf16x2 multiplier
    uint32_t s2;  // second multiplier (used when two != 0)
    uint32_t two;
};

__device__ __forceinline__ Scale make_scale(uint32_t e_byte) {
    Scale s;
    if (e_byte <= 134u) {
        const uint32_t b = (e_byte + 120u) << 7;  // bf16 pattern of 2^(e-7)
        s.s1 = b | (b << 16);
        s.s2 = 0u;
        s.two = 0u;
    } else {
        s.s1 = 0x7B807B80u;                       // 2^120
        const uint32_t b = e_byte << 7;           // 2^(e-127); 255 -> +inf
        s.s2 = b | (b << 16);
        s.two = 1u;
    }
    return s;
}

// Four codes packed in w (byte i = code i) -> lo = bf16x2(code0, code1),
// hi = bf16x2(code2, code3), each scaled as above.  NaN codes are not handled here.
__device__ __forceinline__ void rebuild4(uint32_t w, const Scale &s, uint32_t &lo, uint32_t &hi) {
    uint32_t t0, t1;
    // byte pattern [sx(b1), b1, sx(b0), b0]: after << 4 the sign copy of each code sits
    // on bit 15 of its half and the magnitude on bits 10..4.
    asm("prmt.b32 %0, %1, 0, 0x9180;" : "=r"(t0) : "r"(w));
    asm("prmt.b32 %0, %1, 0, 0xB3A2;" : "=r"(t1) : "r"(w));
    t0 = (t0 << 4) & 0x87F087F0u;
    t1 = (t1 << 4) & 0x87F087F0u;
    lo = bf16x2_mul(t0, s.s1);
    hi = bf16x2_mul(t1, s.s1);
    if (s.two) {
        lo = bf16x2_mul(lo, s.s2);
        hi = bf16x2_mul(hi, s.s2);
    }
}

// Non-zero iff some byte of w is 0x7F or 0xFF (an e4m3 NaN code).
__device__ __forceinline__ uint32_t nan_code_mask(uint32_t w) {
    return ((w & 0x7F7F7F7Fu) + 0x01010101u) & 0x80808080u;
}

// Puts a quiet NaN into every half of (lo, hi) whose code in w is an e4m3 NaN
// (returned as .x = lo, .y = hi).  Kept out of line: it only runs when a NaN code is
// present.
static __device__ __noinline__ uint2 patch_nan_codes_impl(uint32_t w, uint32_t lo, uint32_t hi) {
    const uint32_t m = nan_code_mask(w);
    if (m & 0x00000080u) lo = (lo & 0xFFFF0000u) | 0x7FC0u;
    if (m & 0x00008000u) lo = (lo & 0x0000FFFFu) | 0x7FC00000u;
    if (m & 0x00800000u) hi = (hi & 0xFFFF0000u) | 0x7FC0u;
    if (m & 0x80000000u) hi = (hi & 0x0000FFFFu) | 0x7FC00000u;
    return make_uint2(lo, hi);
}

__device__ __forceinline__ void patch_nan_codes(uint32_t w, uint32_t &lo, uint32_t &hi) {
    const uint2 r = patch_nan_codes_impl(w, lo, hi);
    lo = r.x;
    hi = r.y;
}

}  // namespace bsf8
