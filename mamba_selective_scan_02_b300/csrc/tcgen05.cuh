// tcgen05.cuh — inline-PTX wrappers for the sm_100-family tensor-core path:
// tensor memory (TMEM) allocation, register <-> TMEM copies, the MMA issued by
// one thread with its shared-memory operand descriptor and instruction
// descriptor, and completion tracking through an mbarrier.
#pragma once

#include <stdint.h>

#include "ssm_device.cuh"

namespace ssm {
namespace tc {

// TMEM address: lane in bits 31..16, column in bits 15..0.
__device__ __forceinline__ uint32_t taddr(uint32_t base, uint32_t lane, uint32_t col) {
    return base + (lane << 16) + col;
}

// Allocates `ncols` (a power of two >= 32) TMEM columns for this CTA; one warp
// executes it and the base address lands in shared memory at `dst`.
__device__ __forceinline__ void alloc(uint32_t *dst, uint32_t ncols) {
    asm volatile("tcgen05.alloc.cta_group::1.sync.aligned.shared::cta.b32 [%0], %1;" ::"r"(smem_u32(dst)),
                 "r"(ncols)
                 : "memory");
    asm volatile("tcgen05.relinquish_alloc_permit.cta_group::1.sync.aligned;" ::: "memory");
}
__device__ __forceinline__ void dealloc(uint32_t base, uint32_t ncols) {
    asm volatile("tcgen05.dealloc.cta_group::1.sync.aligned.b32 %0, %1;" ::"r"(base), "r"(ncols) : "memory");
}

__device__ __forceinline__ void fence_before_sync() {
    asm volatile("tcgen05.fence::before_thread_sync;" ::: "memory");
}
__device__ __forceinline__ void fence_after_sync() {
    asm volatile("tcgen05.fence::after_thread_sync;" ::: "memory");
}

// Eight 32-bit columns per lane of the warp's 32-lane quarter (shape 32x32b):
// thread i writes TMEM lane (lane field of `ta`) + i, columns col .. col+7.
__device__ __forceinline__ void st8(uint32_t ta, const float *v) {
    asm volatile(
        "tcgen05.st.sync.aligned.32x32b.x8.b32 [%0], {%1, %2, %3, %4, %5, %6, %7, %8};" ::"r"(ta),
        "f"(v[0]), "f"(v[1]), "f"(v[2]), "f"(v[3]), "f"(v[4]), "f"(v[5]), "f"(v[6]), "f"(v[7])
        : "memory");
}
__device__ __forceinline__ void st8(uint32_t ta, float2 a, float2 b, float2 c, float2 d) {
    asm volatile(
        "tcgen05.st.sync.aligned.32x32b.x8.b32 [%0], {%1, %2, %3, %4, %5, %6, %7, %8};" ::"r"(ta),
        "f"(a.x), "f"(a.y), "f"(b.x), "f"(b.y), "f"(c.x), "f"(c.y), "f"(d.x), "f"(d.y)
        : "memory");
}
// Four 32-bit columns per lane (32x32b shape).
__device__ __forceinline__ void st4(uint32_t ta, uint32_t a, uint32_t b, uint32_t c, uint32_t d) {
    asm volatile("tcgen05.st.sync.aligned.32x32b.x4.b32 [%0], {%1, %2, %3, %4};" ::"r"(ta), "r"(a), "r"(b), "r"(c),
                 "r"(d)
                 : "memory");
}
// Two 32-bit columns per lane (32x32b shape).
__device__ __forceinline__ void st2(uint32_t ta, uint32_t a, uint32_t b) {
    asm volatile("tcgen05.st.sync.aligned.32x32b.x2.b32 [%0], {%1, %2};" ::"r"(ta), "r"(a), "r"(b) : "memory");
}
__device__ __forceinline__ void wait_st() { asm volatile("tcgen05.wait::st.sync.aligned;" ::: "memory"); }

__device__ __forceinline__ void ld8(uint32_t ta, float *v) {
    uint32_t r[8];
    asm volatile("tcgen05.ld.sync.aligned.32x32b.x8.b32 {%0, %1, %2, %3, %4, %5, %6, %7}, [%8];"
                 : "=r"(r[0]), "=r"(r[1]), "=r"(r[2]), "=r"(r[3]), "=r"(r[4]), "=r"(r[5]), "=r"(r[6]), "=r"(r[7])
                 : "r"(ta)
                 : "memory");
    asm volatile("tcgen05.wait::ld.sync.aligned;" ::: "memory");
#pragma unroll
    for (int i = 0; i < 8; ++i) v[i] = __uint_as_float(r[i]);
}

// The same load without the wait: the registers are valid after wait_ld().
__device__ __forceinline__ void ld8_nowait(uint32_t ta, uint32_t *r) {
    asm volatile("tcgen05.ld.sync.aligned.32x32b.x8.b32 {%0, %1, %2, %3, %4, %5, %6, %7}, [%8];"
                 : "=r"(r[0]), "=r"(r[1]), "=r"(r[2]), "=r"(r[3]), "=r"(r[4]), "=r"(r[5]), "=r"(r[6]), "=r"(r[7])
                 : "r"(ta)
                 : "memory");
}
__device__ __forceinline__ void wait_ld() { asm volatile("tcgen05.wait::ld.sync.aligned;" ::: "memory"); }

// Shared-memory operand descriptor, K-major, no swizzle: 8-row × 16-byte core
// matrices, `lbo` bytes apart along K and `sbo` bytes apart along M / N.
__device__ __forceinline__ uint64_t desc_kmajor(uint32_t saddr, uint32_t lbo, uint32_t sbo) {
    return (uint64_t)((saddr & 0x3FFFF) >> 4) | ((uint64_t)(lbo >> 4) << 16) | ((uint64_t)(sbo >> 4) << 32) |
           (1ull << 46);  // descriptor version of the sm_100 family
}

// Instruction descriptor: fp32 accumulator, tf32 A and B, both K-major, M × N.
__host__ __device__ constexpr uint32_t idesc_tf32(uint32_t M, uint32_t N) {
    return (1u << 4) | (2u << 7) | (2u << 10) | ((N >> 3) << 17) | ((M >> 4) << 24);
}

// Instruction descriptor: fp32 accumulator, f16 A and B, both K-major, M × N.
__host__ __device__ constexpr uint32_t idesc_f16(uint32_t M, uint32_t N) {
    return (1u << 4) | (0u << 7) | (0u << 10) | ((N >> 3) << 17) | ((M >> 4) << 24);
}

// D (TMEM) (+)= A (TMEM) · B (shared memory), kind::f16 (K = 16), issued by one thread.
__device__ __forceinline__ void mma_f16_ts(uint32_t d, uint32_t a, uint64_t bdesc, uint32_t idesc, bool acc) {
    asm volatile(
        "{\n\t.reg .pred p;\n\tsetp.ne.b32 p, %4, 0;\n\t"
        "tcgen05.mma.cta_group::1.kind::f16 [%0], [%1], %2, %3, p;\n\t}" ::"r"(d),
        "r"(a), "l"(bdesc), "r"(idesc), "r"((uint32_t)acc)
        : "memory");
}

// D (TMEM) (+)= A (TMEM) · B (shared memory), kind::tf32, issued by one thread.
__device__ __forceinline__ void mma_tf32_ts(uint32_t d, uint32_t a, uint64_t bdesc, uint32_t idesc, bool acc) {
    asm volatile(
        "{\n\t.reg .pred p;\n\tsetp.ne.b32 p, %4, 0;\n\t"
        "tcgen05.mma.cta_group::1.kind::tf32 [%0], [%1], %2, %3, p;\n\t}" ::"r"(d),
        "r"(a), "l"(bdesc), "r"(idesc), "r"((uint32_t)acc)
        : "memory");
}

// The 8 MMAs of one read-out block, issued by one elected lane of the calling
// warp (all lanes execute the operand arithmetic, so it stays warp-uniform):
// D (TMEM, columns d ..) = Σ_j A_j · B_j with A_j at TMEM columns a + 8·j
// (16 f16 values of K per lane) and B_j the shared-memory operand whose
// descriptor is bdesc + j·(256 B >> 4); the first MMA overwrites D.  Then one
// commit arrives on each of `bar0` and `bar1` when the MMAs are complete.
__device__ __forceinline__ void mma8_f16_ts_commit2(uint32_t d, uint32_t a, uint64_t bdesc, uint32_t idesc,
                                                    uint64_t *bar0, uint64_t *bar1) {
    asm volatile(
        "{\n\t.reg .pred e;\n\t.reg .b32 a1, a2, a3, a4, a5, a6, a7;\n\t"
        ".reg .b64 b1, b2, b3, b4, b5, b6, b7;\n\t"
        "add.u32 a1, %1, 8;\n\tadd.u32 a2, %1, 16;\n\tadd.u32 a3, %1, 24;\n\tadd.u32 a4, %1, 32;\n\t"
        "add.u32 a5, %1, 40;\n\tadd.u32 a6, %1, 48;\n\tadd.u32 a7, %1, 56;\n\t"
        "add.u64 b1, %2, 16;\n\tadd.u64 b2, %2, 32;\n\tadd.u64 b3, %2, 48;\n\tadd.u64 b4, %2, 64;\n\t"
        "add.u64 b5, %2, 80;\n\tadd.u64 b6, %2, 96;\n\tadd.u64 b7, %2, 112;\n\t"
        "elect.sync _|e, 0xffffffff;\n\t"
        "@e tcgen05.mma.cta_group::1.kind::f16 [%0], [%1], %2, %3, 0;\n\t"
        "@e tcgen05.mma.cta_group::1.kind::f16 [%0], [a1], b1, %3, 1;\n\t"
        "@e tcgen05.mma.cta_group::1.kind::f16 [%0], [a2], b2, %3, 1;\n\t"
        "@e tcgen05.mma.cta_group::1.kind::f16 [%0], [a3], b3, %3, 1;\n\t"
        "@e tcgen05.mma.cta_group::1.kind::f16 [%0], [a4], b4, %3, 1;\n\t"
        "@e tcgen05.mma.cta_group::1.kind::f16 [%0], [a5], b5, %3, 1;\n\t"
        "@e tcgen05.mma.cta_group::1.kind::f16 [%0], [a6], b6, %3, 1;\n\t"
        "@e tcgen05.mma.cta_group::1.kind::f16 [%0], [a7], b7, %3, 1;\n\t"
        "@e tcgen05.commit.cta_group::1.mbarrier::arrive::one.shared::cluster.b64 [%4];\n\t"
        "@e tcgen05.commit.cta_group::1.mbarrier::arrive::one.shared::cluster.b64 [%5];\n\t}" ::"r"(d),
        "r"(a), "l"(bdesc), "r"(idesc), "r"(smem_u32(bar0)), "r"(smem_u32(bar1))
        : "memory");
}

// Arrives once on `bar` when every tcgen05 operation this thread issued so far
// has completed.
__device__ __forceinline__ void commit(uint64_t *bar) {
    asm volatile("tcgen05.commit.cta_group::1.mbarrier::arrive::one.shared::cluster.b64 [%0];" ::"r"(
                     smem_u32(bar))
                 : "memory");
}

}  // namespace tc
}  // namespace ssm
