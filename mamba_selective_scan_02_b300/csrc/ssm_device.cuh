// ssm_device.cuh — device helpers shared by the scan and decode kernels of
// libssmscan (sm_103a): MUFU wrappers, the step-size and gate nonlinearities,
// I/O conversions, and the mbarrier / TMA (cp.async.bulk.tensor) primitives.
#pragma once

#include <cuda.h>
#include <cuda_bf16.h>
#include <cuda_runtime.h>
#include <stdint.h>

namespace ssm {

constexpr float kLog2e = 1.4426950408889634f;
constexpr float kLn2 = 0.6931471805599453f;

// ---------------------------------------------------------------- MUFU
__device__ __forceinline__ float ex2(float x) {
    float y;
    asm("ex2.approx.ftz.f32 %0, %1;" : "=f"(y) : "f"(x));
    return y;
}
__device__ __forceinline__ float lg2(float x) {
    float y;
    asm("lg2.approx.ftz.f32 %0, %1;" : "=f"(y) : "f"(x));
    return y;
}
__device__ __forceinline__ float tanh_approx(float x) {
    float y;
    asm("tanh.approx.f32 %0, %1;" : "=f"(y) : "f"(x));
    return y;
}
__device__ __forceinline__ float rcp_approx(float x) {
    float y;
    asm("rcp.approx.ftz.f32 %0, %1;" : "=f"(y) : "f"(x));
    return y;
}

// ---------------------------------------------------------------- softplus
// softplus(x) = max(x, 0) + log1p(w), w = e^{-|x|} in (0, 1].
// log1p(w) is a truncated alternating series for w < 1/16 (next term w^7/7,
// relative 4e-9) and ln2·lg2(1 + w) above, where lg2.approx's absolute error
// (~2^-22) is small against log1p(w) >= 0.06.
__device__ __forceinline__ float softplus(float x) {
    const float w = ex2(-fabsf(x) * kLog2e);
    float series = fmaf(w, -1.0f / 6.0f, 1.0f / 5.0f);
    series = fmaf(w, series, -1.0f / 4.0f);
    series = fmaf(w, series, 1.0f / 3.0f);
    series = fmaf(w, series, -1.0f / 2.0f);
    series = fmaf(w, series, 1.0f);
    series *= w;
    const float viaLog = lg2(1.0f + w) * kLn2;
    return fmaxf(x, 0.0f) + (w < 0.0625f ? series : viaLog);
}

// silu(z) = z·σ(z).  Accurate form (fp32 I/O): z / (1 + 2^{-z·log2e}).
__device__ __forceinline__ float silu_accurate(float z) {
    return z * rcp_approx(1.0f + ex2(-z * kLog2e));
}
// Fast form (bf16 I/O): σ(z) = ½ + ½·tanh(z/2); tanh.approx has ~2^-11 relative
// error, far below the bf16 rounding of the output.
__device__ __forceinline__ float silu_fast(float z) {
    const float hz = 0.5f * z;
    return fmaf(hz, tanh_approx(hz), hz);
}

// ---------------------------------------------------------------- I/O types
template <typename T> struct IO;
template <> struct IO<float> {
    __device__ __forceinline__ static float to_f(float v) { return v; }
    __device__ __forceinline__ static float from_f(float v) { return v; }
    static constexpr bool kFastGate = false;
};
template <> struct IO<__nv_bfloat16> {
    __device__ __forceinline__ static float to_f(__nv_bfloat16 v) { return __bfloat162float(v); }
    __device__ __forceinline__ static __nv_bfloat16 from_f(float v) { return __float2bfloat16_rn(v); }
    static constexpr bool kFastGate = true;
};

template <typename T>
__device__ __forceinline__ float gate_of(float z) {
    return IO<T>::kFastGate ? silu_fast(z) : silu_accurate(z);
}

// ---------------------------------------------------------------- mbarrier / TMA
__device__ __forceinline__ uint32_t smem_u32(const void *p) {
    return static_cast<uint32_t>(__cvta_generic_to_shared(p));
}
__device__ __forceinline__ void mbar_init(uint64_t *bar, uint32_t count) {
    asm volatile("mbarrier.init.shared::cta.b64 [%0], %1;" ::"r"(smem_u32(bar)), "r"(count));
}
__device__ __forceinline__ void fence_mbar_init() {
    asm volatile("fence.mbarrier_init.release.cluster;" ::: "memory");
}
__device__ __forceinline__ void fence_proxy_async_smem() {
    asm volatile("fence.proxy.async.shared::cta;" ::: "memory");
}
__device__ __forceinline__ void mbar_arrive_expect_tx(uint64_t *bar, uint32_t bytes) {
    asm volatile("mbarrier.arrive.expect_tx.shared::cta.b64 _, [%0], %1;" ::"r"(smem_u32(bar)),
                 "r"(bytes)
                 : "memory");
}
__device__ __forceinline__ bool mbar_try_wait(uint64_t *bar, uint32_t parity) {
    uint32_t ok;
    asm volatile(
        "{\n\t.reg .pred p;\n\t"
        "mbarrier.try_wait.parity.shared::cta.b64 p, [%1], %2;\n\t"
        "selp.u32 %0, 1, 0, p;\n\t}"
        : "=r"(ok)
        : "r"(smem_u32(bar)), "r"(parity)
        : "memory");
    return ok != 0;
}
// Bounded wait: gives up after `limit` polls (each poll may itself suspend for
// a hardware-defined interval).  Returns false when the limit ran out.
__device__ __forceinline__ bool mbar_wait_bounded(uint64_t *bar, uint32_t parity, uint32_t limit) {
    for (uint32_t i = 0; i < limit; ++i)
        if (mbar_try_wait(bar, parity)) return true;
    return false;
}
__device__ __forceinline__ void tma_load_3d(void *dst, const CUtensorMap *map, uint64_t *bar,
                                            int c0, int c1, int c2) {
    asm volatile(
        "cp.async.bulk.tensor.3d.shared::cluster.global.tile.mbarrier::complete_tx::bytes"
        " [%0], [%1, {%2, %3, %4}], [%5];" ::"r"(smem_u32(dst)),
        "l"(reinterpret_cast<uint64_t>(map)), "r"(c0), "r"(c1), "r"(c2), "r"(smem_u32(bar))
        : "memory");
}
__device__ __forceinline__ void tma_store_3d(const CUtensorMap *map, const void *src, int c0, int c1,
                                             int c2) {
    asm volatile("cp.async.bulk.tensor.3d.global.shared::cta.tile.bulk_group [%0, {%1, %2, %3}], [%4];" ::"l"(
                     reinterpret_cast<uint64_t>(map)),
                 "r"(c0), "r"(c1), "r"(c2), "r"(smem_u32(src))
                 : "memory");
}
__device__ __forceinline__ void bulk_commit() { asm volatile("cp.async.bulk.commit_group;" ::: "memory"); }
__device__ __forceinline__ void bulk_wait_read0() {
    asm volatile("cp.async.bulk.wait_group.read 0;" ::: "memory");
}
__device__ __forceinline__ void bulk_wait0() { asm volatile("cp.async.bulk.wait_group 0;" ::: "memory"); }

// Records the first device-side error in the workspace status word.
__device__ __forceinline__ void record_error(int *status, int code) {
    if (status) atomicCAS(status, 0, code);
}

}  // namespace ssm
