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

// log1p(w) for w in [0, 1] on the FMA pipe only: w·q(w), q of degree 7 fitted
// to log1p(w)/w towards minimax relative error (csrc/fit_log1p.py prints the
// coefficients); relative error 3.7e-7 in fp32.
__device__ __forceinline__ float log1p_unit(float w) {
    float q = fmaf(w, -0.008539210073649883f, 0.04408963769674301f);
    q = fmaf(w, q, -0.10768172144889832f);
    q = fmaf(w, q, 0.17745241522789001f);
    q = fmaf(w, q, -0.24495463073253632f);
    q = fmaf(w, q, 0.33275479078292847f);
    q = fmaf(w, q, -0.4999740421772003f);
    q = fmaf(w, q, 0.9999998211860657f);
    return w * q;
}
// Branch-free softplus, one MUFU op: max(x, 0) + log1p(e^{-|x|}).
__device__ __forceinline__ float softplus_poly(float x) {
    return fmaxf(x, 0.0f) + log1p_unit(ex2(-fabsf(x) * kLog2e));
}
// Two MUFU ops, four FMA-pipe ops: log1p(w) = ln2·lg2(1 + w).  The rounding of
// 1 + w and lg2.approx leave an absolute error near 2e-7 in Δ, far below the
// bf16 rounding of the inputs it is used with.
__device__ __forceinline__ float softplus_mufu(float x) {
    const float w = ex2(-fabsf(x) * kLog2e);
    return fmaf(lg2(1.0f + w), kLn2, fmaxf(x, 0.0f));
}

// Exact zero-order hold: B̄ = (e^{ΔA} − 1)/A · B = Δ·φ(x)·B with x = Δ·A and
// φ(x) = (e^x − 1)/x ("Discretisation: zero-order hold", first-principles page).
// φ is a Taylor polynomial for |x| < 1/8 (next term x^6/5040 < 8e-11), where
// e^x − 1 would cancel, and (Ā − 1)/x above; `abar` is e^x already computed.
__device__ __forceinline__ float zoh_phi(float x, float abar) {
    float p = fmaf(x, 1.0f / 720.0f, 1.0f / 120.0f);
    p = fmaf(x, p, 1.0f / 24.0f);
    p = fmaf(x, p, 1.0f / 6.0f);
    p = fmaf(x, p, 0.5f);
    p = fmaf(x, p, 1.0f);
    return fabsf(x) < 0.125f ? p : __fdividef(abar - 1.0f, x);
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
    // 8 consecutive values from shared memory (16-byte aligned) to fp32.
    __device__ __forceinline__ static void load8(const float *p, float *o) {
        const float4 a = reinterpret_cast<const float4 *>(p)[0], b = reinterpret_cast<const float4 *>(p)[1];
        o[0] = a.x; o[1] = a.y; o[2] = a.z; o[3] = a.w; o[4] = b.x; o[5] = b.y; o[6] = b.z; o[7] = b.w;
    }
    __device__ __forceinline__ static float4 load4(const float *p) { return *reinterpret_cast<const float4 *>(p); }
    __device__ __forceinline__ static void store2(float *p, float2 v) { *reinterpret_cast<float2 *>(p) = v; }
    __device__ __forceinline__ static float softplus(float x) { return softplus_poly(x); }
};
template <> struct IO<__nv_bfloat16> {
    __device__ __forceinline__ static float to_f(__nv_bfloat16 v) { return __bfloat162float(v); }
    __device__ __forceinline__ static __nv_bfloat16 from_f(float v) { return __float2bfloat16_rn(v); }
    static constexpr bool kFastGate = true;
    __device__ __forceinline__ static float lo(uint32_t w) { return __uint_as_float(w << 16); }
    __device__ __forceinline__ static float hi(uint32_t w) { return __uint_as_float(w & 0xffff0000u); }
    __device__ __forceinline__ static void load8(const __nv_bfloat16 *p, float *o) {
        const uint4 v = *reinterpret_cast<const uint4 *>(p);
        o[0] = lo(v.x); o[1] = hi(v.x); o[2] = lo(v.y); o[3] = hi(v.y);
        o[4] = lo(v.z); o[5] = hi(v.z); o[6] = lo(v.w); o[7] = hi(v.w);
    }
    __device__ __forceinline__ static float4 load4(const __nv_bfloat16 *p) {
        const uint2 v = *reinterpret_cast<const uint2 *>(p);
        return make_float4(lo(v.x), hi(v.x), lo(v.y), hi(v.y));
    }
    __device__ __forceinline__ static void store2(__nv_bfloat16 *p, float2 v) {
        *reinterpret_cast<__nv_bfloat162 *>(p) = __floats2bfloat162_rn(v.x, v.y);
    }
    __device__ __forceinline__ static float softplus(float x) { return softplus_mufu(x); }
};

template <typename T>
__device__ __forceinline__ float gate_of(float z) {
    return IO<T>::kFastGate ? silu_fast(z) : silu_accurate(z);
}
// silu of two values; the fast form runs its multiply-adds packed.
template <typename T>
__device__ __forceinline__ float2 gate2(float2 z) {
    if (IO<T>::kFastGate) {
        const float2 hz = __fmul2_rn(z, make_float2(0.5f, 0.5f));
        return __ffma2_rn(hz, make_float2(tanh_approx(hz.x), tanh_approx(hz.y)), hz);
    }
    return make_float2(silu_accurate(z.x), silu_accurate(z.y));
}

// ---------------------------------------------------------------- mbarrier / TMA
__device__ __forceinline__ uint32_t smem_u32(const void *p) {
    return static_cast<uint32_t>(__cvta_generic_to_shared(p));
}
__device__ __forceinline__ void mbar_init(uint64_t *bar, uint32_t count) {
    asm volatile("mbarrier.init.shared::cta.b64 [%0], %1;" ::"r"(smem_u32(bar)), "r"(count));
}
// Ends an mbarrier's life so that the location can be initialised again;
// nothing may be pending on it (no waiter, no transaction in flight).
__device__ __forceinline__ void mbar_inval(uint64_t *bar) {
    asm volatile("mbarrier.inval.shared::cta.b64 [%0];" ::"r"(smem_u32(bar)) : "memory");
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
// Untiled bulk copies: both addresses 16-byte aligned, size a multiple of 16.
__device__ __forceinline__ void bulk_load(void *dst, const void *src, uint32_t bytes, uint64_t *bar) {
    asm volatile("cp.async.bulk.shared::cluster.global.mbarrier::complete_tx::bytes [%0], [%1], %2, [%3];" ::"r"(
                     smem_u32(dst)),
                 "l"(reinterpret_cast<uint64_t>(src)), "r"(bytes), "r"(smem_u32(bar))
                 : "memory");
}
__device__ __forceinline__ void bulk_store(void *dst, const void *src, uint32_t bytes) {
    asm volatile("cp.async.bulk.global.shared::cta.bulk_group [%0], [%1], %2;" ::"l"(reinterpret_cast<uint64_t>(dst)),
                 "r"(smem_u32(src)), "r"(bytes)
                 : "memory");
}
// Waits until at most two committed bulk groups are still reading shared memory.
__device__ __forceinline__ void bulk_wait_read2() {
    asm volatile("cp.async.bulk.wait_group.read 2;" ::: "memory");
}
__device__ __forceinline__ void bulk_commit() { asm volatile("cp.async.bulk.commit_group;" ::: "memory"); }
__device__ __forceinline__ void bulk_wait_read0() {
    asm volatile("cp.async.bulk.wait_group.read 0;" ::: "memory");
}
// Waits until at most one committed bulk group is still reading shared memory.
__device__ __forceinline__ void bulk_wait_read1() {
    asm volatile("cp.async.bulk.wait_group.read 1;" ::: "memory");
}
__device__ __forceinline__ void bulk_wait0() { asm volatile("cp.async.bulk.wait_group 0;" ::: "memory"); }

// ---------------------------------------------------------------- debug build
// Built with -DSSM_DEBUG, every global store checks its element range against
// the buffer it writes: a range outside is skipped and recorded (the first one
// wins) in this source file's debug word, which the host reads through
// ssm_debug_status.  Without SSM_DEBUG the check is `true` and compiles away.
#ifdef SSM_DEBUG
static __device__ int g_ssm_debug_word;
#endif
__device__ __forceinline__ bool in_range(int64_t first, int64_t count, int64_t size) {
#ifdef SSM_DEBUG
    if (first >= 0 && count >= 0 && first + count <= size) return true;
    atomicCAS(&g_ssm_debug_word, 0, 5);   // SSM_ERR_BOUNDS
    return false;
#else
    (void)first, (void)count, (void)size;
    return true;
#endif
}
// Defines `int NAME(bool reset)`, the host's reader of this source file's debug
// word (always 0 without SSM_DEBUG).
#ifdef SSM_DEBUG
#define SSM_DEBUG_WORD_READER(NAME)                                              \
    int NAME(bool reset) {                                                       \
        int v = 0;                                                               \
        if (cudaMemcpyFromSymbol(&v, g_ssm_debug_word, sizeof(int)) != cudaSuccess) return -1; \
        if (reset) {                                                             \
            const int z = 0;                                                     \
            if (cudaMemcpyToSymbol(g_ssm_debug_word, &z, sizeof(int)) != cudaSuccess) return -1; \
        }                                                                        \
        return v;                                                                \
    }
#else
#define SSM_DEBUG_WORD_READER(NAME) \
    int NAME(bool) { return 0; }
#endif

// Records the first device-side error in the workspace status word.
__device__ __forceinline__ void record_error(int *status, int code) {
    if (status) atomicCAS(status, 0, code);
}

// ---------------------------------------------------------------- chained hand-offs
// A work item publishes "chunks done" with a release store after writing its
// state; the item that continues from it waits with acquire loads.
__device__ __forceinline__ int flag_acquire(const int *p) {
    int v;
    asm volatile("ld.acquire.gpu.global.b32 %0, [%1];" : "=r"(v) : "l"(p) : "memory");
    return v;
}
__device__ __forceinline__ void flag_release(int *p, int v) {
    asm volatile("st.release.gpu.global.b32 [%0], %1;" ::"l"(p), "r"(v) : "memory");
}
// Polls *flag until it reaches `target`, sleeping between polls, at most
// `limit` polls.  Returns false if it gave up; callers record SSM_ERR_TIMEOUT
// and carry on, so a launch always ends.
__device__ __forceinline__ bool wait_flag(const int *flag, int target, int limit) {
    int polls = 0;
    while (flag_acquire(flag) < target) {
        if (++polls >= limit) return false;
        __nanosleep(64);
    }
    return true;
}

}  // namespace ssm
