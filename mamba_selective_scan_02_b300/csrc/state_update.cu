// state_update.cu — single-token decode step for sm_103a.
//
// The recurrence with L = 1 on a carried state: the state stays a fixed
// b × D × N block however many tokens have been read, and each token folds into
// it at constant cost ("Mamba and selective state spaces, from first
// principles" — "A fixed state against a growing cache"; "State space models
// and Mamba" — "One system, two views", streaming inference).  Decode is bound
// by memory traffic (same page as above), so the kernel is one streaming pass:
// the fp32 state is read once and written once, 16 bytes per thread, fully
// coalesced; the per-channel and per-sequence inputs are a few bytes beside it.
//
// Two thread layouts:
//   * step_wide_kernel (N = 16, 16-byte aligned rows): four lanes per channel,
//     each thread handling four such 16-byte state words one block-width apart,
//     all loaded before any arithmetic, written back with streaming stores.
//   * step_kernel (any N <= 16, any alignment): NG = ceil(N/4) adjacent lanes
//     per channel, lane g owns states 4g .. 4g+3; C·h is summed across the group
//     with xor shuffles.
#include "ssm_device.cuh"
#include "ssm_internal.h"

namespace ssm {

template <typename T, int NG, bool VEC, bool HAS_Z>
__global__ void __launch_bounds__(256) step_kernel(const StepArgs a) {
    const size_t gid = (size_t)blockIdx.x * blockDim.x + threadIdx.x;
    const size_t items = (size_t)a.batch * a.dim * NG;
    // Lanes past the end still take part in the group shuffles below.
    const bool live = gid < items;
    const size_t ch = live ? gid / NG : 0;    // channel index b*D + d
    const int g = (int)(gid % NG);
    const int N = a.dstate;
    const int d = (int)(ch % a.dim);
    const size_t bb = ch / a.dim;

    const T *u = static_cast<const T *>(a.u);
    const T *dl = static_cast<const T *>(a.delta);
    const T *B = static_cast<const T *>(a.B);
    const T *C = static_cast<const T *>(a.C);

    float hv[4] = {0.f, 0.f, 0.f, 0.f};
    float *st = a.state + ch * N + 4 * g;
    // Padded groups (4g >= N) own no state and must not touch the state row.
    const bool own = live && 4 * g < N;
    if (own) {
        if (VEC) {
            const float4 v = *reinterpret_cast<const float4 *>(st);
            hv[0] = v.x; hv[1] = v.y; hv[2] = v.z; hv[3] = v.w;
        } else {
#pragma unroll
            for (int j = 0; j < 4; ++j)
                if (4 * g + j < N) hv[j] = st[j];
        }
    }
    const float uv = live ? IO<T>::to_f(u[ch]) : 0.f;
    float dv = live ? IO<T>::to_f(dl[ch]) + (a.bias ? a.bias[d] : 0.f) : 0.f;
    if (a.delta_softplus) dv = softplus(dv);
    const float du = dv * uv;
    float part = 0.f;
#pragma unroll
    for (int j = 0; j < 4; ++j) {
        const int n = 4 * g + j;
        if (live && n < N) {
            const float abar = ex2(dv * (a.A[(size_t)d * N + n] * kLog2e));
            hv[j] = fmaf(abar, hv[j], IO<T>::to_f(B[bb * N + n]) * du);
            part = fmaf(IO<T>::to_f(C[bb * N + n]), hv[j], part);
        }
    }
#pragma unroll
    for (int m = 1; m < NG; m <<= 1) part += __shfl_xor_sync(0xffffffffu, part, m);
    if (!own) return;
    if (VEC) {
        *reinterpret_cast<float4 *>(st) = make_float4(hv[0], hv[1], hv[2], hv[3]);
    } else {
#pragma unroll
        for (int j = 0; j < 4; ++j)
            if (4 * g + j < N) st[j] = hv[j];
    }
    if (g == 0) {
        float out = part + (a.Dskip ? a.Dskip[d] : 0.f) * uv;
        if (HAS_Z) out *= gate_of<T>(IO<T>::to_f(static_cast<const T *>(a.z)[ch]));
        static_cast<T *>(a.y)[ch] = IO<T>::from_f(out);
    }
}

// Decode with several channels per thread (N = 16, 16-byte aligned rows).
// Four lanes share a channel, each owning four states (one 16-byte word of
// the state row), so every state load and store of a warp covers 512
// contiguous bytes.  Each thread handles IPT such words, IPT × 128 threads
// apart within the block, and issues all of their state loads before any
// arithmetic: that keeps IPT × 16 bytes of state in flight per thread.
constexpr int kStepThreads = 128;
#ifndef SSM_STEP_IPT
#define SSM_STEP_IPT 4
#endif
constexpr int kStepIPT = SSM_STEP_IPT;

template <typename T, bool HAS_Z>
__global__ void __launch_bounds__(kStepThreads) step_wide_kernel(const StepArgs a) {
    const size_t words = (size_t)a.batch * a.dim * 4;  // 16-byte state words
    const size_t base = (size_t)blockIdx.x * (kStepThreads * kStepIPT) + threadIdx.x;
    const int g = threadIdx.x & 3;  // state word within the channel: states 4g .. 4g+3
    const T *Bp = static_cast<const T *>(a.B), *Cp = static_cast<const T *>(a.C);
    const T *up = static_cast<const T *>(a.u), *dp = static_cast<const T *>(a.delta);
    const T *zp = static_cast<const T *>(a.z);
    // Every load of every item is issued before any arithmetic: the state words
    // stream from HBM, the rest comes from L2.
    float4 hv[kStepIPT], av[kStepIPT];
    float bv[kStepIPT][4], cv[kStepIPT][4];
    T uv[kStepIPT], dv[kStepIPT], zv[kStepIPT];
    float bias[kStepIPT], skip[kStepIPT];
#pragma unroll
    for (int i = 0; i < kStepIPT; ++i) {
        const size_t w = base + (size_t)i * kStepThreads;
        const bool live = w < words;
        const size_t ch = live ? w / 4 : 0;  // b·D + d
        const int d = (int)(ch % a.dim);
        const size_t bb = ch / a.dim;
        hv[i] = live ? __ldcs(reinterpret_cast<const float4 *>(a.state) + w) : make_float4(0.f, 0.f, 0.f, 0.f);
        av[i] = __ldg(reinterpret_cast<const float4 *>(a.A + (size_t)d * 16) + g);
        if (sizeof(T) == 2) {
            const uint2 bw = __ldg(reinterpret_cast<const uint2 *>(Bp + bb * 16) + g);
            const uint2 cw = __ldg(reinterpret_cast<const uint2 *>(Cp + bb * 16) + g);
            bv[i][0] = __uint_as_float(bw.x << 16); bv[i][1] = __uint_as_float(bw.x & 0xffff0000u);
            bv[i][2] = __uint_as_float(bw.y << 16); bv[i][3] = __uint_as_float(bw.y & 0xffff0000u);
            cv[i][0] = __uint_as_float(cw.x << 16); cv[i][1] = __uint_as_float(cw.x & 0xffff0000u);
            cv[i][2] = __uint_as_float(cw.y << 16); cv[i][3] = __uint_as_float(cw.y & 0xffff0000u);
        } else {
            const float4 b4 = __ldg(reinterpret_cast<const float4 *>(Bp + bb * 16) + g);
            const float4 c4 = __ldg(reinterpret_cast<const float4 *>(Cp + bb * 16) + g);
            bv[i][0] = b4.x; bv[i][1] = b4.y; bv[i][2] = b4.z; bv[i][3] = b4.w;
            cv[i][0] = c4.x; cv[i][1] = c4.y; cv[i][2] = c4.z; cv[i][3] = c4.w;
        }
        uv[i] = up[ch];
        dv[i] = dp[ch];
        zv[i] = HAS_Z ? zp[ch] : T(0.f);
        bias[i] = a.bias ? __ldg(a.bias + d) : 0.f;
        skip[i] = a.Dskip ? __ldg(a.Dskip + d) : 0.f;
    }
#pragma unroll
    for (int i = 0; i < kStepIPT; ++i) {
        const size_t w = base + (size_t)i * kStepThreads;
        const float u = IO<T>::to_f(uv[i]);
        float delta = IO<T>::to_f(dv[i]) + bias[i];
        if (a.delta_softplus) delta = softplus(delta);
        const float du = delta * u;
        const float avv[4] = {av[i].x, av[i].y, av[i].z, av[i].w};
        float h4[4] = {hv[i].x, hv[i].y, hv[i].z, hv[i].w};
        float part = 0.f;
#pragma unroll
        for (int j = 0; j < 4; ++j) {
            const float abar = ex2(delta * (avv[j] * kLog2e));
            h4[j] = fmaf(abar, h4[j], bv[i][j] * du);
            part = fmaf(cv[i][j], h4[j], part);
        }
        part += __shfl_xor_sync(0xffffffffu, part, 1);
        part += __shfl_xor_sync(0xffffffffu, part, 2);
        if (w >= words) continue;
        __stcs(reinterpret_cast<float4 *>(a.state) + w, make_float4(h4[0], h4[1], h4[2], h4[3]));
        if (g == 0) {
            float out = part + skip[i] * u;
            if (HAS_Z) out *= gate_of<T>(IO<T>::to_f(zv[i]));
            static_cast<T *>(a.y)[w / 4] = IO<T>::from_f(out);
        }
    }
}

namespace {
template <typename T>
cudaError_t wide_dispatch(const StepArgs &a, cudaStream_t st) {
    const size_t words = (size_t)a.batch * a.dim * 4;
    const unsigned blocks = (unsigned)((words + kStepThreads * kStepIPT - 1) / (kStepThreads * kStepIPT));
    if (a.z) step_wide_kernel<T, true><<<blocks, kStepThreads, 0, st>>>(a);
    else step_wide_kernel<T, false><<<blocks, kStepThreads, 0, st>>>(a);
    return cudaGetLastError();
}

template <typename T, int NG>
cudaError_t step_dispatch(const StepArgs &a, cudaStream_t st) {
    const size_t items = (size_t)a.batch * a.dim * NG;
    const unsigned blocks = (unsigned)((items + 255) / 256);
    const bool vec = a.dstate % 4 == 0 && (reinterpret_cast<uintptr_t>(a.state) & 15) == 0;
    const bool z = a.z != nullptr;
    if (vec && z) step_kernel<T, NG, true, true><<<blocks, 256, 0, st>>>(a);
    else if (vec) step_kernel<T, NG, true, false><<<blocks, 256, 0, st>>>(a);
    else if (z) step_kernel<T, NG, false, true><<<blocks, 256, 0, st>>>(a);
    else step_kernel<T, NG, false, false><<<blocks, 256, 0, st>>>(a);
    return cudaGetLastError();
}
template <typename T>
cudaError_t step_ng(const StepArgs &a, cudaStream_t st) {
    switch (scan_groups(a.dstate)) {
        case 1: return step_dispatch<T, 1>(a, st);
        case 2: return step_dispatch<T, 2>(a, st);
        default: return step_dispatch<T, 4>(a, st);
    }
}
}  // namespace

bool aligned16(const void *p) { return (reinterpret_cast<uintptr_t>(p) & 15) == 0; }

cudaError_t step_launch(const StepArgs &a, bool bf16, cudaStream_t st) {
    // The wide kernel reads rows of 16 states as 16-byte words: N = 16 and
    // 16-byte aligned state, A, B and C (a 16-state row is 32 or 64 bytes).
    const bool wide = a.dstate == 16 && aligned16(a.state) && aligned16(a.A) && aligned16(a.B) && aligned16(a.C);
    if (wide) return bf16 ? wide_dispatch<__nv_bfloat16>(a, st) : wide_dispatch<float>(a, st);
    return bf16 ? step_ng<__nv_bfloat16>(a, st) : step_ng<float>(a, st);
}

}  // namespace ssm
