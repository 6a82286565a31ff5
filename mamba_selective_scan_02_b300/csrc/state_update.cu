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
// Thread layout: NG = ceil(N/4) adjacent lanes per channel (b, d), lane g owns
// states 4g .. 4g+3; C·h is summed across the group with xor shuffles.
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

namespace {
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

cudaError_t step_launch(const StepArgs &a, bool bf16, cudaStream_t st) {
    return bf16 ? step_ng<__nv_bfloat16>(a, st) : step_ng<float>(a, st);
}

}  // namespace ssm
