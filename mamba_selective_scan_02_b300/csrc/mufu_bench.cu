// mufu_bench.cu — MUFU ex2 throughput kernel, the exponential half of the
// scan's roofline (one Ā = exp(Δ·A) per channel, state and token).
//
// Each thread runs 16 independent chains x ← 2^{-x} (x stays in (0.5, 1)), so
// the only work is ex2.approx.ftz.f32 issue; one float per thread is written so
// the chains stay live.  Count = blocks × 256 × iters × 16 exponentials.
#include "ssm_device.cuh"
#include "ssm_internal.h"

namespace ssm {

__global__ void __launch_bounds__(256) mufu_ex2_kernel(float *sink, int iters) {
    float x[16];
#pragma unroll
    for (int i = 0; i < 16; ++i) x[i] = 0.5f + 0.01f * (float)((threadIdx.x + i) & 31);
    for (int it = 0; it < iters; ++it) {
#pragma unroll
        for (int i = 0; i < 16; ++i) x[i] = ex2(-x[i]);
    }
    float s = 0.f;
#pragma unroll
    for (int i = 0; i < 16; ++i) s += x[i];
    sink[(size_t)blockIdx.x * blockDim.x + threadIdx.x] = s;
}

cudaError_t mufu_ex2_launch(float *sink, int blocks, int iters, cudaStream_t st) {
    mufu_ex2_kernel<<<blocks, 256, 0, st>>>(sink, iters);
    return cudaGetLastError();
}

}  // namespace ssm
