// ssm_internal.h — argument structs shared by the C-ABI layer and the kernels.
#pragma once

#include <cuda_runtime.h>
#include <stdint.h>

namespace ssm {

// Validated, device-side view of one forward scan (sizes fit in int32).
struct ScanArgs {
    int batch, dim, dstate, seqlen;
    const void *u, *delta, *z, *B, *C;
    const float *A, *Dskip, *bias;
    int delta_softplus;
    const float *h0;
    void *y;
    float *hL;
    float2 *agg;     // [b][D][K-1][N] (Π Ā, h_end from zero) per chunk
    float *carry;    // [b][D][K][N] state entering chunk k
    int *status;     // device status word (0 = ok)
    int chunk_len;   // tokens per chunk (multiple of 64)
    int nchunks;     // K
};

struct StepArgs {
    int batch, dim, dstate;
    float *state;
    const void *u, *delta, *z, *B, *C;
    const float *A, *Dskip, *bias;
    int delta_softplus;
    void *y;
};

int scan_groups(int64_t dstate);
int64_t scan_chunk_len(int64_t batch, int64_t dim, int64_t dstate, int64_t seqlen, int64_t requested);
cudaError_t scan_launch(const ScanArgs &a, bool bf16, cudaStream_t stream);
cudaError_t step_launch(const StepArgs &a, bool bf16, cudaStream_t stream);
cudaError_t mufu_ex2_launch(float *sink, int blocks, int iters, cudaStream_t stream);

}  // namespace ssm
