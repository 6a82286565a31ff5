// ssm_internal.h — argument structs shared by the C-ABI layer and the kernels.
#pragma once

#include <cuda.h>
#include <cuda_runtime.h>
#include <stdint.h>

#include <mutex>

namespace ssm {

// One launch-configuration value per device (a kernel's raised dynamic
// shared-memory limit and its occupancy are properties of the kernel on one
// device).  Each launch site keeps one of these as a function-local static;
// the first launch on a device computes that device's value under the lock,
// setting whatever kernel attributes it needs on the way.
class PerDevice {
  public:
    template <typename Fill>
    cudaError_t get(Fill fill, int *out) {
        int dev = 0;
        cudaError_t e = cudaGetDevice(&dev);
        if (e != cudaSuccess) return e;
        if (dev < 0 || dev >= kMaxDevices) return cudaErrorInvalidDevice;
        std::lock_guard<std::mutex> hold(lock_);
        if (!ready_[dev]) {
            int v = 0;
            e = fill(&v);
            if (e != cudaSuccess) return e;
            value_[dev] = v;
            ready_[dev] = true;
        }
        *out = value_[dev];
        return cudaSuccess;
    }

  private:
    static constexpr int kMaxDevices = 64;
    std::mutex lock_;
    int value_[kMaxDevices] = {};
    bool ready_[kMaxDevices] = {};
};

// cuTensorMapEncodeTiled, fetched from the driver once per process (thread
// safe); null when the driver does not provide it.
using TensorMapEncodeFn = CUresult (*)(CUtensorMap *, CUtensorMapDataType, cuuint32_t, void *, const cuuint64_t *,
                                       const cuuint64_t *, const cuuint32_t *, const cuuint32_t *,
                                       CUtensorMapInterleave, CUtensorMapSwizzle, CUtensorMapL2promotion,
                                       CUtensorMapFloatOOBfill);
TensorMapEncodeFn tensor_map_encoder();

// Streaming multiprocessors of the current device (148 on a B300).
inline int sm_count() {
    int dev = 0, sms = 0;
    if (cudaGetDevice(&dev) != cudaSuccess ||
        cudaDeviceGetAttribute(&sms, cudaDevAttrMultiProcessorCount, dev) != cudaSuccess || sms <= 0)
        return 148;
    return sms;
}

// Validated, device-side view of one forward scan (sizes fit in int32).
struct ScanArgs {
    int batch, dim, dstate, seqlen;
    const void *u, *delta, *z, *B, *C;
    const float *A, *Dskip, *bias;
    int delta_softplus;
    int zoh;         // 1: exact zero-order-hold B̄
    const float *h0;
    void *y;
    float *hL;
    float2 *agg;     // look-back: [b][D][K-1][N] (Π Ā, h_end from zero) per chunk
    float *carry;    // look-back: [b][D][K][N], slot k + 1 the state leaving chunk k;
                     // chained: [b][D][N] hand-off
    int *status;     // device status word (0 = ok)
    int *tickets;    // two work counters (main items, aggregate items), zero at launch
    int *flags;      // chained: chunks finished per channel group; look-back: per
                     // (group, chunk) 0 / 1 pair out / 2 leaving state out; zero at launch
    int chunk_len;   // tokens per chunk (multiple of 64)
    int nchunks;     // K
    int groups;      // channel groups: batch × ceil(dim / channels per warp)
    int chained;     // 1: chunk k waits for chunk k-1's state; 0 with K > 1: look-back
    float *Bt, *Ct;  // B and C widened to fp32, token-major: [b][L][np], zero beyond N
    int np;          // states per token row of Bt / Ct (N rounded up to 4, 8 or 16)
    float *ckpt;     // checkpoint launch only: the state at every 16-token tile start,
    int ckpt_tiles;  // [group][tile][2][32 lanes] float4 as the backward's reverse pass reads it
};

// How a scan is cut into work items.  One warp owns a group of channels for
// one chunk of the sequence.  Chained: the chunks of a group run in order,
// each taking the previous one's final state (enough groups to fill the GPU).
// Look-back: every chunk first computes its pair from a zero state, so that
// all chunks run at once and each finds its starting state by composing its
// predecessors' pairs (few groups, long sequences); one launch either way.
struct ScanPlan {
    int np;             // B / C row length after widening (N rounded up to 4, 8 or 16)
    int cpw;            // channels per warp
    int64_t groups;     // batch × ceil(dim / cpw)
    bool chained;
    int64_t chunk_len;  // multiple of 64
    int64_t nchunks;
};

struct StepArgs {
    int batch, dim, dstate;
    float *state;
    const void *u, *delta, *z, *B, *C;
    const float *A, *Dskip, *bias;
    int delta_softplus;
    int zoh;
    void *y;
};

// Backward scan: gradients of the forward scan for upstream dy (and dhL).
struct BwdArgs {
    int batch, dim, dstate, seqlen;
    const void *u, *delta, *z, *B, *C, *dy;
    const float *A, *Dskip, *bias, *h0, *dhL;
    int delta_softplus;
    int zoh;
    void *du, *ddelta, *dz;          // b × D × L, I/O type (dz may be null)
    float *dB, *dC;                  // b × N × L fp32, zeroed before the launches
    float *dA;                       // D × N fp32, zeroed
    float *dDskip, *dbias;           // D fp32 or null, zeroed
    float *dh0;                      // b × D × N fp32 or null
    int *status;                     // device status word
    int *tickets;                    // two work counters (checkpoint pass, reverse pass)
    int *flags_fwd, *flags_rev;      // chunks finished per channel group, per pass
    float *carry_fwd, *carry_rev;    // b × D × N hand-offs: the state forward, the adjoint backward
    float *ckpt;                     // [group][tile][2][32 lanes] float4: the state at every tile start
    int chunk_len, nchunks, groups, ntiles;
    int ckpt_ready;                  // 1: the forward scan already wrote ckpt (no checkpoint pass)
};

// Mamba-2 (SSD) layer: heads of P channels with a scalar A each.
struct SsdArgs {
    int batch, seqlen, nheads;
    const void *x, *dt, *B, *C;      // x: b × L × H × P; dt: b × L × H; B, C: b × L × N (bf16)
    const float *A, *Dskip, *dt_bias;
    int dt_softplus;
    const float *h0;                 // b × H × P × N fp32 or null
    void *y;                         // b × L × H × P
    float *hL;                       // b × H × P × N fp32 or null
    int *status;                     // device status word or null
    int seg_chunks;                  // chunks per segment of a chain (all of them: one segment)
    int *ticket;                     // work counter, zero at launch (null: item = block index)
    int *flags;                      // b × H: segments of the chain finished, zero at launch
    float *carry;                    // b × H × P × N fp32: the state a segment hands on
};
// Segments per (sequence, head) chain of the SSD kernel, and the launch's
// work items: every chain's first segment, then every chain's second, ...
struct SsdPlan {
    int seg_chunks, nseg;
};
SsdPlan ssd_plan(int64_t batch, int64_t seqlen, int64_t nheads, bool split);

// Causal depthwise convolution + bias + optional SiLU over whole sequences.
struct ConvArgs {
    int64_t batch, dim, seqlen;
    int width;               // W in [1, 4]
    const void *x;           // b × D × L
    const float *w;          // D × W, taps oldest first
    const float *bias;       // D or nullptr
    const void *state_in;    // b × D × (W-1) or nullptr
    void *u;                 // b × D × L
    void *state_out;         // b × D × (W-1) or nullptr
    int silu;
};

// One decode token of the convolution; the state shifts in place.
struct ConvStepArgs {
    int64_t batch, dim;
    int width;
    void *state;             // b × D × (W-1)
    const void *x;           // b × D
    const float *w, *bias;
    void *u;                 // b × D
    int silu;
};

int scan_groups(int64_t dstate);
ScanPlan scan_plan(int64_t batch, int64_t dim, int64_t dstate, int64_t seqlen, int64_t requested);
cudaError_t scan_launch(const ScanArgs &a, bool bf16, cudaStream_t stream);
// The backward's checkpoint pass on the forward's warp-specialised kernel: no y,
// the state at every 16-token tile start into a.ckpt.  Supported for bf16 I/O,
// first order, 9 <= N <= 16, a row pitch TMA can describe and a chained plan.
bool scan_ckpt_supported(const ScanPlan &plan, int64_t dstate, int64_t seqlen, bool bf16, int zoh);
cudaError_t scan_ckpt_launch(const ScanArgs &a, cudaStream_t stream);
cudaError_t step_launch(const StepArgs &a, bool bf16, cudaStream_t stream);
cudaError_t conv_launch(const ConvArgs &a, bool bf16, cudaStream_t stream);
bool ssd_supported(int64_t headdim, int64_t dstate);
cudaError_t ssd_launch(const SsdArgs &a, int nseg, cudaStream_t stream);
cudaError_t bwd_launch(const BwdArgs &a, bool bf16, cudaStream_t stream);
int bwd_cpw(int64_t dstate);             // channels per warp of the backward kernels
constexpr int kBwdTile = 16;             // tokens per checkpoint / recompute tile
constexpr int kBwdChunk = 128;           // tokens per work item of the backward passes
cudaError_t conv_step_launch(const ConvStepArgs &a, bool bf16, cudaStream_t stream);
// Each kernel source's debug word (see in_range): the first index check that
// failed there, 0 if none or in a release build; `reset` clears it.
int debug_word_conv(bool reset);
int debug_word_step(bool reset);
int debug_word_bwd(bool reset);
int debug_word_fwd(bool reset);
int debug_word_ssd(bool reset);
cudaError_t mufu_ex2_launch(float *sink, int blocks, int iters, cudaStream_t stream);
cudaError_t flag_wait_selftest_launch(int *status, const int *flag, int polls, cudaStream_t stream);

}  // namespace ssm
