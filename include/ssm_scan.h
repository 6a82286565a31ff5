/*
 * ssm_scan.h — C ABI of libssmscan, the B300 (sm_103a) Mamba selective scan.
 *
 * Operation (forward scan), per batch b, channel d, state n and token t:
 *
 *   Δ_t     = softplus(Δraw[b,d,t] + bias[d])   (or Δraw + bias, see delta_softplus)
 *   Ā_t,n   = exp(Δ_t · A[d,n])
 *   B̄_t,n   = Δ_t · B[b,n,t]                    (first order; zoh = 1 selects the
 *                                                 exact zero-order hold (Ā−1)/A · B)
 *   h_t,n   = Ā_t,n · h_{t−1},n + B̄_t,n · u[b,d,t],   h_{−1} = h0 (zeros if NULL)
 *   y[b,d,t]= (Σ_n C[b,n,t] · h_t,n + Dskip[d] · u[b,d,t]) · silu(z[b,d,t])
 *   hL[b,d,n] = h_{L−1},n
 *
 * Sources: the SSM, its zero-order-hold discretisation and the first-order
 * B̄ = ΔB — "Mamba and selective state spaces, from first principles",
 * sections "A state space model", "Discretisation: zero-order hold"; the
 * input-dependent Δ = softplus(bias + ·), B_t, C_t — same page, "Selection:
 * B, C and Δ from the token"; the D·u skip — "State space models and Mamba",
 * "One system, two views"; the silu gate branch — first-principles page,
 * "The Mamba block"; the fused scan that writes only y — first-principles page,
 * "The hardware-aware scan".
 *
 * The decode step (ssm_state_update) is the same recurrence with L = 1 on a
 * carried state ("A fixed state against a growing cache", first-principles
 * page; streaming inference in "One system, two views").
 *
 * Conventions for every entry point:
 *   - All tensor pointers are DEVICE pointers, row-major and contiguous, with
 *     the shapes given below.  The caller owns all memory; the library
 *     allocates nothing (no cudaMalloc, no host allocation per call).
 *   - Work is enqueued asynchronously on `stream` (0 = legacy default stream).
 *   - Invalid arguments return SSM_ERR_INVALID_ARG / SSM_ERR_UNSUPPORTED and
 *     launch nothing.  A failed launch returns SSM_ERR_CUDA.  Errors detected
 *     on the device (a bounded wait that ran out) are recorded in the
 *     workspace and read back by ssm_workspace_status.
 *   - ssm_scan_fwd: u, delta, z, B, C, y, h0, hL and workspace must be
 *     16-byte aligned; A, Dskip and delta_bias 4-byte aligned.
 *     ssm_state_update: every pointer aligned to its element size.
 *     y must not overlap any input.  hL may be the same buffer as h0.
 */
#ifndef SSM_SCAN_H
#define SSM_SCAN_H

#include <stddef.h>
#include <stdint.h>

#ifdef __cplusplus
extern "C" {
#endif

typedef struct CUstream_st *ssm_stream_t; /* the same type as cudaStream_t */

typedef enum {
    SSM_OK = 0,
    SSM_ERR_INVALID_ARG = 1, /* null pointer, bad size, misaligned pointer, small workspace */
    SSM_ERR_UNSUPPORTED = 2, /* a valid request this build does not implement (e.g. dstate > 16) */
    SSM_ERR_CUDA = 3,        /* a CUDA runtime call or launch failed */
    SSM_ERR_TIMEOUT = 4,     /* a device-side bounded wait ran out (reported via the workspace) */
    SSM_ERR_BOUNDS = 5       /* debug build only: an index check found a store outside its buffer */
} ssm_status;

typedef enum { SSM_F32 = 0, SSM_BF16 = 1 } ssm_dtype;

/* Largest state size N the kernels are built for. */
#define SSM_MAX_DSTATE 16

typedef struct {
    int64_t batch;          /* b  >= 1 */
    int64_t dim;            /* D  >= 1 (channels) */
    int64_t dstate;         /* N  in [1, SSM_MAX_DSTATE] */
    int64_t seqlen;         /* L  >= 1 */
    ssm_dtype io_dtype;     /* dtype of u, delta, z, B, C and y */
    const void *u;          /* b × D × L, io_dtype */
    const void *delta;      /* b × D × L, io_dtype: Δraw before bias / softplus */
    const void *z;          /* b × D × L, io_dtype; NULL = no gate (factor 1) */
    const void *B;          /* b × N × L, io_dtype */
    const void *C;          /* b × N × L, io_dtype */
    const float *A;         /* D × N fp32, any values (S4D-Real init is −(n+1)) */
    const float *Dskip;     /* D fp32; NULL = 0 */
    const float *delta_bias;/* D fp32; NULL = 0 */
    int delta_softplus;     /* 1: Δ = softplus(Δraw + bias); 0: Δ = Δraw + bias */
    int zoh;                /* 0: B̄ = Δ·B (first order); 1: exact ZOH (Ā − 1)/A · B */
    const float *h0;        /* b × D × N fp32 initial state; NULL = zeros */
    void *y;                /* out: b × D × L, io_dtype */
    float *hL;              /* out: b × D × N fp32 final state; NULL = not written */
    void *workspace;        /* device scratch of >= ssm_scan_workspace_size(...) bytes */
    size_t workspace_bytes;
    int64_t chunk_len;      /* 0 = automatic.  Otherwise the sequence is cut into
                               chunks of this many tokens (a multiple of 64),
                               joined by carried states (see ssm_scan_plan). */
} ssm_scan_params;

/* Bytes of workspace ssm_scan_fwd needs for these sizes and chunk_len (never 0:
 * the workspace always holds the device status word).  Returns 0 only when the
 * sizes are invalid. */
size_t ssm_scan_workspace_size(const ssm_scan_params *p);

/* How ssm_scan_fwd will cut this scan into work items (host-side, no GPU
 * needed).  On SSM_OK fills out[0] = tokens per chunk, out[1] = number of
 * chunks K, out[2] = 1 if chunk k starts from the state chunk k-1 hands over
 * (chained) or 0 if, when K > 1, the chunks run at once and carry their
 * starting states by decoupled look-back: aggregate work items scan each
 * chunk but the last from a zero state for its pair (Π Ā, h_end) and publish
 * it; each chunk's main item composes its predecessors' pairs from h0 in chunk
 * order (bit for bit the same whichever predecessor the walk stops at),
 * publishes the state it leaves and scans, out[3] = number of channel
 * groups (one scanning warp each).  Either way the scan is one launch,
 * preceded by one small launch that widens B and C to fp32 token-major rows
 * in the workspace.  Returns SSM_ERR_INVALID_ARG for invalid sizes or a NULL
 * out. */
ssm_status ssm_scan_plan(const ssm_scan_params *p, int64_t out[4]);

/* Forward selective scan: writes y and (if non-NULL) hL.  Also clears the
 * workspace status word before launching.  With K > 1 the launch's warps
 * wait on one another (bounded spins on flags in the workspace); its grid is
 * sized to the CTAs the device holds at once, so work that occupies SMs for
 * long on another stream can delay it, and a wait that reaches its bound is
 * reported as SSM_ERR_TIMEOUT through ssm_workspace_status. */
ssm_status ssm_scan_fwd(const ssm_scan_params *p, ssm_stream_t stream);

typedef struct {
    int64_t batch;          /* b >= 1 (independent sequences) */
    int64_t dim;            /* D >= 1 */
    int64_t dstate;         /* N in [1, SSM_MAX_DSTATE] */
    ssm_dtype io_dtype;     /* dtype of u, delta, z, B, C and y */
    float *state;           /* b × D × N fp32 carried state, read and updated in place */
    const void *u;          /* b × D, io_dtype: this token's input */
    const void *delta;      /* b × D, io_dtype */
    const void *z;          /* b × D, io_dtype; NULL = no gate */
    const void *B;          /* b × N, io_dtype */
    const void *C;          /* b × N, io_dtype */
    const float *A;         /* D × N fp32 */
    const float *Dskip;     /* D fp32; NULL = 0 */
    const float *delta_bias;/* D fp32; NULL = 0 */
    int delta_softplus;
    int zoh;
    void *y;                /* out: b × D, io_dtype */
} ssm_step_params;

/* One decode token for every (b, d): the recurrence with L = 1 on `state`. */
ssm_status ssm_state_update(const ssm_step_params *p, ssm_stream_t stream);

/* ------------------------------------------------------------------------
 * Backward scan: the gradient of ssm_scan_fwd.
 *
 * For upstream gradients dy = ∂loss/∂y and dhL = ∂loss/∂hL it returns
 * ∂loss/∂ of u, Δraw, z, B, C, A, Dskip, delta_bias and h0.  The adjoint state
 * runs backwards in time,
 *
 *   λ_t = C_t · ŷ_t + Ā_{t+1} ⊙ λ_{t+1},   λ_{L−1} starts from dhL,
 *   ŷ_t = dy_t · silu(z_t)                  (dy_t without a gate),
 *
 * and the gradients are read off it by the chain rule: du_t = ŷ_t·D +
 * Σ_n λ_t,n B̄_t,n; dC_t,n = Σ_d ŷ_t h_t,n; dB, dΔ, dA from ∂Ā/∂Δ = A·Ā,
 * ∂Ā/∂A = Δ·Ā and the B̄ of the chosen discretisation; dΔraw = dΔ·σ(Δraw +
 * bias) with softplus; dz_t = dy_t·(C·h + D·u)_t·silu'(z_t); dh0 = Ā_0 ⊙ λ_0.
 * Source: the backward pass recomputes the intermediate states rather than
 * storing them ("Mamba and selective state spaces, from first principles",
 * "The hardware-aware scan"; erikxu.me notes, "GPU Memory Hierarchy").  The
 * pages give no formulas: these are the derivatives of the forward operation
 * above.
 *
 * The forward inputs are those of ssm_scan_fwd (same meaning and layout); y
 * itself is not needed.  All pointers are device pointers aligned to their
 * element size (4 bytes for fp32); workspace 16-byte aligned.  The library
 * zeroes dB, dC, dA, dDskip and ddelta_bias and accumulates into them on the
 * device, so their values are sums in an unspecified order.
 * ------------------------------------------------------------------------ */
typedef struct {
    int64_t batch, dim, dstate, seqlen;   /* as in ssm_scan_params; dstate <= 16 */
    ssm_dtype io_dtype;                   /* dtype of u, delta, z, B, C, dy, du, ddelta, dz */
    const void *u, *delta, *z, *B, *C;    /* the forward inputs; z may be NULL */
    const float *A, *Dskip, *delta_bias;  /* as in ssm_scan_params (NULL = 0 for the last two) */
    int delta_softplus, zoh;              /* as in ssm_scan_params */
    const float *h0;                      /* b × D × N fp32 initial state; NULL = zeros */
    const void *dy;                       /* b × D × L, io_dtype: ∂loss/∂y */
    const float *dhL;                     /* b × D × N fp32: ∂loss/∂hL; NULL = 0 */
    void *du, *ddelta;                    /* out: b × D × L, io_dtype */
    void *dz;                             /* out: b × D × L, io_dtype; NULL = not written */
    float *dB, *dC;                       /* out: b × N × L fp32 */
    float *dA;                            /* out: D × N fp32 */
    float *dDskip, *ddelta_bias;          /* out: D fp32; NULL = not computed */
    float *dh0;                           /* out: b × D × N fp32; NULL = not written */
    void *workspace;                      /* >= ssm_scan_bwd_workspace_size(...) bytes */
    size_t workspace_bytes;
    int64_t chunk_len;                    /* 0 = automatic (128); else a multiple of 16 */
} ssm_scan_bwd_params;

/* Bytes of workspace ssm_scan_bwd needs for the sizes, io_dtype, zoh and
 * chunk_len in *p (the pointers are not read): the status word and work
 * counters, two chained hand-off states of b × D × N fp32, and the recurrence
 * state at every 16th token (4 bytes per (b, d, t) element for N = 16).  With
 * bf16 I/O, first order, 9 <= N <= 16 and enough channel groups for a chained
 * forward plan, the checkpoints come from the forward scan kernel, which adds
 * its flags, one more b × D × N hand-off state and B, C as fp32 rows
 * (2 × b × L × 16 × 4 bytes); a workspace without that room still works,
 * with the backward's own checkpoint pass.  0 for invalid sizes. */
size_t ssm_scan_bwd_workspace_size(const ssm_scan_bwd_params *p);

/* The backward scan on `stream`, after clearing the accumulated outputs: a
 * checkpoint pass (the forward recurrence, writing the state at every 16th
 * token — on the forward scan's warp-specialised kernel where the workspace
 * size above includes its room, else on a kernel of its own) and the reverse
 * pass.  Device-side wait failures are reported through ssm_workspace_status
 * on this workspace. */
ssm_status ssm_scan_bwd(const ssm_scan_bwd_params *p, ssm_stream_t stream);

/* ------------------------------------------------------------------------
 * Mamba-2 layer scan (state space duality, SSD).
 *
 * Per batch b, head h (P channels, scalar A_h) and token t:
 *   Δ_t   = softplus(dt[b,t,h] + dt_bias[h])   (or without softplus)
 *   a_t   = exp(Δ_t · A[h])
 *   S_t   = a_t · S_{t−1} + Δ_t · x_t ⊗ B_t     (S: P × N per head, S_{−1} = h0)
 *   y_t   = S_t · C_t + Dskip[h] · x_t
 * Source: "Mamba and selective state spaces, from first principles", section
 * "Mamba-2: state space duality" (A a scalar times the identity per head,
 * heads of P channels sharing a_t, B_t, C_t; the chunked algorithm that turns
 * the layer into tensor-core products).  One group of B, C for all heads, as
 * in the Mamba-2 2.7B projection the section describes.
 *
 * This build supports headdim P = 64, dstate N = 128 and bf16 I/O
 * (SSM_ERR_UNSUPPORTED otherwise); the products take bf16 operands with fp32
 * accumulation, the carried state is fp32.  Pointers are device pointers;
 * x, B, C and y 16-byte aligned, the rest aligned to their element size.
 * ------------------------------------------------------------------------ */
typedef struct {
    int64_t batch, seqlen, nheads;   /* b, L, H */
    int64_t headdim, dstate;         /* P (64), N (128) */
    ssm_dtype io_dtype;              /* SSM_BF16 */
    const void *x;                   /* b × L × H × P */
    const void *dt;                  /* b × L × H: Δraw per head */
    const float *A;                  /* H: the head's scalar A (negative for a decay) */
    const void *B, *C;               /* b × L × N */
    const float *Dskip, *dt_bias;    /* H fp32; NULL = 0 */
    int dt_softplus;                 /* 1: Δ = softplus(dt + dt_bias); 0: Δ = dt + dt_bias */
    const float *h0;                 /* b × H × P × N fp32; NULL = zeros */
    void *y;                         /* out: b × L × H × P */
    float *hL;                       /* out: b × H × P × N fp32; NULL = not written */
    int32_t *status;                 /* device int or NULL: a bounded wait inside the kernel
                                        that ran out stores SSM_ERR_TIMEOUT here if it still
                                        holds 0 (the caller zeroes it and reads it back) */
    void *workspace;                 /* device, 256-byte aligned, ssm_ssd_workspace_size bytes;
                                        or NULL */
    size_t workspace_bytes;
} ssm_ssd_params;

/* Workspace bytes ssm_ssd_fwd uses to split each (sequence, head) chain into
 * segments (0 for invalid sizes): a 256-byte header (a work counter), a flag
 * per chain and one fp32 P × N state per chain, which a segment hands to the
 * next.  With the workspace the launch takes every chain's first segment,
 * then every chain's second, and so on, from the counter, so that the SMs
 * stay busy to the end; without it (NULL) one CTA walks a whole chain.  Both
 * give bit-identical results.  The call clears the counter and the flags
 * (an asynchronous memset on the stream) before the launch. */
size_t ssm_ssd_workspace_size(const ssm_ssd_params *p);

/* The Mamba-2 layer scan: a memset of the workspace header (when a workspace
 * is given) and one launch.  The kernel's waits on its own copies and
 * products, and a segment's wait for the previous segment's state, are
 * bounded; when one runs out, y and hL are incomplete and the status word (if
 * given) says SSM_ERR_TIMEOUT.  A workspace smaller than
 * ssm_ssd_workspace_size, or not 256-byte aligned, is SSM_ERR_INVALID_ARG. */
ssm_status ssm_ssd_fwd(const ssm_ssd_params *p, ssm_stream_t stream);

/* ------------------------------------------------------------------------
 * The short convolution in front of the SSM.
 *
 * Operation, per batch b, channel d and token t (W = width):
 *
 *   u[b,d,t] = silu(bias[d] + Σ_{k=0}^{W−1} weight[d,k] · x[b,d,t−(W−1)+k])
 *              (or without the silu when silu = 0)
 *
 * where x at a time before the sequence is read from state_in (the W−1 inputs
 * just before x[b,d,0], oldest first; zeros if NULL).  The taps are in time
 * order: weight[d,W−1] multiplies the current input.  state_out receives the
 * last W−1 inputs of the sequence, oldest first, reaching into state_in when
 * L < W−1, so that a later call on the continuation carries on exactly.
 *
 * Source: a causal depthwise convolution of width 4 followed by SiLU feeds the
 * SSM branch of the block ("Mamba and selective state spaces, from first
 * principles", "The Mamba block"; the erikxu.me notes, "Mamba Architecture");
 * its three carried inputs per channel are part of the decode state (same
 * first-principles page, "A fixed state against a growing cache").  Its output
 * u is the scan's input u and the input of the projections that form Δ, B and
 * C, so it is written to memory rather than fused into the scan.
 *
 * Pointers are device pointers, aligned to their element size (4 bytes for the
 * fp32 weight and bias); 16-byte aligned x and u with L a multiple of 8 take
 * the vectorised path, anything else a slower scalar one.  u must not overlap
 * x; state_out must not overlap x, u or state_in.
 * ------------------------------------------------------------------------ */

/* Largest convolution width the kernels are built for. */
#define SSM_MAX_CONV_WIDTH 4

typedef struct {
    int64_t batch;          /* b >= 1 */
    int64_t dim;            /* D >= 1 (channels) */
    int64_t seqlen;         /* L >= 1 */
    int64_t width;          /* W in [1, SSM_MAX_CONV_WIDTH] (the block uses 4) */
    ssm_dtype io_dtype;     /* dtype of x, u, state_in and state_out */
    const void *x;          /* b × D × L: the convolution's input */
    const float *weight;    /* D × W fp32, taps oldest first */
    const float *bias;      /* D fp32; NULL = 0 */
    int silu;               /* 1: apply SiLU; 0: plain convolution + bias */
    const void *state_in;   /* b × D × (W−1); NULL = zeros (ignored when W = 1) */
    void *u;                /* out: b × D × L */
    void *state_out;        /* out: b × D × (W−1); NULL = not written */
} ssm_conv_params;

/* Causal depthwise convolution (+ bias, + SiLU) over whole sequences. */
ssm_status ssm_conv1d_fwd(const ssm_conv_params *p, ssm_stream_t stream);

typedef struct {
    int64_t batch;          /* b >= 1 */
    int64_t dim;            /* D >= 1 */
    int64_t width;          /* W in [1, SSM_MAX_CONV_WIDTH] */
    ssm_dtype io_dtype;     /* dtype of state, x and u */
    void *state;            /* b × D × (W−1): the last W−1 inputs, oldest first; read,
                               then shifted by one input in place (may be NULL when W = 1) */
    const void *x;          /* b × D: this token's input */
    const float *weight;    /* D × W fp32 */
    const float *bias;      /* D fp32; NULL = 0 */
    int silu;
    void *u;                /* out: b × D */
} ssm_conv_step_params;

/* One decode token of the convolution: u from the carried inputs and x, then
 * the state drops its oldest input and appends x.  u must not overlap x or
 * the state. */
ssm_status ssm_conv1d_step(const ssm_conv_step_params *p, ssm_stream_t stream);

/* Size of the scratch array that ssm_scan_fwd_noalloc keeps inside the
 * library (16 MiB, held on every GPU that loads the library until exit). */
#define SSM_NOALLOC_SCRATCH_BYTES (16u << 20)

/* ssm_scan_fwd for callers that cannot allocate device memory at all (a
 * plugin whose host framework owns every allocation and offers it no
 * allocator, or a loop that must not call cudaMalloc because it can
 * synchronise the device).  The pages have no counterpart; it is a service of
 * this library.
 *
 * It computes exactly what ssm_scan_fwd computes, but the chunk scratch lives
 * in a fixed device array of SSM_NOALLOC_SCRATCH_BYTES inside the library, so
 * p->workspace and p->workspace_bytes are ignored.  It allocates nothing and
 * frees nothing.
 *   - The first call on a device looks up the array's device address with
 *     cudaGetSymbolAddress (with that device current) and caches it; make that
 *     first call before any stream capture.  cudaDeviceReset destroys the
 *     array with the context and the cached address then points at freed
 *     memory: a process that resets a device must not call this entry point
 *     on that device again.
 *   - The library's kernels and this array are set up per device, so a
 *     process may call it on several devices, each with its own array.
 *   - Sizes whose scratch need (ssm_scan_workspace_size) exceeds
 *     SSM_NOALLOC_SCRATCH_BYTES are rejected with SSM_ERR_UNSUPPORTED before
 *     anything is launched; other argument errors are those of ssm_scan_fwd.
 *   - Every call on a device shares the one array, which keeps the last
 *     call's contents.  Calls whose work overlaps on the GPU (different
 *     streams, not ordered by events) race on it: serialise them.
 *   - A device-side timeout is recorded in the shared array, where
 *     ssm_workspace_status cannot reach it; callers that need that report use
 *     ssm_scan_fwd with their own workspace. */
ssm_status ssm_scan_fwd_noalloc(const ssm_scan_params *p, ssm_stream_t stream);

/* Synchronises `stream`, then returns SSM_OK or the error a kernel recorded in
 * this workspace (SSM_ERR_TIMEOUT), or SSM_ERR_CUDA if the copy fails. */
ssm_status ssm_workspace_status(const void *workspace, ssm_stream_t stream);

/* Static description of a status code. */
const char *ssm_status_string(ssm_status s);

/* Debug build (compiled with -DSSM_DEBUG, libssmscan_debug.so): every kernel
 * checks the element range of each global store against the buffer it writes,
 * skips a store that falls outside and records SSM_ERR_BOUNDS in a device word
 * of its source file; no check traps.  Synchronises the device, then returns
 * SSM_OK or SSM_ERR_BOUNDS (SSM_ERR_CUDA if a word cannot be read); `reset`
 * non-zero clears the words.  The release build returns SSM_ERR_UNSUPPORTED. */
ssm_status ssm_debug_status(int reset);

/* Measurement helper (not part of the method): launches `blocks` × 256 threads
 * that each evaluate 16 × iters dependent-free ex2.approx.ftz.f32 chains and
 * write one float per thread to `sink` (blocks × 256 floats).  Timing it gives
 * the MUFU ex2 throughput the scan's roofline is taken against. */
ssm_status ssm_bench_mufu_ex2(float *sink, int blocks, int iters, ssm_stream_t stream);

/* Self-test of the device-side failure path (not part of the method).
 * Clears the status word and a flag in the workspace's 256-byte header, then
 * launches one thread that waits for that flag — which nothing sets — with the
 * bounded wait the chained scans use for a predecessor's hand-off.  After
 * `polls` polls (1 .. 2^24; about a microsecond each) it records
 * SSM_ERR_TIMEOUT in the status word, exactly as a scan whose hand-off never
 * came would.  ssm_workspace_status then returns SSM_ERR_TIMEOUT and the
 * context stays usable.  workspace: a device buffer of at least 256 bytes,
 * 16-byte aligned.  Returns SSM_ERR_INVALID_ARG for bad arguments (nothing
 * launched) or SSM_ERR_CUDA if the launch fails. */
ssm_status ssm_selftest_flag_wait(void *workspace, size_t workspace_bytes, int polls, ssm_stream_t stream);

/* Library build identification, e.g. "libssmscan sm_103a". */
const char *ssm_version(void);

#ifdef __cplusplus
}
#endif

#endif /* SSM_SCAN_H */
