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

template <typename T, int NG, bool VEC, bool HAS_Z, bool ZOH>
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
            const float an = a.A[(size_t)d * N + n];
            const float abar = ex2(dv * (an * kLog2e));
            const float bbar = ZOH ? zoh_phi(dv * an, abar) : 1.f;  // exact ZOH: B̄ = Δ·φ(ΔA)·B
            hv[j] = fmaf(abar, hv[j], IO<T>::to_f(B[bb * N + n]) * du * bbar);
            part = fmaf(IO<T>::to_f(C[bb * N + n]), hv[j], part);
        }
    }
#pragma unroll
    for (int m = 1; m < NG; m <<= 1) part += __shfl_xor_sync(0xffffffffu, part, m);
    if (!own || !in_range((int64_t)(ch * N + 4 * g), N - 4 * g < 4 ? N - 4 * g : 4, (int64_t)a.batch * a.dim * N))
        return;
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
        if (in_range((int64_t)ch, 1, (int64_t)a.batch * a.dim)) static_cast<T *>(a.y)[ch] = IO<T>::from_f(out);
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

template <typename T, bool HAS_Z, bool ZOH>
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
            const float bbar = ZOH ? zoh_phi(delta * avv[j], abar) : 1.f;
            h4[j] = fmaf(abar, h4[j], bv[i][j] * du * bbar);
            part = fmaf(cv[i][j], h4[j], part);
        }
        part += __shfl_xor_sync(0xffffffffu, part, 1);
        part += __shfl_xor_sync(0xffffffffu, part, 2);
        if (w >= words || !in_range((int64_t)w * 4, 4, (int64_t)a.batch * a.dim * 16)) continue;
        __stcs(reinterpret_cast<float4 *>(a.state) + w, make_float4(h4[0], h4[1], h4[2], h4[3]));
        if (g == 0 && in_range((int64_t)w / 4, 1, (int64_t)a.batch * a.dim)) {
            float out = part + skip[i] * u;
            if (HAS_Z) out *= gate_of<T>(IO<T>::to_f(zv[i]));
            static_cast<T *>(a.y)[w / 4] = IO<T>::from_f(out);
        }
    }
}

// Decode as a TMA-fed stream (N = 16, D a multiple of 128, 16-byte aligned
// pointers).  A persistent CTA walks tiles of 128 consecutive channels; per
// tile one thread moves the 8 KB state tile, the channels' u, Δraw and z, and
// the sequence's B and C rows into shared memory with cp.async.bulk on an
// mbarrier, kStreamAhead tiles ahead; a stage is refilled only once the bulk
// store issued from it two tiles earlier has read it.  The A rows, bias and D,
// the same for every sequence and resident in L2, are read by the threads
// themselves one tile ahead.  The 128 threads
// update the state in place in shared memory (four lanes per channel, one
// 16-byte word each, conflict-free), and the tile leaves with bulk stores.
constexpr int kStreamCh = 128;     // channels per tile
#ifndef SSM_STREAM_STAGES
#define SSM_STREAM_STAGES 3   // 3: 32.7 µs per token; 4: 33.6; 6: 38.1; 8: 44.3 (fewer CTAs fit)
#endif
constexpr int kStreamStages = SSM_STREAM_STAGES;  // stages in shared memory
constexpr int kStreamAhead = kStreamStages - 2;   // tiles loading ahead of the one being updated

template <typename T> struct StreamTile {
    static constexpr int ES = (int)sizeof(T);
    static constexpr int off_h = 0;                                  // 128 × 16 fp32
    static constexpr int off_u = off_h + kStreamCh * 64;             // 128 T
    static constexpr int off_d = off_u + kStreamCh * ES;
    static constexpr int off_z = off_d + kStreamCh * ES;
    static constexpr int off_B = off_z + kStreamCh * ES;             // 16 T
    static constexpr int off_C = off_B + 16 * ES;
    static constexpr int off_y = off_C + 16 * ES;                    // 128 T
    static constexpr int bytes = (off_y + kStreamCh * ES + 127) / 128 * 128;
};

template <typename T, bool HAS_Z, bool ZOH>
__global__ void __launch_bounds__(kStreamCh) step_stream_kernel(const StepArgs a) {
    using S = StreamTile<T>;
    extern __shared__ __align__(128) unsigned char smem[];
    uint64_t *bar = reinterpret_cast<uint64_t *>(smem + kStreamStages * S::bytes);
    const int tid = threadIdx.x;
    const int ntiles = (int)((size_t)a.batch * a.dim / kStreamCh);
    const int tiles_per_seq = a.dim / kStreamCh;
    const int nmine = ntiles > (int)blockIdx.x ? (ntiles - 1 - (int)blockIdx.x) / gridDim.x + 1 : 0;
    const T *up = static_cast<const T *>(a.u), *dp = static_cast<const T *>(a.delta);
    const T *zp = static_cast<const T *>(a.z);
    const T *Bp = static_cast<const T *>(a.B), *Cp = static_cast<const T *>(a.C);

    auto issue = [&](int j) {  // j-th tile of this CTA into stage j % kStreamStages
        const int tile = blockIdx.x + j * gridDim.x;
        const size_t ch0 = (size_t)tile * kStreamCh;
        const size_t bb = tile / tiles_per_seq;
        const int d0 = (tile % tiles_per_seq) * kStreamCh;
        unsigned char *st = smem + (j % kStreamStages) * S::bytes;
        uint64_t *b = &bar[j % kStreamStages];
        (void)d0;
        uint32_t bytes = kStreamCh * 64 + 2 * kStreamCh * S::ES + 2 * 16 * S::ES;
        if (HAS_Z) bytes += kStreamCh * S::ES;
        mbar_arrive_expect_tx(b, bytes);
        bulk_load(st + S::off_h, a.state + ch0 * 16, kStreamCh * 64, b);
        bulk_load(st + S::off_u, up + ch0, kStreamCh * S::ES, b);
        bulk_load(st + S::off_d, dp + ch0, kStreamCh * S::ES, b);
        if (HAS_Z) bulk_load(st + S::off_z, zp + ch0, kStreamCh * S::ES, b);
        bulk_load(st + S::off_B, Bp + bb * 16, 16 * S::ES, b);
        bulk_load(st + S::off_C, Cp + bb * 16, 16 * S::ES, b);
    };

    if (tid == 0) {
        for (int s = 0; s < kStreamStages; ++s) mbar_init(&bar[s], 1);
        fence_mbar_init();
        for (int j = 0; j < kStreamAhead && j < nmine; ++j) issue(j);
    }
    __syncthreads();

    // Per-thread rows that do not depend on the sequence: A words, bias, D,
    // loaded one tile ahead into registers.
    const int g = tid & 3;
    float4 an[4];
    float bn[4], kn[4];
    auto prefetch = [&](int j) {
        const int tile = blockIdx.x + j * gridDim.x;
        const int d0 = (tile % tiles_per_seq) * kStreamCh;
#pragma unroll
        for (int i = 0; i < 4; ++i) {
            const int c = (i * kStreamCh + tid) >> 2;
            an[i] = __ldg(reinterpret_cast<const float4 *>(a.A + (size_t)(d0 + c) * 16) + g);
            bn[i] = a.bias ? __ldg(a.bias + d0 + c) : 0.f;
            kn[i] = a.Dskip ? __ldg(a.Dskip + d0 + c) : 0.f;
        }
    };
    if (nmine > 0) prefetch(0);

    bool failed = false;
    for (int j = 0; j < nmine; ++j) {
        const int s = j % kStreamStages;
        unsigned char *st = smem + s * S::bytes;
        // Load tile j + ahead into the stage of tile j + ahead - stages (= j - 2),
        // whose store (the older of the two pending) must have read it first.
        if (tid == 0 && j + kStreamAhead < nmine) {
            bulk_wait_read1();
            issue(j + kStreamAhead);
        }
        float4 ac[4];
        float bc[4], kc[4];
#pragma unroll
        for (int i = 0; i < 4; ++i) {
            ac[i] = an[i];
            bc[i] = bn[i];
            kc[i] = kn[i];
        }
        if (j + 1 < nmine) prefetch(j + 1);
        const bool ok = mbar_wait_bounded(&bar[s], (j / kStreamStages) & 1, 1u << 22);
        if (__syncthreads_or(!ok)) {
            failed = true;
            break;
        }
        const int tile = blockIdx.x + j * gridDim.x;
        float4 *hs = reinterpret_cast<float4 *>(st + S::off_h);
        const T *us = reinterpret_cast<const T *>(st + S::off_u);
        const T *ds = reinterpret_cast<const T *>(st + S::off_d);
        const T *zs = reinterpret_cast<const T *>(st + S::off_z);
        const T *Bs = reinterpret_cast<const T *>(st + S::off_B);
        const T *Cs = reinterpret_cast<const T *>(st + S::off_C);
        T *ys = reinterpret_cast<T *>(st + S::off_y);
        float bv[4], cv[4];
#pragma unroll
        for (int k = 0; k < 4; ++k) {
            bv[k] = IO<T>::to_f(Bs[4 * g + k]);
            cv[k] = IO<T>::to_f(Cs[4 * g + k]);
        }
#pragma unroll
        for (int i = 0; i < 4; ++i) {
            const int w = i * kStreamCh + tid;  // state word: channel w / 4, states 4g .. 4g+3
            const int c = w >> 2;
            const float4 hv = hs[w];
            const float4 av = ac[i];
            const float u = IO<T>::to_f(us[c]);
            float dl = IO<T>::to_f(ds[c]) + bc[i];
            if (a.delta_softplus) dl = softplus(dl);
            const float du = dl * u;
            const float avv[4] = {av.x, av.y, av.z, av.w};
            float h4[4] = {hv.x, hv.y, hv.z, hv.w};
            float part = 0.f;
#pragma unroll
            for (int k = 0; k < 4; ++k) {
                const float abar = ex2(dl * (avv[k] * kLog2e));
                const float bbar = ZOH ? zoh_phi(dl * avv[k], abar) : 1.f;
                h4[k] = fmaf(abar, h4[k], bv[k] * du * bbar);
                part = fmaf(cv[k], h4[k], part);
            }
            part += __shfl_xor_sync(0xffffffffu, part, 1);
            part += __shfl_xor_sync(0xffffffffu, part, 2);
            hs[w] = make_float4(h4[0], h4[1], h4[2], h4[3]);
            if (g == 0) {
                float out = part + kc[i] * u;
                if (HAS_Z) out *= gate_of<T>(IO<T>::to_f(zs[c]));
                ys[c] = IO<T>::from_f(out);
            }
        }
        fence_proxy_async_smem();
        __syncthreads();
        if (tid == 0) {
            const size_t ch0 = (size_t)tile * kStreamCh;
            const int64_t chans = (int64_t)a.batch * a.dim;
            if (in_range((int64_t)ch0 * 16, kStreamCh * 16, chans * 16))
                bulk_store(a.state + ch0 * 16, st + S::off_h, kStreamCh * 64);
            if (in_range((int64_t)ch0, kStreamCh, chans))
                bulk_store(static_cast<T *>(a.y) + ch0, st + S::off_y, kStreamCh * S::ES);
            bulk_commit();
        }
    }
    // A wait that ran out (never expected) leaves the remaining tiles of this
    // CTA unprocessed; the copies already issued are drained first.
    if (tid == 0) {
        bulk_wait0();
        if (failed)
            for (int s = 0; s < kStreamStages; ++s) (void)mbar_wait_bounded(&bar[s], 0, 1u << 20);
    }
}

namespace {
template <typename T>
cudaError_t stream_dispatch(const StepArgs &a, cudaStream_t st) {
    using S = StreamTile<T>;
    const int smem = kStreamStages * S::bytes + 64;
    const int ntiles = (int)((size_t)a.batch * a.dim / kStreamCh);
    static PerDevice per_device;
    int grid_cap = 0;
    const cudaError_t e = per_device.get(
        [&](int *v) {
            auto k0 = step_stream_kernel<T, false, false>;
            auto k1 = step_stream_kernel<T, true, false>;
            auto k2 = step_stream_kernel<T, false, true>;
            auto k3 = step_stream_kernel<T, true, true>;
            cudaError_t r = cudaSuccess;
            for (auto k : {k0, k1, k2, k3})
                if (r == cudaSuccess) r = cudaFuncSetAttribute(k, cudaFuncAttributeMaxDynamicSharedMemorySize, smem);
            if (r != cudaSuccess) return r;
            int per_sm = 0;
            r = cudaOccupancyMaxActiveBlocksPerMultiprocessor(&per_sm, k1, kStreamCh, smem);
            *v = sm_count() * (per_sm > 0 ? per_sm : 1);
            return r;
        },
        &grid_cap);
    if (e != cudaSuccess) return e;
    const int grid = ntiles < grid_cap ? ntiles : grid_cap;
    if (a.zoh) {
        if (a.z) step_stream_kernel<T, true, true><<<grid, kStreamCh, smem, st>>>(a);
        else step_stream_kernel<T, false, true><<<grid, kStreamCh, smem, st>>>(a);
    } else {
        if (a.z) step_stream_kernel<T, true, false><<<grid, kStreamCh, smem, st>>>(a);
        else step_stream_kernel<T, false, false><<<grid, kStreamCh, smem, st>>>(a);
    }
    return cudaGetLastError();
}

template <typename T>
cudaError_t wide_dispatch(const StepArgs &a, cudaStream_t st) {
    const size_t words = (size_t)a.batch * a.dim * 4;
    const unsigned blocks = (unsigned)((words + kStepThreads * kStepIPT - 1) / (kStepThreads * kStepIPT));
    if (a.zoh) {
        if (a.z) step_wide_kernel<T, true, true><<<blocks, kStepThreads, 0, st>>>(a);
        else step_wide_kernel<T, false, true><<<blocks, kStepThreads, 0, st>>>(a);
    } else {
        if (a.z) step_wide_kernel<T, true, false><<<blocks, kStepThreads, 0, st>>>(a);
        else step_wide_kernel<T, false, false><<<blocks, kStepThreads, 0, st>>>(a);
    }
    return cudaGetLastError();
}

template <typename T, int NG, bool ZOH>
cudaError_t step_dispatch_z(const StepArgs &a, cudaStream_t st) {
    const size_t items = (size_t)a.batch * a.dim * NG;
    const unsigned blocks = (unsigned)((items + 255) / 256);
    const bool vec = a.dstate % 4 == 0 && (reinterpret_cast<uintptr_t>(a.state) & 15) == 0;
    const bool z = a.z != nullptr;
    if (vec && z) step_kernel<T, NG, true, true, ZOH><<<blocks, 256, 0, st>>>(a);
    else if (vec) step_kernel<T, NG, true, false, ZOH><<<blocks, 256, 0, st>>>(a);
    else if (z) step_kernel<T, NG, false, true, ZOH><<<blocks, 256, 0, st>>>(a);
    else step_kernel<T, NG, false, false, ZOH><<<blocks, 256, 0, st>>>(a);
    return cudaGetLastError();
}
template <typename T, int NG>
cudaError_t step_dispatch(const StepArgs &a, cudaStream_t st) {
    return a.zoh ? step_dispatch_z<T, NG, true>(a, st) : step_dispatch_z<T, NG, false>(a, st);
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
    // The bulk-copy stream also needs whole 128-channel tiles within one
    // sequence and 16-byte aligned per-channel arrays.
#ifndef SSM_STEP_STREAM
#define SSM_STEP_STREAM 1
#endif
    const bool stream = SSM_STEP_STREAM && wide && a.dim % kStreamCh == 0 && aligned16(a.u) && aligned16(a.delta) &&
                        (!a.z || aligned16(a.z)) && (!a.bias || aligned16(a.bias)) && (!a.Dskip || aligned16(a.Dskip)) &&
                        aligned16(a.y);
    if (stream) return bf16 ? stream_dispatch<__nv_bfloat16>(a, st) : stream_dispatch<float>(a, st);
    if (wide) return bf16 ? wide_dispatch<__nv_bfloat16>(a, st) : wide_dispatch<float>(a, st);
    return bf16 ? step_ng<__nv_bfloat16>(a, st) : step_ng<float>(a, st);
}

SSM_DEBUG_WORD_READER(debug_word_step)

}  // namespace ssm
