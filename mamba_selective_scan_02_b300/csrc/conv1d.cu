// conv1d.cu — the short causal depthwise convolution in front of the SSM, with
// its bias and SiLU: u_t = silu(bias + Σ_k w_k · x_{t−(W−1)+k}) for every
// channel, the inputs before the sequence taken from a carried state of the
// last W−1 inputs ("Mamba and selective state spaces, from first principles" —
// "The Mamba block": a causal depthwise convolution of width 4 and a SiLU feed
// the SSM branch; "A fixed state against a growing cache": three inputs per
// channel are part of the decode state).
//
// The output u is what the selection projections read to form Δ, B and C
// (same page, "Selection: B, C and Δ from the token"), so it has to reach HBM
// before the scan runs; the convolution is a kernel of its own, bound by HBM:
// one read of x and one write of u per element.
//
// Sequence kernel: a warp walks row segments of 256 × kGran tokens; each
// lane holds 8 consecutive tokens of a granule (one 16-byte load for bf16, two
// for fp32), so a warp instruction moves 512 or 1,024 contiguous bytes.  The
// W−1 inputs before a lane's first token are the last ones of the lane to its
// left (a shuffle); lane 0 takes them from the previous granule's lane 31, or
// at a segment start from global memory or the carried state.  Rows whose
// pitch is not a multiple of 16 bytes, or ragged tails, take bounded scalar
// loads instead.
//
// Decode kernel: one thread per channel reads the carried inputs and this
// token's input, writes u and shifts the state by one in place.
#include <algorithm>

#include "ssm_device.cuh"
#include "ssm_internal.h"

namespace ssm {
namespace {

constexpr int kConvThreads = 256;   // 8 warps, one segment each
constexpr int kGran = 4;            // 256-token granules per warp segment
constexpr int kSegTokens = 256 * kGran;

template <typename T> struct Vec8;
template <> struct Vec8<float> {
    __device__ __forceinline__ static void load(const float *p, float *o) {
        const float4 a = __ldg(reinterpret_cast<const float4 *>(p));
        const float4 b = __ldg(reinterpret_cast<const float4 *>(p) + 1);
        o[0] = a.x; o[1] = a.y; o[2] = a.z; o[3] = a.w; o[4] = b.x; o[5] = b.y; o[6] = b.z; o[7] = b.w;
    }
    __device__ __forceinline__ static void store(float *p, const float *v) {
        reinterpret_cast<float4 *>(p)[0] = make_float4(v[0], v[1], v[2], v[3]);
        reinterpret_cast<float4 *>(p)[1] = make_float4(v[4], v[5], v[6], v[7]);
    }
};
template <> struct Vec8<__nv_bfloat16> {
    __device__ __forceinline__ static void load(const __nv_bfloat16 *p, float *o) {
        const uint4 v = __ldg(reinterpret_cast<const uint4 *>(p));
        using B = IO<__nv_bfloat16>;
        o[0] = B::lo(v.x); o[1] = B::hi(v.x); o[2] = B::lo(v.y); o[3] = B::hi(v.y);
        o[4] = B::lo(v.z); o[5] = B::hi(v.z); o[6] = B::lo(v.w); o[7] = B::hi(v.w);
    }
    __device__ __forceinline__ static uint32_t pk(float a, float b) {
        const __nv_bfloat162 v = __floats2bfloat162_rn(a, b);
        return *reinterpret_cast<const uint32_t *>(&v);
    }
    __device__ __forceinline__ static void store(__nv_bfloat16 *p, const float *v) {
        *reinterpret_cast<uint4 *>(p) = make_uint4(pk(v[0], v[1]), pk(v[2], v[3]), pk(v[4], v[5]), pk(v[6], v[7]));
    }
};

template <typename T, bool SILU>
__device__ __forceinline__ float activate(float v) {
    if (!SILU) return v;
    return IO<T>::kFastGate ? silu_fast(v) : silu_accurate(v);
}

template <typename T, int W, bool SILU, bool VEC>
__global__ void __launch_bounds__(kConvThreads)
conv1d_kernel(const ConvArgs a) {
    constexpr int H = W - 1;                 // carried inputs
    constexpr unsigned FULL = 0xffffffffu;
    const int lane = threadIdx.x & 31;
    const int64_t L = a.seqlen;
    const int64_t segs = (L + kSegTokens - 1) / kSegTokens;
    const int64_t unit = (int64_t)blockIdx.x * (kConvThreads / 32) + threadIdx.x / 32;
    const int64_t rows = a.batch * a.dim;
    if (unit >= rows * segs) return;         // whole warps leave together
    const int64_t row = unit / segs, seg = unit % segs;
    const int64_t d = row % a.dim;
    const T *x = static_cast<const T *>(a.x) + row * L;
    T *u = static_cast<T *>(a.u) + row * L;
    const T *sin = a.state_in ? static_cast<const T *>(a.state_in) + row * H : nullptr;

    float w[W];
#pragma unroll
    for (int k = 0; k < W; ++k) w[k] = __ldg(a.w + d * W + k);
    const float bias = a.bias ? __ldg(a.bias + d) : 0.f;
    const int64_t tseg = seg * kSegTokens;

    // the input at time s (s may be negative: the carried state)
    auto x_at = [&](int64_t s) -> float {
        if (s >= 0) return s < L ? IO<T>::to_f(x[s]) : 0.f;
        return sin ? IO<T>::to_f(sin[H + s]) : 0.f;
    };

    float xv[kGran][8];
#pragma unroll
    for (int r = 0; r < kGran; ++r) {
        const int64_t t = tseg + 256 * r + 8 * lane;
        if (VEC) {
            // L is a multiple of 8 here: a granule is wholly inside or outside
            if (t < L) {
                Vec8<T>::load(x + t, xv[r]);
            } else {
#pragma unroll
                for (int i = 0; i < 8; ++i) xv[r][i] = 0.f;
            }
        } else {
#pragma unroll
            for (int i = 0; i < 8; ++i) xv[r][i] = (t + i < L) ? IO<T>::to_f(x[t + i]) : 0.f;
        }
    }

#pragma unroll
    for (int r = 0; r < kGran; ++r) {
        const int64_t t = tseg + 256 * r + 8 * lane;
        float win[H + 8];
#pragma unroll
        for (int i = 0; i < H; ++i) {
            const float left = __shfl_up_sync(FULL, xv[r][8 - H + i], 1);
            float wrap = 0.f;
            if (r > 0) wrap = __shfl_sync(FULL, xv[r - 1][8 - H + i], 31);
            win[i] = lane > 0 ? left : (r > 0 ? wrap : x_at(t - H + i));
        }
#pragma unroll
        for (int i = 0; i < 8; ++i) win[H + i] = xv[r][i];
        if (t >= L) continue;
        float out[8];
#pragma unroll
        for (int i = 0; i < 8; ++i) {
            float acc = bias;
#pragma unroll
            for (int k = 0; k < W; ++k) acc = fmaf(w[k], win[i + k], acc);
            out[i] = activate<T, SILU>(acc);
        }
        if (VEC) {
            if (in_range(row * L + t, 8, rows * L)) Vec8<T>::store(u + t, out);
        } else {
#pragma unroll
            for (int i = 0; i < 8; ++i)
                if (t + i < L && in_range(row * L + t + i, 1, rows * L)) u[t + i] = IO<T>::from_f(out[i]);
        }
    }

    // the row's last segment leaves the final carried inputs
    if (H > 0 && a.state_out && seg == segs - 1 && lane < H) {
        T *so = static_cast<T *>(a.state_out) + row * H;
        const int64_t s = L - H + lane;
        if (in_range(row * H + lane, 1, rows * H)) so[lane] = s >= 0 ? x[s] : (sin ? sin[H + s] : IO<T>::from_f(0.f));
    }
}

// Raw 8-token granule as loaded from global memory (converted to fp32 only
// when it is used, so a prefetched granule costs 4 or 8 registers).
template <typename T> struct Raw8;
template <> struct Raw8<float> {
    float4 a, b;
    __device__ __forceinline__ void load(const float *p) {
        a = __ldcs(reinterpret_cast<const float4 *>(p));
        b = __ldcs(reinterpret_cast<const float4 *>(p) + 1);
    }
    __device__ __forceinline__ void zero() { a = b = make_float4(0.f, 0.f, 0.f, 0.f); }
    __device__ __forceinline__ void unpack(float *o) const {
        o[0] = a.x; o[1] = a.y; o[2] = a.z; o[3] = a.w; o[4] = b.x; o[5] = b.y; o[6] = b.z; o[7] = b.w;
    }
    __device__ __forceinline__ static void store(float *p, const float *v) {
        __stcs(reinterpret_cast<float4 *>(p), make_float4(v[0], v[1], v[2], v[3]));
        __stcs(reinterpret_cast<float4 *>(p) + 1, make_float4(v[4], v[5], v[6], v[7]));
    }
};
template <> struct Raw8<__nv_bfloat16> {
    uint4 v;
    __device__ __forceinline__ void load(const __nv_bfloat16 *p) { v = __ldcs(reinterpret_cast<const uint4 *>(p)); }
    __device__ __forceinline__ void zero() { v = make_uint4(0u, 0u, 0u, 0u); }
    __device__ __forceinline__ void unpack(float *o) const {
        using B = IO<__nv_bfloat16>;
        o[0] = B::lo(v.x); o[1] = B::hi(v.x); o[2] = B::lo(v.y); o[3] = B::hi(v.y);
        o[4] = B::lo(v.z); o[5] = B::hi(v.z); o[6] = B::lo(v.w); o[7] = B::hi(v.w);
    }
    __device__ __forceinline__ static void store(__nv_bfloat16 *p, const float *o) {
        __stcs(reinterpret_cast<uint4 *>(p), make_uint4(Vec8<__nv_bfloat16>::pk(o[0], o[1]),
                                                       Vec8<__nv_bfloat16>::pk(o[2], o[3]),
                                                       Vec8<__nv_bfloat16>::pk(o[4], o[5]),
                                                       Vec8<__nv_bfloat16>::pk(o[6], o[7])));
    }
};

// Sequence form for rows whose pitch is a multiple of 16 bytes (L % 8 == 0,
// 16-byte aligned x and u).  Persistent warps stride over the (row, segment)
// units; the next unit's granules, carried inputs and taps are loaded before
// the current unit is computed, so every warp keeps two units of loads in
// flight.
template <typename T, int W, bool SILU>
__global__ void __launch_bounds__(kConvThreads)
conv1d_stream_kernel(const ConvArgs a) {
    constexpr int H = W - 1;
    constexpr unsigned FULL = 0xffffffffu;
    const int lane = threadIdx.x & 31;
    const int64_t L = a.seqlen;
    // unit = row · segs + seg, row = b · D + d; the host keeps units below 2^31
    const int segs = (int)((L + kSegTokens - 1) / kSegTokens);
    const int dim = (int)a.dim;
    const int units = (int)(a.batch * a.dim) * segs;
    const int stride = gridDim.x * (kConvThreads / 32);
    int unit = blockIdx.x * (kConvThreads / 32) + threadIdx.x / 32;
    if (unit >= units) return;               // whole warps leave together

    // (row, seg, d) of a unit, advanced by `stride` units without dividing
    struct Pos {
        int row, seg, d;
    };
    const int sq = stride / segs, sr = stride % segs, dq = sq % dim;
    auto advance = [&](Pos p) {
        p.seg += sr;
        p.row += sq;
        p.d += dq;
        if (p.d >= dim) p.d -= dim;
        if (p.seg >= segs) {
            p.seg -= segs;
            ++p.row;
            if (++p.d == dim) p.d = 0;
        }
        return p;
    };

    struct Unit {
        Raw8<T> g[kGran];
        float halo[H > 0 ? H : 1];           // lane 0: the inputs before the segment
        float w[W], bias;
    };
    auto fetch = [&](const Pos &p, Unit &f) {
        const T *x = static_cast<const T *>(a.x) + (int64_t)p.row * L;
        const int64_t tseg = (int64_t)p.seg * kSegTokens;
#pragma unroll
        for (int r = 0; r < kGran; ++r) {
            const int64_t t = tseg + 256 * r + 8 * lane;
            if (t < L) f.g[r].load(x + t);
            else f.g[r].zero();
        }
#pragma unroll
        for (int i = 0; i < H; ++i) {
            f.halo[i] = 0.f;
            if (lane == 0) {
                const int64_t s = tseg - H + i;
                if (s >= 0) f.halo[i] = IO<T>::to_f(x[s]);
                else if (a.state_in)
                    f.halo[i] = IO<T>::to_f(static_cast<const T *>(a.state_in)[(int64_t)p.row * H + H + s]);
            }
        }
#pragma unroll
        for (int k = 0; k < W; ++k) f.w[k] = __ldg(a.w + (int64_t)p.d * W + k);
        f.bias = a.bias ? __ldg(a.bias + p.d) : 0.f;
    };

    Pos pos{unit / segs, unit % segs, (unit / segs) % dim};
    Unit cur;
    fetch(pos, cur);
    while (true) {
        const bool more = unit + stride < units;
        const Pos npos = advance(pos);
        Unit nxt;
        if (more) fetch(npos, nxt);

        T *u = static_cast<T *>(a.u) + (int64_t)pos.row * L;
        const int64_t tseg = (int64_t)pos.seg * kSegTokens;
        float tail[H > 0 ? H : 1];           // last H inputs of the previous granule
#pragma unroll
        for (int r = 0; r < kGran; ++r) {
            const int64_t t = tseg + 256 * r + 8 * lane;
            float xv[8];
            cur.g[r].unpack(xv);
            float win[H + 8];
#pragma unroll
            for (int i = 0; i < H; ++i) {
                const float left = __shfl_up_sync(FULL, xv[8 - H + i], 1);
                float wrap = 0.f;
                if (r > 0) wrap = __shfl_sync(FULL, tail[i], 31);
                win[i] = lane > 0 ? left : (r > 0 ? wrap : cur.halo[i]);
            }
#pragma unroll
            for (int i = 0; i < H; ++i) tail[i] = xv[8 - H + i];
#pragma unroll
            for (int i = 0; i < 8; ++i) win[H + i] = xv[i];
            if (t < L) {
                float out[8];
#pragma unroll
                for (int m = 0; m < 4; ++m) {
                    float2 acc = make_float2(cur.bias, cur.bias);
#pragma unroll
                    for (int k = 0; k < W; ++k)
                        acc = __ffma2_rn(make_float2(cur.w[k], cur.w[k]), make_float2(win[2 * m + k], win[2 * m + 1 + k]),
                                         acc);
                    if (SILU) acc = gate2<T>(acc);
                    out[2 * m] = acc.x;
                    out[2 * m + 1] = acc.y;
                }
                if (in_range((int64_t)pos.row * L + t, 8, a.batch * a.dim * L)) Raw8<T>::store(u + t, out);
                // the lane holding the row's last 8 inputs (L % 8 == 0, so L >= 8 > H)
                // leaves the final carried inputs from its registers
                if (H > 0 && a.state_out && t + 8 == L && in_range((int64_t)pos.row * H, H, a.batch * a.dim * H)) {
                    T *so = static_cast<T *>(a.state_out) + (int64_t)pos.row * H;
#pragma unroll
                    for (int i = 0; i < H; ++i) so[i] = IO<T>::from_f(xv[8 - H + i]);
                }
            }
        }
        if (!more) break;
        unit += stride;
        pos = npos;
        cur = nxt;
    }
}

// Decode step: a thread takes 8 consecutive channels of kStepRows batch rows
// (D % 8 == 0, 16-byte aligned state, x, u, taps and bias).  The taps and the
// bias of its channels are loaded once for all its rows; the carried inputs,
// x and u move as 16-byte words.
constexpr int kStepRows = 4;

template <typename T, int W, bool SILU>
__global__ void __launch_bounds__(128)
conv1d_step8_kernel(const ConvStepArgs a) {
    constexpr int H = W - 1;
    constexpr int SW = (8 * H * (int)sizeof(T)) / 16;   // 16-byte words of 8 channels' state
    const int64_t groups = a.dim / 8;
    const int64_t tid = (int64_t)blockIdx.x * blockDim.x + threadIdx.x;
    const int64_t g = tid % groups, rb = tid / groups;   // channel octet, block of rows
    const int64_t b0 = rb * kStepRows;
    if (b0 >= a.batch) return;
    const int64_t d0 = g * 8;
    const int nrows = a.batch - b0 < kStepRows ? (int)(a.batch - b0) : kStepRows;

    uint4 raw[kStepRows][SW > 0 ? SW : 1];
    Raw8<T> xr[kStepRows];
#pragma unroll
    for (int j = 0; j < kStepRows; ++j) {
        if (j < nrows) {
            const int64_t c0 = (b0 + j) * a.dim + d0;
            const uint4 *stp = reinterpret_cast<const uint4 *>(static_cast<const T *>(a.state) + c0 * H);
#pragma unroll
            for (int q = 0; q < SW; ++q) raw[j][q] = __ldcs(stp + q);
            xr[j].load(static_cast<const T *>(a.x) + c0);
        }
    }
    float4 wt[2 * W];
#pragma unroll
    for (int q = 0; q < 2 * W; ++q) wt[q] = __ldg(reinterpret_cast<const float4 *>(a.w + d0 * W) + q);
    float bias[8] = {0.f, 0.f, 0.f, 0.f, 0.f, 0.f, 0.f, 0.f};
    if (a.bias) {
        const float4 b0v = __ldg(reinterpret_cast<const float4 *>(a.bias + d0));
        const float4 b1v = __ldg(reinterpret_cast<const float4 *>(a.bias + d0) + 1);
        bias[0] = b0v.x; bias[1] = b0v.y; bias[2] = b0v.z; bias[3] = b0v.w;
        bias[4] = b1v.x; bias[5] = b1v.y; bias[6] = b1v.z; bias[7] = b1v.w;
    }
    const float *wf = reinterpret_cast<const float *>(wt);   // [8 channels][W]

#pragma unroll
    for (int j = 0; j < kStepRows; ++j) {
        if (j >= nrows) break;
        const int64_t c0 = (b0 + j) * a.dim + d0;
        const T *sv = reinterpret_cast<const T *>(raw[j]);
        float xin[8];
        xr[j].unpack(xin);
        float out[8];
#pragma unroll
        for (int c = 0; c < 8; ++c) {
            float acc = bias[c];
#pragma unroll
            for (int k = 0; k < H; ++k) acc = fmaf(wf[c * W + k], IO<T>::to_f(sv[c * H + k]), acc);
            acc = fmaf(wf[c * W + H], xin[c], acc);
            out[c] = activate<T, SILU>(acc);
        }
        if (in_range(c0, 8, a.batch * a.dim)) Raw8<T>::store(static_cast<T *>(a.u) + c0, out);
        if (H > 0 && in_range(c0 * H, 8 * H, a.batch * a.dim * H)) {
            // the state drops its oldest input and appends this token's, moved
            // as the loaded bits
            uint4 nw[SW > 0 ? SW : 1];
            T *nv = reinterpret_cast<T *>(nw);
            const T *xv = reinterpret_cast<const T *>(&xr[j]);
#pragma unroll
            for (int c = 0; c < 8; ++c) {
#pragma unroll
                for (int k = 0; k + 1 < H; ++k) nv[c * H + k] = sv[c * H + k + 1];
                nv[c * H + H - 1] = xv[c];
            }
            uint4 *stp = reinterpret_cast<uint4 *>(static_cast<T *>(a.state) + c0 * H);
#pragma unroll
            for (int q = 0; q < SW; ++q) __stcs(stp + q, nw[q]);
        }
    }
}

template <typename T, int W, bool SILU>
__global__ void __launch_bounds__(256)
conv1d_step_kernel(const ConvStepArgs a) {
    constexpr int H = W - 1;
    const int64_t c = (int64_t)blockIdx.x * blockDim.x + threadIdx.x;
    if (c >= a.batch * a.dim) return;
    const int64_t d = c % a.dim;
    T *st = static_cast<T *>(a.state) + c * H;
    float win[W];
#pragma unroll
    for (int k = 0; k < H; ++k) win[k] = IO<T>::to_f(st[k]);
    const T xin = static_cast<const T *>(a.x)[c];
    win[H] = IO<T>::to_f(xin);
    float acc = a.bias ? __ldg(a.bias + d) : 0.f;
#pragma unroll
    for (int k = 0; k < W; ++k) acc = fmaf(__ldg(a.w + d * W + k), win[k], acc);
    if (in_range(c, 1, a.batch * a.dim)) static_cast<T *>(a.u)[c] = IO<T>::from_f(activate<T, SILU>(acc));
    if (!in_range(c * H, H, a.batch * a.dim * H)) return;
#pragma unroll
    for (int k = 0; k + 1 < H; ++k) st[k] = IO<T>::from_f(win[k + 1]);
    if (H > 0) st[H - 1] = xin;
}

template <typename T, int W, bool SILU>
cudaError_t launch_seq(const ConvArgs &a, cudaStream_t stream) {
    const int64_t segs = (a.seqlen + kSegTokens - 1) / kSegTokens;
    const int64_t units = a.batch * a.dim * segs;
    const int64_t blocks = (units + kConvThreads / 32 - 1) / (kConvThreads / 32);
    if (blocks > INT32_MAX) return cudaErrorInvalidConfiguration;
    const size_t es = sizeof(T);
    // the streaming kernel indexes units and rows in 32 bits
    const bool vec = a.seqlen % 8 == 0 && (reinterpret_cast<uintptr_t>(a.x) % 16) == 0 &&
                     (reinterpret_cast<uintptr_t>(a.u) % 16) == 0 && es * 8 % 16 == 0 && units < (INT32_MAX / 2);
    if (vec) {
        // persistent: as many blocks as fit at once
        static PerDevice per_device;  // blocks per SM, per instantiation
        int resident = 0;
        const cudaError_t e = per_device.get(
            [&](int *v) {
                int per_sm = 0;
                const cudaError_t r = cudaOccupancyMaxActiveBlocksPerMultiprocessor(
                    &per_sm, conv1d_stream_kernel<T, W, SILU>, kConvThreads, 0);
                *v = per_sm > 0 ? per_sm : 1;
                return r;
            },
            &resident);
        if (e != cudaSuccess) return e;
        const int64_t grid = std::min<int64_t>(blocks, (int64_t)resident * sm_count());
        conv1d_stream_kernel<T, W, SILU><<<(unsigned)grid, kConvThreads, 0, stream>>>(a);
    } else {
        conv1d_kernel<T, W, SILU, false><<<(unsigned)blocks, kConvThreads, 0, stream>>>(a);
    }
    return cudaGetLastError();
}

template <typename T, int W>
cudaError_t launch_seq_w(const ConvArgs &a, cudaStream_t stream) {
    return a.silu ? launch_seq<T, W, true>(a, stream) : launch_seq<T, W, false>(a, stream);
}

template <typename T>
cudaError_t launch_seq_t(const ConvArgs &a, cudaStream_t stream) {
    switch (a.width) {
        case 1: return launch_seq_w<T, 1>(a, stream);
        case 2: return launch_seq_w<T, 2>(a, stream);
        case 3: return launch_seq_w<T, 3>(a, stream);
        case 4: return launch_seq_w<T, 4>(a, stream);
    }
    return cudaErrorInvalidValue;
}

template <typename T, int W>
cudaError_t launch_step_w(const ConvStepArgs &a, cudaStream_t stream) {
    const int64_t n = a.batch * a.dim;
    auto al16 = [](const void *p) { return (reinterpret_cast<uintptr_t>(p) & 15) == 0; };
    const bool wide = a.dim % 8 == 0 && al16(a.x) && al16(a.u) && al16(a.w) && (!a.bias || al16(a.bias)) &&
                      (W == 1 || al16(a.state));
    if (wide) {
        const int64_t threads = (a.dim / 8) * ((a.batch + kStepRows - 1) / kStepRows);
        const int64_t blocks = (threads + 127) / 128;
        if (blocks > INT32_MAX) return cudaErrorInvalidConfiguration;
        if (a.silu)
            conv1d_step8_kernel<T, W, true><<<(unsigned)blocks, 128, 0, stream>>>(a);
        else
            conv1d_step8_kernel<T, W, false><<<(unsigned)blocks, 128, 0, stream>>>(a);
        return cudaGetLastError();
    }
    const int64_t blocks = (n + 255) / 256;
    if (blocks > INT32_MAX) return cudaErrorInvalidConfiguration;
    if (a.silu)
        conv1d_step_kernel<T, W, true><<<(unsigned)blocks, 256, 0, stream>>>(a);
    else
        conv1d_step_kernel<T, W, false><<<(unsigned)blocks, 256, 0, stream>>>(a);
    return cudaGetLastError();
}

template <typename T>
cudaError_t launch_step_t(const ConvStepArgs &a, cudaStream_t stream) {
    switch (a.width) {
        case 1: return launch_step_w<T, 1>(a, stream);
        case 2: return launch_step_w<T, 2>(a, stream);
        case 3: return launch_step_w<T, 3>(a, stream);
        case 4: return launch_step_w<T, 4>(a, stream);
    }
    return cudaErrorInvalidValue;
}

}  // namespace

cudaError_t conv_launch(const ConvArgs &a, bool bf16, cudaStream_t stream) {
    return bf16 ? launch_seq_t<__nv_bfloat16>(a, stream) : launch_seq_t<float>(a, stream);
}

cudaError_t conv_step_launch(const ConvStepArgs &a, bool bf16, cudaStream_t stream) {
    return bf16 ? launch_step_t<__nv_bfloat16>(a, stream) : launch_step_t<float>(a, stream);
}

SSM_DEBUG_WORD_READER(debug_word_conv)

}  // namespace ssm
