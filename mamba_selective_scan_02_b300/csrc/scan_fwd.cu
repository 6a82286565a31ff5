// scan_fwd.cu — the fused Mamba selective scan for sm_103a.
//
// What one launch computes is the recurrence of "Mamba and selective state
// spaces, from first principles" ("Selection", "Discretisation: zero-order
// hold", "The hardware-aware scan"): for every channel (b, d) and state n,
//   Δ = softplus(Δraw + bias), Ā = exp(Δ·A), h = Ā·h + Δ·B·u,
//   y = (C·h + D·u)·silu(z),
// writing only y (b × D × L) and the final state — never Ā, B̄ or any h_t.
//
// Design (B300-first, not the pages' kernel).  On this part one state update
// costs one MUFU exponential and four FP32 operations (Δ·A, B·Δu, Ā·h + B̄u,
// C·h); the SM retires 32 exponentials but only 128 FP32 lanes per clock, and
// issues one instruction per scheduler per clock, so the kernel is built to
// spend as few instructions per state update as possible:
//   * Channels are the parallel axis.  A thread owns SPT consecutive states of
//     one channel and walks the time axis sequentially with them in registers;
//     NG = N/SPT adjacent lanes share a channel.  State arithmetic is packed
//     f32x2 (two states per instruction); Ā is ex2.approx on Δ·A·log2e.
//   * Per tile of TT tokens, one elected thread moves u, Δraw, z (CH channels ×
//     TT tokens) and B, C (N × TT, shared by every channel of the CTA) into
//     shared memory with 3-D TMA copies on an mbarrier; the y tile leaves with
//     a TMA store.  The next tile's copies overlap the current tile's scan.
//   * Three phases per tile.  Pre-pass: the per-token nonlinearities (softplus,
//     Δ·u, silu(z), D·u·gate) once per (channel, token), and B, C widened to
//     fp32 in token-major rows so a thread reads its states with one 16-byte
//     load.  Scan: only loads of those fp32 rows, packed FMAs and ex2; each lane
//     leaves its partial C·h per token in shared memory.  Epilogue: the NG
//     partials of a token are added, gated, rounded and staged for the store.
//   * Long sequences are cut into chunks that run concurrently.  The
//     composition of affine steps is associative (first-principles page,
//     "The hardware-aware scan"): an aggregate pass computes each chunk's pair
//     (Π Ā, h_end from zero), a carry pass chains the pairs from h0, and the
//     main pass rescans every chunk from its carried state.
#include <algorithm>
#include <cstring>

#include "ssm_device.cuh"
#include "ssm_internal.h"

#ifndef SSM_SCAN_SPT
#define SSM_SCAN_SPT 8
#endif
#ifndef SSM_SCAN_TT
#define SSM_SCAN_TT 16
#endif

namespace ssm {

constexpr int kSPT = SSM_SCAN_SPT;     // states per thread for N = 16
constexpr int kTT = SSM_SCAN_TT;       // tokens per tile
constexpr int kNT = 128;               // threads per CTA
constexpr int kWaitLimit = 1 << 22;    // mbarrier polls before giving up

constexpr int al128(int x) { return (x + 127) / 128 * 128; }

// Shared-memory layout of one CTA (byte offsets; TMA destinations 128-B aligned).
template <typename T, int SPT, int NG, int TT> struct Tile {
    static_assert(SPT % 4 == 0 && TT % 8 == 0, "tile shape");
    static constexpr int CH = kNT / NG;        // channels per CTA
    static constexpr int NP = SPT * NG;        // states covered (>= N)
    static constexpr int BCP = NP + 4;         // fp32 B/C row pitch in floats (16-B rows)
    static constexpr int DDP = TT + 1;         // (Δ, Δ, Δu, Δu) row pitch in float4
    static constexpr int GDP = TT / 2 + 1;     // (g0, g1, D·u·g0, D·u·g1) row pitch in float4
    static constexpr int PTP = TT + 4;         // partial C·h row pitch in floats
    static constexpr int ES = (int)sizeof(T);
    static constexpr int raw_seq = CH * TT * ES;
    static constexpr int raw_bc = NP * TT * ES;
    static constexpr int off_u = 0;
    static constexpr int off_d = off_u + al128(raw_seq);
    static constexpr int off_z = off_d + al128(raw_seq);
    static constexpr int off_B = off_z + al128(raw_seq);
    static constexpr int off_C = off_B + al128(raw_bc);
    static constexpr int off_out = off_C + al128(raw_bc);
    static constexpr int off_dd = off_out + al128(raw_seq);
    static constexpr int off_gd = off_dd + al128(CH * DDP * 16);
    static constexpr int off_Bf = off_gd + al128(CH * GDP * 16);
    static constexpr int off_Cf = off_Bf + al128(TT * BCP * 4);
    static constexpr int off_part = off_Cf + al128(TT * BCP * 4);
    static constexpr int off_bias = off_part + al128(CH * NG * PTP * 4);
    static constexpr int off_skip = off_bias + CH * 4;
    static constexpr int off_bar = (off_skip + CH * 4 + 15) / 16 * 16;
    static constexpr int bytes = off_bar + 16;
};

struct Maps {
    CUtensorMap u, d, z, B, C, y;
};

// MODE 0: full scan writing y (and hL for the last chunk).
// MODE 1: chunk aggregate (Π Ā, h_end from zero) for chunks 0..K-2.
template <typename T, int SPT, int NG, int TT, bool HAS_Z, bool TMA, int MODE>
__global__ void __launch_bounds__(kNT)
scan_kernel(const __grid_constant__ Maps maps, const ScanArgs a) {
    using S = Tile<T, SPT, NG, TT>;
    constexpr int CH = S::CH, NP = S::NP;
    constexpr int NQ = SPT / 2;  // float2 state pairs per thread
    extern __shared__ __align__(128) unsigned char smem[];
    T *u_s = reinterpret_cast<T *>(smem + S::off_u);
    T *d_s = reinterpret_cast<T *>(smem + S::off_d);
    T *z_s = reinterpret_cast<T *>(smem + S::off_z);
    T *B_s = reinterpret_cast<T *>(smem + S::off_B);
    T *C_s = reinterpret_cast<T *>(smem + S::off_C);
    T *out_s = reinterpret_cast<T *>(smem + S::off_out);
    float4 *dd = reinterpret_cast<float4 *>(smem + S::off_dd);
    float4 *gd = reinterpret_cast<float4 *>(smem + S::off_gd);
    float *Bf = reinterpret_cast<float *>(smem + S::off_Bf);
    float *Cf = reinterpret_cast<float *>(smem + S::off_Cf);
    float *part = reinterpret_cast<float *>(smem + S::off_part);
    float *bias_s = reinterpret_cast<float *>(smem + S::off_bias);
    float *skip_s = reinterpret_cast<float *>(smem + S::off_skip);
    uint64_t *bar = reinterpret_cast<uint64_t *>(smem + S::off_bar);

    const int tid = threadIdx.x;
    const int c = tid / NG;          // channel within the CTA
    const int g = tid % NG;          // state group: states SPT·g .. SPT·g + SPT-1
    const int d0 = blockIdx.x * CH;
    const int b = blockIdx.y;
    const int k = blockIdx.z;        // chunk
    const int D = a.dim, N = a.dstate, L = a.seqlen;
    const int d = d0 + c;
    const bool live = d < D;
    const int t_begin = k * a.chunk_len;
    const int t_end = min(L, t_begin + a.chunk_len);
    const int ntiles = (t_end - t_begin + TT - 1) / TT;

    // ---- per-thread constants: A·log2e for the thread's states, initial state
    float2 A2[NQ], h[NQ];
#pragma unroll
    for (int q = 0; q < NQ; ++q) {
        float av[2] = {0.f, 0.f}, hv[2] = {0.f, 0.f};
#pragma unroll
        for (int j = 0; j < 2; ++j) {
            const int n = SPT * g + 2 * q + j;
            if (live && n < N) {
                av[j] = a.A[(size_t)d * N + n] * kLog2e;
                if (MODE == 0) {
                    // With several chunks h0 is read only by the carry pass, so
                    // hL may share h0's buffer.
                    if (a.nchunks > 1)
                        hv[j] = a.carry[(((size_t)b * D + d) * a.nchunks + k) * N + n];
                    else if (a.h0)
                        hv[j] = a.h0[((size_t)b * D + d) * N + n];
                }
            }
        }
        A2[q] = make_float2(av[0], av[1]);
        h[q] = make_float2(hv[0], hv[1]);
    }
    for (int i = tid; i < CH; i += kNT) {
        const int dd_ = d0 + i;
        bias_s[i] = (dd_ < D && a.bias) ? a.bias[dd_] : 0.f;
        skip_s[i] = (dd_ < D && a.Dskip) ? a.Dskip[dd_] : 0.f;
    }
    // Padded state columns of the fp32 B/C rows stay zero for the whole launch.
    for (int i = tid; i < TT * S::BCP; i += kNT) {
        Bf[i] = 0.f;
        Cf[i] = 0.f;
    }
    if (TMA && tid == 0) {
        mbar_init(bar, 1);
        fence_mbar_init();
    }
    __syncthreads();

    constexpr uint32_t seq_bytes = CH * TT * sizeof(T);
    const uint32_t bc_bytes = (uint32_t)N * TT * sizeof(T);
    auto issue_loads = [&](int tile) {
        const int t0 = t_begin + tile * TT;
        const uint32_t bytes = (MODE == 0 ? (HAS_Z ? 3u : 2u) : 2u) * seq_bytes +
                               (MODE == 0 ? 2u : 1u) * bc_bytes;
        mbar_arrive_expect_tx(bar, bytes);
        tma_load_3d(u_s, &maps.u, bar, t0, d0, b);
        tma_load_3d(d_s, &maps.d, bar, t0, d0, b);
        if (MODE == 0 && HAS_Z) tma_load_3d(z_s, &maps.z, bar, t0, d0, b);
        tma_load_3d(B_s, &maps.B, bar, t0, 0, b);
        if (MODE == 0) tma_load_3d(C_s, &maps.C, bar, t0, 0, b);
    };
    // Plain loads for shapes TMA cannot describe (row pitch not a multiple of 16 B).
    auto generic_loads = [&](int tile) {
        const int t0 = t_begin + tile * TT;
        const T *gu = static_cast<const T *>(a.u), *gdl = static_cast<const T *>(a.delta);
        const T *gz = static_cast<const T *>(a.z);
        for (int i = tid; i < CH * TT; i += kNT) {
            const int cc = i / TT, tt = i % TT, dch = d0 + cc, t = t0 + tt;
            const bool in = dch < D && t < L;
            const size_t off = ((size_t)b * D + dch) * L + t;
            u_s[i] = in ? gu[off] : T(0.f);
            d_s[i] = in ? gdl[off] : T(0.f);
            if (MODE == 0 && HAS_Z) z_s[i] = in ? gz[off] : T(0.f);
        }
        const T *gB = static_cast<const T *>(a.B), *gC = static_cast<const T *>(a.C);
        for (int i = tid; i < N * TT; i += kNT) {
            const int n = i / TT, tt = i % TT, t = t0 + tt;
            const bool in = t < L;
            const size_t off = ((size_t)b * N + n) * L + t;
            B_s[i] = in ? gB[off] : T(0.f);
            if (MODE == 0) C_s[i] = in ? gC[off] : T(0.f);
        }
    };

    if (TMA && tid == 0 && ntiles > 0) issue_loads(0);

    float dsum = 0.f;  // Σ Δ over the chunk (MODE 1)
    bool failed = false;

    for (int tile = 0; tile < ntiles; ++tile) {
        const int t0 = t_begin + tile * TT;
        if (TMA) {
            failed = !mbar_wait_bounded(bar, tile & 1, kWaitLimit);
        } else {
            generic_loads(tile);
            __syncthreads();
        }

        // ---- pre-pass A: per (channel, token), 8 consecutive tokens per item
        constexpr int MB = TT / 8;
        for (int it = tid; it < CH * MB; it += kNT) {
            const int cc = it / MB, tb = 8 * (it % MB);
            float uf[8], df[8], zf[8];
            IO<T>::load8(u_s + cc * TT + tb, uf);
            IO<T>::load8(d_s + cc * TT + tb, df);
            if (MODE == 0 && HAS_Z) IO<T>::load8(z_s + cc * TT + tb, zf);
            const float bias = bias_s[cc];
            const float skip = skip_s[cc];
            const int valid = t_end - (t0 + tb);  // tokens of this item inside the chunk
#pragma unroll
            for (int j = 0; j < 8; j += 2) {
                float dl0 = df[j] + bias, dl1 = df[j + 1] + bias;
                if (a.delta_softplus) {
                    dl0 = IO<T>::softplus(dl0);
                    dl1 = IO<T>::softplus(dl1);
                }
                if (j >= valid) dl0 = 0.f;  // Δ = 0 keeps the state: Ā = 1, B̄u = 0
                if (j + 1 >= valid) dl1 = 0.f;
                const float2 du = __fmul2_rn(make_float2(dl0, dl1), make_float2(uf[j], uf[j + 1]));
                dd[cc * S::DDP + tb + j] = make_float4(dl0, dl0, du.x, du.x);
                dd[cc * S::DDP + tb + j + 1] = make_float4(dl1, dl1, du.y, du.y);
                if (MODE == 0) {
                    float2 gt = make_float2(1.f, 1.f);
                    if (HAS_Z) gt = make_float2(gate_of<T>(zf[j]), gate_of<T>(zf[j + 1]));
                    const float2 su = __fmul2_rn(make_float2(skip, skip), make_float2(uf[j], uf[j + 1]));
                    const float2 dug = __fmul2_rn(su, gt);
                    gd[cc * S::GDP + (tb + j) / 2] = make_float4(gt.x, gt.y, dug.x, dug.y);
                }
            }
        }
        // ---- pre-pass B: B (and C) widened to fp32, token-major rows, 4 × 4 blocks
        {
            constexpr int NB = NP / 4, TB = TT / 4;
            constexpr int UNITS = (MODE == 0 ? 2 : 1) * NB * TB;
            for (int it = tid; it < UNITS; it += kNT) {
                const int mat = it / (NB * TB), r = it % (NB * TB);
                const int nb = r / TB, tb = r % TB;
                const T *src = mat ? C_s : B_s;
                float *dst = mat ? Cf : Bf;
                float4 v[4];
#pragma unroll
                for (int i = 0; i < 4; ++i) {
                    const int n = 4 * nb + i;
                    v[i] = n < N ? IO<T>::load4(src + n * TT + 4 * tb) : make_float4(0.f, 0.f, 0.f, 0.f);
                }
                float *row = dst + (4 * tb) * S::BCP + 4 * nb;
                *reinterpret_cast<float4 *>(row) = make_float4(v[0].x, v[1].x, v[2].x, v[3].x);
                *reinterpret_cast<float4 *>(row + S::BCP) = make_float4(v[0].y, v[1].y, v[2].y, v[3].y);
                *reinterpret_cast<float4 *>(row + 2 * S::BCP) = make_float4(v[0].z, v[1].z, v[2].z, v[3].z);
                *reinterpret_cast<float4 *>(row + 3 * S::BCP) = make_float4(v[0].w, v[1].w, v[2].w, v[3].w);
            }
        }
        if (TMA && MODE == 0 && tid == 0) bulk_wait_read0();  // out_s free again
        if (__syncthreads_or(failed)) {
            record_error(a.status, 4 /* SSM_ERR_TIMEOUT */);
            if (TMA && MODE == 0 && tid == 0) bulk_wait0();
            return;
        }
        if (TMA && tid == 0 && tile + 1 < ntiles) {
            fence_proxy_async_smem();
            issue_loads(tile + 1);
        }

        // ---- scan: TT tokens, four at a time, SPT states per thread
        const float4 *ddc = dd + c * S::DDP;
#pragma unroll 1
        for (int tb = 0; tb < TT; tb += 4) {
            float p[4];
#pragma unroll
            for (int kk = 0; kk < 4; ++kk) {
                const int t = tb + kk;
                const float4 dv = ddc[t];
                const float2 d2 = make_float2(dv.x, dv.y), du2 = make_float2(dv.z, dv.w);
                const float *Brow = Bf + t * S::BCP + SPT * g;
                const float *Crow = Cf + t * S::BCP + SPT * g;
                float2 acc = make_float2(0.f, 0.f);
#pragma unroll
                for (int q4 = 0; q4 < SPT / 4; ++q4) {
                    const float4 bq = *reinterpret_cast<const float4 *>(Brow + 4 * q4);
                    const float2 x0 = __fmul2_rn(d2, A2[2 * q4]);
                    const float2 x1 = __fmul2_rn(d2, A2[2 * q4 + 1]);
                    const float2 a0 = make_float2(ex2(x0.x), ex2(x0.y));
                    const float2 a1 = make_float2(ex2(x1.x), ex2(x1.y));
                    const float2 bu0 = __fmul2_rn(make_float2(bq.x, bq.y), du2);
                    const float2 bu1 = __fmul2_rn(make_float2(bq.z, bq.w), du2);
                    h[2 * q4] = __ffma2_rn(a0, h[2 * q4], bu0);
                    h[2 * q4 + 1] = __ffma2_rn(a1, h[2 * q4 + 1], bu1);
                    if (MODE == 0) {
                        const float4 cq = *reinterpret_cast<const float4 *>(Crow + 4 * q4);
                        acc = q4 == 0 ? __fmul2_rn(make_float2(cq.x, cq.y), h[0])
                                      : __ffma2_rn(make_float2(cq.x, cq.y), h[2 * q4], acc);
                        acc = __ffma2_rn(make_float2(cq.z, cq.w), h[2 * q4 + 1], acc);
                    }
                }
                if (MODE == 0) p[kk] = acc.x + acc.y;
                else dsum += dv.x;
            }
            if (MODE == 0)
                *reinterpret_cast<float4 *>(part + (c * NG + g) * S::PTP + tb) = make_float4(p[0], p[1], p[2], p[3]);
        }
        __syncthreads();  // partial sums complete; pre-pass buffers free

        if (MODE == 0) {
            // ---- epilogue: y for token pairs = (Σ_g partials)·gate + D·u·gate
            constexpr int PAIRS = TT / 2;
            for (int it = tid; it < CH * PAIRS; it += kNT) {
                const int cc = it / PAIRS, tp = it % PAIRS;
                const float *pr = part + cc * NG * S::PTP + 2 * tp;
                float2 sum = *reinterpret_cast<const float2 *>(pr);
#pragma unroll
                for (int gg = 1; gg < NG; ++gg)
                    sum = __fadd2_rn(sum, *reinterpret_cast<const float2 *>(pr + gg * S::PTP));
                const float4 gv = gd[cc * S::GDP + tp];
                const float2 y2 = __ffma2_rn(sum, make_float2(gv.x, gv.y), make_float2(gv.z, gv.w));
                IO<T>::store2(out_s + cc * TT + 2 * tp, y2);
            }
            if (TMA) {
                fence_proxy_async_smem();
                __syncthreads();
                if (tid == 0) {
                    tma_store_3d(&maps.y, out_s, t0, d0, b);
                    bulk_commit();
                }
            } else {
                __syncthreads();
                T *gy = static_cast<T *>(a.y);
                for (int i = tid; i < CH * TT; i += kNT) {
                    const int cc = i / TT, tt = i % TT, dch = d0 + cc, t = t0 + tt;
                    if (dch < D && t < t_end) gy[((size_t)b * D + dch) * L + t] = out_s[i];
                }
            }
        }
    }
    if (TMA && MODE == 0 && tid == 0) bulk_wait0();

    if (MODE == 0) {
        if (k == a.nchunks - 1 && a.hL && live) {
#pragma unroll
            for (int q = 0; q < NQ; ++q) {
                const int n = SPT * g + 2 * q;
                if (n < N) a.hL[((size_t)b * D + d) * N + n] = h[q].x;
                if (n + 1 < N) a.hL[((size_t)b * D + d) * N + n + 1] = h[q].y;
            }
        }
    } else if (live) {
#pragma unroll
        for (int q = 0; q < NQ; ++q) {
#pragma unroll
            for (int j = 0; j < 2; ++j) {
                const int n = SPT * g + 2 * q + j;
                const float av = j ? A2[q].y : A2[q].x;
                const float hv = j ? h[q].y : h[q].x;
                if (n < N)
                    a.agg[(((size_t)b * D + d) * (a.nchunks - 1) + k) * N + n] = make_float2(ex2(av * dsum), hv);
            }
        }
    }
}

// Chains the chunk aggregates from h0: carry[0] = h0 and
// carry[k+1] = P_k · carry[k] + S_k, the state chunk k+1 starts from.
// One thread per (b, d, n).
__global__ void carry_kernel(const ScanArgs a) {
    const size_t i = (size_t)blockIdx.x * blockDim.x + threadIdx.x;
    const size_t total = (size_t)a.batch * a.dim * a.dstate;
    if (i >= total) return;
    const size_t bd = i / a.dstate;
    const int n = (int)(i % a.dstate);
    const int K = a.nchunks;
    float h = a.h0 ? a.h0[i] : 0.f;
    a.carry[(bd * K) * a.dstate + n] = h;
    for (int k = 0; k + 1 < K; ++k) {
        const float2 ps = a.agg[(bd * (K - 1) + k) * a.dstate + n];
        h = fmaf(ps.x, h, ps.y);
        a.carry[(bd * K + k + 1) * a.dstate + n] = h;
    }
}

// ------------------------------------------------------------------ host side

namespace {

using EncodeFn = CUresult (*)(CUtensorMap *, CUtensorMapDataType, cuuint32_t, void *, const cuuint64_t *,
                              const cuuint64_t *, const cuuint32_t *, const cuuint32_t *, CUtensorMapInterleave,
                              CUtensorMapSwizzle, CUtensorMapL2promotion, CUtensorMapFloatOOBfill);

EncodeFn encode_fn() {
    static EncodeFn fn = nullptr;
    static bool tried = false;
    if (!tried) {
        tried = true;
        void *p = nullptr;
        cudaDriverEntryPointQueryResult q;
        if (cudaGetDriverEntryPointByVersion("cuTensorMapEncodeTiled", &p, 12000, cudaEnableDefault, &q) ==
                cudaSuccess &&
            q == cudaDriverEntryPointSuccess)
            fn = reinterpret_cast<EncodeFn>(p);
    }
    return fn;
}

// 3-D map over a (dim2 × dim1 × dim0) row-major tensor, box (box0, box1, 1).
bool make_map(CUtensorMap *m, CUtensorMapDataType dt, size_t es, const void *ptr, uint64_t dim0, uint64_t dim1,
              uint64_t dim2, uint32_t box0, uint32_t box1) {
    EncodeFn fn = encode_fn();
    if (!fn) return false;
    const cuuint64_t dims[3] = {dim0, dim1, dim2};
    const cuuint64_t strides[2] = {dim0 * es, dim0 * dim1 * es};
    const cuuint32_t box[3] = {box0, box1, 1};
    const cuuint32_t estr[3] = {1, 1, 1};
    return fn(m, dt, 3, const_cast<void *>(ptr), dims, strides, box, estr, CU_TENSOR_MAP_INTERLEAVE_NONE,
              CU_TENSOR_MAP_SWIZZLE_NONE, CU_TENSOR_MAP_L2_PROMOTION_L2_256B,
              CU_TENSOR_MAP_FLOAT_OOB_FILL_NONE) == CUDA_SUCCESS;
}

template <typename T, int SPT, int NG, bool HAS_Z, bool TMA, int MODE>
cudaError_t launch_one(const Maps &maps, const ScanArgs &a, dim3 grid, cudaStream_t st) {
    using S = Tile<T, SPT, NG, kTT>;
    auto kern = scan_kernel<T, SPT, NG, kTT, HAS_Z, TMA, MODE>;
    static bool attr_set = false;
    if (!attr_set) {
        cudaError_t e = cudaFuncSetAttribute(kern, cudaFuncAttributeMaxDynamicSharedMemorySize, S::bytes);
        if (e != cudaSuccess) return e;
        attr_set = true;
    }
    kern<<<grid, kNT, S::bytes, st>>>(maps, a);
    return cudaGetLastError();
}

template <typename T, int SPT, int NG, bool HAS_Z, bool TMA>
cudaError_t launch_all(const Maps &maps, const ScanArgs &a, cudaStream_t st) {
    constexpr int CH = kNT / NG;
    const unsigned gx = (unsigned)((a.dim + CH - 1) / CH);
    cudaError_t e;
    if (a.nchunks > 1) {
        e = launch_one<T, SPT, NG, false, TMA, 1>(maps, a, dim3(gx, a.batch, a.nchunks - 1), st);
        if (e != cudaSuccess) return e;
        const size_t total = (size_t)a.batch * a.dim * a.dstate;
        carry_kernel<<<(unsigned)((total + 255) / 256), 256, 0, st>>>(a);
        e = cudaGetLastError();
        if (e != cudaSuccess) return e;
    }
    return launch_one<T, SPT, NG, HAS_Z, TMA, 0>(maps, a, dim3(gx, a.batch, a.nchunks), st);
}

template <typename T, int SPT, int NG>
cudaError_t dispatch_z_tma(const Maps &maps, const ScanArgs &a, bool tma, cudaStream_t st) {
    const bool z = a.z != nullptr;
    if (tma)
        return z ? launch_all<T, SPT, NG, true, true>(maps, a, st) : launch_all<T, SPT, NG, false, true>(maps, a, st);
    return z ? launch_all<T, SPT, NG, true, false>(maps, a, st) : launch_all<T, SPT, NG, false, false>(maps, a, st);
}

// States per thread and threads per channel for a state size N: four states
// per thread for N <= 4, otherwise kSPT with as many lanes as N needs.
struct Split {
    int spt, ng;
};
Split split_for(int64_t dstate) {
    if (dstate <= 4) return {4, 1};
    int ng = (int)((dstate + kSPT - 1) / kSPT);
    ng = ng <= 1 ? 1 : (ng <= 2 ? 2 : 4);
    return {kSPT, ng};
}

template <typename T>
cudaError_t dispatch_split(const Maps &maps, const ScanArgs &a, Split sp, bool tma, cudaStream_t st) {
    if (sp.spt == 4 && sp.ng == 1) return dispatch_z_tma<T, 4, 1>(maps, a, tma, st);
#if SSM_SCAN_SPT == 4
    if (sp.ng == 2) return dispatch_z_tma<T, 4, 2>(maps, a, tma, st);
    return dispatch_z_tma<T, 4, 4>(maps, a, tma, st);
#elif SSM_SCAN_SPT == 8
    if (sp.ng == 1) return dispatch_z_tma<T, 8, 1>(maps, a, tma, st);
    return dispatch_z_tma<T, 8, 2>(maps, a, tma, st);
#elif SSM_SCAN_SPT == 16
    return dispatch_z_tma<T, 16, 1>(maps, a, tma, st);
#else
#error "SSM_SCAN_SPT must be 4, 8 or 16"
#endif
}

}  // namespace

int scan_groups(int64_t dstate) { return dstate <= 4 ? 1 : (dstate <= 8 ? 2 : 4); }

int64_t scan_chunk_len(int64_t batch, int64_t dim, int64_t dstate, int64_t seqlen, int64_t requested) {
    if (requested > 0) return std::min<int64_t>(requested, ((seqlen + 63) / 64) * 64);
    // Enough resident warps to keep every scheduler's pipes busy: the fewer
    // states a thread owns, the more warps it takes (4 per scheduler at four
    // states per thread, 1 at sixteen).
    const Split sp = split_for(dstate);
    const int64_t threads = batch * dim * sp.ng;
    const int64_t want = 148LL * 4 * 32 * (16 / sp.spt);
    int64_t K = (want + threads - 1) / threads;
    K = std::max<int64_t>(1, std::min<int64_t>(K, (seqlen + 511) / 512));
    const int64_t len = (seqlen + K - 1) / K;
    return ((len + 63) / 64) * 64;
}

cudaError_t scan_launch(const ScanArgs &a, bool bf16, cudaStream_t st) {
    const Split sp = split_for(a.dstate);
    const int CH = kNT / sp.ng;
    const size_t es = bf16 ? 2 : 4;
    // TMA needs a row pitch that is a multiple of 16 bytes.
    const bool tma = ((size_t)a.seqlen * es) % 16 == 0;
    Maps maps;
    memset(&maps, 0, sizeof(maps));
    if (tma) {
        const CUtensorMapDataType dt = bf16 ? CU_TENSOR_MAP_DATA_TYPE_BFLOAT16 : CU_TENSOR_MAP_DATA_TYPE_FLOAT32;
        bool ok = make_map(&maps.u, dt, es, a.u, a.seqlen, a.dim, a.batch, kTT, CH) &&
                  make_map(&maps.d, dt, es, a.delta, a.seqlen, a.dim, a.batch, kTT, CH) &&
                  make_map(&maps.B, dt, es, a.B, a.seqlen, a.dstate, a.batch, kTT, a.dstate) &&
                  make_map(&maps.C, dt, es, a.C, a.seqlen, a.dstate, a.batch, kTT, a.dstate) &&
                  make_map(&maps.y, dt, es, a.y, a.seqlen, a.dim, a.batch, kTT, CH);
        if (ok && a.z) ok = make_map(&maps.z, dt, es, a.z, a.seqlen, a.dim, a.batch, kTT, CH);
        if (!ok) return cudaErrorInvalidValue;
    }
    return bf16 ? dispatch_split<__nv_bfloat16>(maps, a, sp, tma, st) : dispatch_split<float>(maps, a, sp, tma, st);
}

}  // namespace ssm
