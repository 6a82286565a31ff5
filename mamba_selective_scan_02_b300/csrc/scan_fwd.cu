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

#ifndef SSM_SCAN_TT
#define SSM_SCAN_TT 32
#endif

namespace ssm {

constexpr int kTT = SSM_SCAN_TT;       // tokens per tile (a multiple of 8; chunks are multiples of 64)
constexpr int kCH = 32;                // channels per CTA: one warp, one lane per channel
constexpr int kWaitLimit = 1 << 22;    // mbarrier polls before giving up

__host__ __device__ constexpr int al128(int x) { return (x + 127) / 128 * 128; }

// Shared-memory layout of one CTA (byte offsets; TMA destinations 128-B aligned).
// u, Δraw, z and y tiles are stored as [TT/8][32 channels][8 tokens] so that a
// lane's 8 tokens are one contiguous 16-byte (bf16) or 32-byte (fp32) run and a
// warp's loads cover consecutive banks; each such block is one TMA box.
template <typename T, int SPT, int TT> struct WTile {
    static_assert(SPT % 4 == 0 && TT % 8 == 0, "tile shape");
    static constexpr int ES = (int)sizeof(T);
    static constexpr int NB8 = TT / 8;            // 8-token blocks per tile
    static constexpr int BLK = kCH * 8 * ES;      // one 8-token block of one input
    static constexpr int SEQ = NB8 * BLK;         // one input tile
    static constexpr int BC = SPT * TT * ES;      // one B or C tile (N <= SPT rows)
    static constexpr int BCP = SPT + 4;           // fp32 B/C row pitch in floats (16-B rows)
    static constexpr int BUF = 3 * al128(SEQ) + 2 * al128(BC);  // one stage: u, Δ, z, B, C
    static constexpr int off_u = 0, off_d = al128(SEQ), off_z = 2 * al128(SEQ);
    static constexpr int off_B = 3 * al128(SEQ), off_C = off_B + al128(BC);
    static constexpr int off_out = 2 * BUF;                      // two y tiles
    static constexpr int off_Bf = off_out + 2 * al128(SEQ);
    static constexpr int off_Cf = off_Bf + al128(TT * BCP * 4);
    static constexpr int off_bar = off_Cf + al128(TT * BCP * 4);
    static constexpr int bytes = off_bar + 16;
    static constexpr int OUT = al128(SEQ);        // one y tile
};

struct Maps {
    CUtensorMap u, d, z, B, C, y;
};

template <typename T> struct Pack8;
template <> struct Pack8<float> {
    __device__ __forceinline__ static void store(float *p, const float *v) {
        reinterpret_cast<float4 *>(p)[0] = make_float4(v[0], v[1], v[2], v[3]);
        reinterpret_cast<float4 *>(p)[1] = make_float4(v[4], v[5], v[6], v[7]);
    }
};
template <> struct Pack8<__nv_bfloat16> {
    __device__ __forceinline__ static uint32_t pk(float a, float b) {
        const __nv_bfloat162 v = __floats2bfloat162_rn(a, b);
        return *reinterpret_cast<const uint32_t *>(&v);
    }
    __device__ __forceinline__ static void store(__nv_bfloat16 *p, const float *v) {
        *reinterpret_cast<uint4 *>(p) = make_uint4(pk(v[0], v[1]), pk(v[2], v[3]), pk(v[4], v[5]), pk(v[6], v[7]));
    }
};

// MODE 0: full scan writing y (and hL for the last chunk).
// MODE 1: chunk aggregate (Π Ā, h_end from zero) for chunks 0..K-2.
// One warp per CTA; lane c owns channel d0 + c and all SPT (>= N) of its states.
template <typename T, int SPT, int TT, bool HAS_Z, bool TMA, int MODE>
__global__ void __launch_bounds__(kCH, 1)
scan_kernel(const __grid_constant__ Maps maps, const ScanArgs a) {
    using S = WTile<T, SPT, TT>;
    constexpr int NQ = SPT / 2;      // float2 state pairs per lane
    constexpr int NB8 = S::NB8;
    extern __shared__ __align__(128) unsigned char smem[];
    float *Bf = reinterpret_cast<float *>(smem + S::off_Bf);
    float *Cf = reinterpret_cast<float *>(smem + S::off_Cf);
    uint64_t *bar = reinterpret_cast<uint64_t *>(smem + S::off_bar);

    const int lane = threadIdx.x;
    const int d0 = blockIdx.x * kCH;
    const int b = blockIdx.y;
    const int k = blockIdx.z;        // chunk
    const int D = a.dim, N = a.dstate, L = a.seqlen;
    const int d = d0 + lane;
    const bool live = d < D;
    const int t_begin = k * a.chunk_len;
    const int t_end = min(L, t_begin + a.chunk_len);
    const int ntiles = (t_end - t_begin + TT - 1) / TT;

    // ---- per-lane constants: A·log2e for the channel's states, initial state
    float2 A2[NQ], h[NQ];
#pragma unroll
    for (int q = 0; q < NQ; ++q) {
        float av[2] = {0.f, 0.f}, hv[2] = {0.f, 0.f};
#pragma unroll
        for (int j = 0; j < 2; ++j) {
            const int n = 2 * q + j;
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
    const float bias = (live && a.bias) ? a.bias[d] : 0.f;
    const float skip = (live && a.Dskip) ? a.Dskip[d] : 0.f;
    if (TMA && lane == 0) {
        mbar_init(&bar[0], 1);
        mbar_init(&bar[1], 1);
        fence_mbar_init();
    }
    __syncwarp();

    const uint32_t bc_bytes = (uint32_t)N * TT * sizeof(T);
    auto stage = [&](int buf) { return smem + buf * S::BUF; };
    auto issue_loads = [&](int tile, int buf) {
        const int t0 = t_begin + tile * TT;
        unsigned char *st = stage(buf);
        const uint32_t bytes = (MODE == 0 ? (HAS_Z ? 3u : 2u) : 2u) * S::SEQ + (MODE == 0 ? 2u : 1u) * bc_bytes;
        mbar_arrive_expect_tx(&bar[buf], bytes);
#pragma unroll
        for (int j = 0; j < NB8; ++j) {
            tma_load_3d(st + S::off_u + j * S::BLK, &maps.u, &bar[buf], t0 + 8 * j, d0, b);
            tma_load_3d(st + S::off_d + j * S::BLK, &maps.d, &bar[buf], t0 + 8 * j, d0, b);
            if (MODE == 0 && HAS_Z) tma_load_3d(st + S::off_z + j * S::BLK, &maps.z, &bar[buf], t0 + 8 * j, d0, b);
        }
        tma_load_3d(st + S::off_B, &maps.B, &bar[buf], t0, 0, b);
        if (MODE == 0) tma_load_3d(st + S::off_C, &maps.C, &bar[buf], t0, 0, b);
    };
    // Plain loads for shapes TMA cannot describe (row pitch not a multiple of 16 B).
    auto generic_loads = [&](int tile, int buf) {
        const int t0 = t_begin + tile * TT;
        unsigned char *st = stage(buf);
        T *us = reinterpret_cast<T *>(st + S::off_u), *ds = reinterpret_cast<T *>(st + S::off_d);
        T *zs = reinterpret_cast<T *>(st + S::off_z);
        const T *gu = static_cast<const T *>(a.u), *gdl = static_cast<const T *>(a.delta);
        const T *gz = static_cast<const T *>(a.z);
        for (int i = lane; i < kCH * TT; i += kCH) {
            const int tt = i / kCH, cc = i % kCH, dch = d0 + cc, t = t0 + tt;
            const bool in = dch < D && t < L;
            const size_t off = ((size_t)b * D + dch) * L + t;
            const int si = (tt / 8) * (kCH * 8) + cc * 8 + (tt % 8);
            us[si] = in ? gu[off] : T(0.f);
            ds[si] = in ? gdl[off] : T(0.f);
            if (MODE == 0 && HAS_Z) zs[si] = in ? gz[off] : T(0.f);
        }
        T *Bs = reinterpret_cast<T *>(st + S::off_B), *Cs = reinterpret_cast<T *>(st + S::off_C);
        const T *gB = static_cast<const T *>(a.B), *gC = static_cast<const T *>(a.C);
        for (int i = lane; i < N * TT; i += kCH) {
            const int n = i / TT, tt = i % TT, t = t0 + tt;
            const bool in = t < L;
            const size_t off = ((size_t)b * N + n) * L + t;
            Bs[i] = in ? gB[off] : T(0.f);
            if (MODE == 0) Cs[i] = in ? gC[off] : T(0.f);
        }
    };

    if (TMA && lane == 0 && ntiles > 0) issue_loads(0, 0);

    float dsum = 0.f;  // Σ Δ over the chunk (MODE 1)

    for (int tile = 0; tile < ntiles; ++tile) {
        const int buf = tile & 1;
        const int t0 = t_begin + tile * TT;
        unsigned char *st = stage(buf);
        if (TMA) {
            const bool ok = mbar_wait_bounded(&bar[buf], (tile >> 1) & 1, kWaitLimit);
            if (__any_sync(0xffffffffu, !ok)) {
                record_error(a.status, 4 /* SSM_ERR_TIMEOUT */);
                if (lane == 0) bulk_wait0();
                return;
            }
            if (lane == 0 && tile + 1 < ntiles) {
                fence_proxy_async_smem();
                issue_loads(tile + 1, buf ^ 1);
            }
        } else {
            generic_loads(tile, buf);
            __syncwarp();
        }

        // ---- B (and C) widened to fp32, token-major rows, in 4 × 4 blocks
        {
            constexpr int NB = SPT / 4, TB = TT / 4;
            constexpr int UNITS = (MODE == 0 ? 2 : 1) * NB * TB;
            const T *Bs = reinterpret_cast<const T *>(st + S::off_B);
            const T *Cs = reinterpret_cast<const T *>(st + S::off_C);
            for (int it = lane; it < UNITS; it += kCH) {
                const int mat = it / (NB * TB), r = it % (NB * TB);
                const int nb = r / TB, tb = r % TB;
                const T *src = mat ? Cs : Bs;
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
        // The y tile written two tiles ago must have left shared memory.
        if (TMA && MODE == 0 && lane == 0) bulk_wait_read1();
        __syncwarp();

        T *out = reinterpret_cast<T *>(smem + S::off_out + buf * S::OUT);
        const T *u_t = reinterpret_cast<const T *>(st + S::off_u);
        const T *d_t = reinterpret_cast<const T *>(st + S::off_d);
        const T *z_t = reinterpret_cast<const T *>(st + S::off_z);
#pragma unroll 1
        for (int blk = 0; blk < NB8; ++blk) {
            // ---- per-token terms of this lane's 8 tokens, two tokens per packed op
            const int eo = blk * (kCH * 8) + lane * 8;
            float uf[8], df[8], zf[8];
            IO<T>::load8(u_t + eo, uf);
            IO<T>::load8(d_t + eo, df);
            if (MODE == 0 && HAS_Z) IO<T>::load8(z_t + eo, zf);
            const int valid = t_end - (t0 + 8 * blk);  // tokens of this block inside the chunk
            float2 dl[4], du[4], gt[4], dug[4];
#pragma unroll
            for (int j = 0; j < 4; ++j) {
                float2 x = __fadd2_rn(make_float2(df[2 * j], df[2 * j + 1]), make_float2(bias, bias));
                if (a.delta_softplus) x = make_float2(IO<T>::softplus(x.x), IO<T>::softplus(x.y));
                if (valid < 8) {  // Δ = 0 keeps the state: Ā = 1, B̄u = 0
                    if (2 * j >= valid) x.x = 0.f;
                    if (2 * j + 1 >= valid) x.y = 0.f;
                }
                const float2 uu = make_float2(uf[2 * j], uf[2 * j + 1]);
                dl[j] = x;
                du[j] = __fmul2_rn(x, uu);
                if (MODE == 0) {
                    gt[j] = HAS_Z ? gate2<T>(make_float2(zf[2 * j], zf[2 * j + 1])) : make_float2(1.f, 1.f);
                    dug[j] = __fmul2_rn(__fmul2_rn(make_float2(skip, skip), uu), gt[j]);
                }
            }
            // ---- the recurrence over the block's 8 tokens, all SPT states.  The
            // decays Ā and inputs B̄u of token j+1 are formed before the state of
            // token j is updated, so the exponentials overlap the FMA chain.
            float2 an[NQ], bn[NQ];
            auto decay_input = [&](int j, float2 *ao, float2 *bo) {
                const float dv = (j & 1) ? dl[j >> 1].y : dl[j >> 1].x;
                const float uv = (j & 1) ? du[j >> 1].y : du[j >> 1].x;
                const float2 d2 = make_float2(dv, dv), du2 = make_float2(uv, uv);
                const float *Brow = Bf + (8 * blk + j) * S::BCP;
#pragma unroll
                for (int q4 = 0; q4 < SPT / 4; ++q4) {
                    const float4 bq = *reinterpret_cast<const float4 *>(Brow + 4 * q4);
                    const float2 x0 = __fmul2_rn(d2, A2[2 * q4]);
                    const float2 x1 = __fmul2_rn(d2, A2[2 * q4 + 1]);
                    ao[2 * q4] = make_float2(ex2(x0.x), ex2(x0.y));
                    ao[2 * q4 + 1] = make_float2(ex2(x1.x), ex2(x1.y));
                    bo[2 * q4] = __fmul2_rn(make_float2(bq.x, bq.y), du2);
                    bo[2 * q4 + 1] = __fmul2_rn(make_float2(bq.z, bq.w), du2);
                }
            };
            decay_input(0, an, bn);
            float y[8];
#pragma unroll
            for (int j = 0; j < 8; ++j) {
                float2 ac[NQ], bc[NQ];
#pragma unroll
                for (int q = 0; q < NQ; ++q) {
                    ac[q] = an[q];
                    bc[q] = bn[q];
                }
                if (j < 7) decay_input(j + 1, an, bn);
                const float *Crow = Cf + (8 * blk + j) * S::BCP;
                float2 acc0 = make_float2(0.f, 0.f), acc1 = make_float2(0.f, 0.f);
#pragma unroll
                for (int q4 = 0; q4 < SPT / 4; ++q4) {
                    h[2 * q4] = __ffma2_rn(ac[2 * q4], h[2 * q4], bc[2 * q4]);
                    h[2 * q4 + 1] = __ffma2_rn(ac[2 * q4 + 1], h[2 * q4 + 1], bc[2 * q4 + 1]);
                    if (MODE == 0) {
                        const float4 cq = *reinterpret_cast<const float4 *>(Crow + 4 * q4);
                        if (q4 == 0) {
                            acc0 = __fmul2_rn(make_float2(cq.x, cq.y), h[0]);
                            acc1 = __fmul2_rn(make_float2(cq.z, cq.w), h[1]);
                        } else {
                            acc0 = __ffma2_rn(make_float2(cq.x, cq.y), h[2 * q4], acc0);
                            acc1 = __ffma2_rn(make_float2(cq.z, cq.w), h[2 * q4 + 1], acc1);
                        }
                    }
                }
                if (MODE == 0) {
                    const float2 s2 = __fadd2_rn(acc0, acc1);
                    const float g = (j & 1) ? gt[j >> 1].y : gt[j >> 1].x;
                    const float e = (j & 1) ? dug[j >> 1].y : dug[j >> 1].x;
                    y[j] = fmaf(s2.x + s2.y, g, e);
                } else {
                    dsum += (j & 1) ? dl[j >> 1].y : dl[j >> 1].x;
                }
            }
            if (MODE == 0) Pack8<T>::store(out + eo, y);
        }

        if (MODE == 0) {
            if (TMA) {
                fence_proxy_async_smem();
                __syncwarp();
                if (lane == 0) {
#pragma unroll
                    for (int j = 0; j < NB8; ++j)
                        tma_store_3d(&maps.y, out + j * (kCH * 8), t0 + 8 * j, d0, b);
                    bulk_commit();
                }
            } else {
                __syncwarp();
                T *gy = static_cast<T *>(a.y);
                for (int i = lane; i < kCH * TT; i += kCH) {
                    const int tt = i / kCH, cc = i % kCH, dch = d0 + cc, t = t0 + tt;
                    if (dch < D && t < t_end)
                        gy[((size_t)b * D + dch) * L + t] = out[(tt / 8) * (kCH * 8) + cc * 8 + (tt % 8)];
                }
            }
        }
        __syncwarp();  // this tile's B/C rows and raw stage are free again
    }
    if (TMA && MODE == 0 && lane == 0) bulk_wait0();

    if (MODE == 0) {
        if (k == a.nchunks - 1 && a.hL && live) {
#pragma unroll
            for (int q = 0; q < NQ; ++q) {
                const int n = 2 * q;
                if (n < N) a.hL[((size_t)b * D + d) * N + n] = h[q].x;
                if (n + 1 < N) a.hL[((size_t)b * D + d) * N + n + 1] = h[q].y;
            }
        }
    } else if (live) {
#pragma unroll
        for (int q = 0; q < NQ; ++q) {
#pragma unroll
            for (int j = 0; j < 2; ++j) {
                const int n = 2 * q + j;
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

template <typename T, int SPT, bool HAS_Z, bool TMA, int MODE>
cudaError_t launch_one(const Maps &maps, const ScanArgs &a, dim3 grid, cudaStream_t st) {
    using S = WTile<T, SPT, kTT>;
    auto kern = scan_kernel<T, SPT, kTT, HAS_Z, TMA, MODE>;
    static bool attr_set = false;
    if (!attr_set) {
        cudaError_t e = cudaFuncSetAttribute(kern, cudaFuncAttributeMaxDynamicSharedMemorySize, S::bytes);
        if (e != cudaSuccess) return e;
        attr_set = true;
    }
    kern<<<grid, kCH, S::bytes, st>>>(maps, a);
    return cudaGetLastError();
}

template <typename T, int SPT, bool HAS_Z, bool TMA>
cudaError_t launch_all(const Maps &maps, const ScanArgs &a, cudaStream_t st) {
    const unsigned gx = (unsigned)((a.dim + kCH - 1) / kCH);
    cudaError_t e;
    if (a.nchunks > 1) {
        e = launch_one<T, SPT, false, TMA, 1>(maps, a, dim3(gx, a.batch, a.nchunks - 1), st);
        if (e != cudaSuccess) return e;
        const size_t total = (size_t)a.batch * a.dim * a.dstate;
        carry_kernel<<<(unsigned)((total + 255) / 256), 256, 0, st>>>(a);
        e = cudaGetLastError();
        if (e != cudaSuccess) return e;
    }
    return launch_one<T, SPT, HAS_Z, TMA, 0>(maps, a, dim3(gx, a.batch, a.nchunks), st);
}

template <typename T, int SPT>
cudaError_t dispatch_z_tma(const Maps &maps, const ScanArgs &a, bool tma, cudaStream_t st) {
    const bool z = a.z != nullptr;
    if (tma) return z ? launch_all<T, SPT, true, true>(maps, a, st) : launch_all<T, SPT, false, true>(maps, a, st);
    return z ? launch_all<T, SPT, true, false>(maps, a, st) : launch_all<T, SPT, false, false>(maps, a, st);
}

// States held per lane: N rounded up to 4, 8 or 16.
int spt_for(int64_t dstate) { return dstate <= 4 ? 4 : (dstate <= 8 ? 8 : 16); }

template <typename T>
cudaError_t dispatch_spt(const Maps &maps, const ScanArgs &a, bool tma, cudaStream_t st) {
    switch (spt_for(a.dstate)) {
        case 4: return dispatch_z_tma<T, 4>(maps, a, tma, st);
        case 8: return dispatch_z_tma<T, 8>(maps, a, tma, st);
        default: return dispatch_z_tma<T, 16>(maps, a, tma, st);
    }
}

}  // namespace

int scan_groups(int64_t dstate) { return dstate <= 4 ? 1 : (dstate <= 8 ? 2 : 4); }

int64_t scan_chunk_len(int64_t batch, int64_t dim, int64_t dstate, int64_t seqlen, int64_t requested) {
    (void)dstate;
    if (requested > 0) return std::min<int64_t>(requested, ((seqlen + 63) / 64) * 64);
    // One lane per channel: split the sequence until there is at least one
    // warp per scheduler (148 SMs × 4), since each chunk beyond the first costs
    // an extra aggregate pass.
    const int64_t threads = batch * dim;
    const int64_t want = 148LL * 4 * 32;
    int64_t K = (want + threads - 1) / threads;
    K = std::max<int64_t>(1, std::min<int64_t>(K, (seqlen + 511) / 512));
    const int64_t len = (seqlen + K - 1) / K;
    return ((len + 63) / 64) * 64;
}

cudaError_t scan_launch(const ScanArgs &a, bool bf16, cudaStream_t st) {
    const size_t es = bf16 ? 2 : 4;
    // TMA needs a row pitch that is a multiple of 16 bytes.
    const bool tma = ((size_t)a.seqlen * es) % 16 == 0;
    Maps maps;
    memset(&maps, 0, sizeof(maps));
    if (tma) {
        const CUtensorMapDataType dt = bf16 ? CU_TENSOR_MAP_DATA_TYPE_BFLOAT16 : CU_TENSOR_MAP_DATA_TYPE_FLOAT32;
        bool ok = make_map(&maps.u, dt, es, a.u, a.seqlen, a.dim, a.batch, 8, kCH) &&
                  make_map(&maps.d, dt, es, a.delta, a.seqlen, a.dim, a.batch, 8, kCH) &&
                  make_map(&maps.B, dt, es, a.B, a.seqlen, a.dstate, a.batch, kTT, a.dstate) &&
                  make_map(&maps.C, dt, es, a.C, a.seqlen, a.dstate, a.batch, kTT, a.dstate) &&
                  make_map(&maps.y, dt, es, a.y, a.seqlen, a.dim, a.batch, 8, kCH);
        if (ok && a.z) ok = make_map(&maps.z, dt, es, a.z, a.seqlen, a.dim, a.batch, 8, kCH);
        if (!ok) return cudaErrorInvalidValue;
    }
    return bf16 ? dispatch_spt<__nv_bfloat16>(maps, a, tma, st) : dispatch_spt<float>(maps, a, tma, st);
}

}  // namespace ssm
