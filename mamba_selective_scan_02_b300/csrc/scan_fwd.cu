// scan_fwd.cu — the fused Mamba selective scan for sm_103a.
//
// What one launch computes is the recurrence of "Mamba and selective state
// spaces, from first principles" ("Selection", "Discretisation: zero-order
// hold", "The hardware-aware scan"): for every channel (b, d) and state n,
//   Δ = softplus(Δraw + bias), Ā = exp(Δ·A), h = Ā·h + Δ·B·u,
//   y = (C·h + D·u)·silu(z),
// writing only y (b × D × L) and the final state — never Ā, B̄ or any h_t.
//
// Design (B300-first, not the pages' kernel):
//   * Channels are the parallel axis.  A thread owns one channel and a group of
//     four consecutive states and walks the time axis sequentially, keeping its
//     four states in registers; NG = ceil(N/4) adjacent lanes share a channel
//     and reduce C·h across their groups with a transposed warp shuffle.
//   * Per 32-token tile, one elected thread moves u, Δraw, z (CH channels × 32
//     tokens) and B, C (N × 32 tokens, shared by all channels) into shared
//     memory with 3-D TMA copies on an mbarrier, and stores the y tile back
//     with a TMA store.  The next tile's copies overlap the current tile's scan.
//   * Per-token nonlinearities (softplus, Δ·u, silu(z), D·u) run once per
//     (channel, token) in a pre-pass; the state loop touches only fp32 shared
//     tiles.  Ā is computed as ex2(Δ·A·log2e) on the MUFU, and the state
//     arithmetic uses packed f32x2 FMA.
//   * Long sequences are cut into chunks that run concurrently.  The
//     composition of affine steps is associative (first-principles page,
//     "The hardware-aware scan"): an aggregate pass computes each chunk's pair
//     (Π Ā, h_end from zero), a carry pass chains the pairs from h0, and the
//     main pass rescans every chunk from its carried state.
#include <algorithm>
#include <cstring>

#include "ssm_device.cuh"
#include "ssm_internal.h"

namespace ssm {

constexpr int TT = 32;                 // tokens per tile
constexpr int kWaitLimit = 1 << 22;    // mbarrier polls before giving up

template <int NG> struct Shape {
    static_assert(NG == 1 || NG == 2 || NG == 4, "state groups per channel");
    static constexpr int kThreads = 128;
    static constexpr int kCH = kThreads / NG;   // channels per CTA
    static constexpr int kNP = 4 * NG;          // padded state count
};

// Shared-memory layout of one CTA (byte offsets; TMA destinations 128-B aligned).
template <typename T, int NG> struct Smem {
    static constexpr int CH = Shape<NG>::kCH, NP = Shape<NG>::kNP;
    static constexpr int kRow2 = TT + 2;                      // padded float2 row
    static constexpr int raw_seq = CH * TT * (int)sizeof(T);  // one u/Δ/z tile
    static constexpr int raw_bc = NP * TT * (int)sizeof(T);   // one B/C tile (N ≤ NP rows used)
    static constexpr int off_u = 0;
    static constexpr int off_d = off_u + ((raw_seq + 127) / 128) * 128;
    static constexpr int off_z = off_d + ((raw_seq + 127) / 128) * 128;
    static constexpr int off_B = off_z + ((raw_seq + 127) / 128) * 128;
    static constexpr int off_C = off_B + ((raw_bc + 127) / 128) * 128;
    static constexpr int off_out = off_C + ((raw_bc + 127) / 128) * 128;
    static constexpr int off_dt = off_out + ((raw_seq + 127) / 128) * 128;  // float2 (Δ, Δ·u)
    static constexpr int off_gd = off_dt + CH * kRow2 * 8;                   // float2 (gate, D·u)
    static constexpr int off_Bf = off_gd + CH * kRow2 * 8;                   // float [TT][NP]
    static constexpr int off_Cf = off_Bf + TT * NP * 4;
    static constexpr int off_bias = off_Cf + TT * NP * 4;
    static constexpr int off_skip = off_bias + CH * 4;
    static constexpr int off_bar = ((off_skip + CH * 4 + 15) / 16) * 16;
    static constexpr int bytes = off_bar + 16;
};

struct Maps {
    CUtensorMap u, d, z, B, C, y;
};

// MODE 0: full scan writing y (and hL for the last chunk).
// MODE 1: chunk aggregate (Π Ā, h_end from zero) for chunks 0..K-2.
template <typename T, int NG, bool HAS_Z, bool TMA, int MODE>
__global__ void __launch_bounds__(Shape<NG>::kThreads)
scan_kernel(const __grid_constant__ Maps maps, const ScanArgs a) {
    using S = Smem<T, NG>;
    constexpr int CH = S::CH, NP = S::NP, NT = Shape<NG>::kThreads;
    extern __shared__ __align__(128) unsigned char smem[];
    T *u_s = reinterpret_cast<T *>(smem + S::off_u);
    T *d_s = reinterpret_cast<T *>(smem + S::off_d);
    T *z_s = reinterpret_cast<T *>(smem + S::off_z);
    T *B_s = reinterpret_cast<T *>(smem + S::off_B);
    T *C_s = reinterpret_cast<T *>(smem + S::off_C);
    T *out_s = reinterpret_cast<T *>(smem + S::off_out);
    float2 *dt2 = reinterpret_cast<float2 *>(smem + S::off_dt);
    float2 *gd2 = reinterpret_cast<float2 *>(smem + S::off_gd);
    float *Bf = reinterpret_cast<float *>(smem + S::off_Bf);
    float *Cf = reinterpret_cast<float *>(smem + S::off_Cf);
    float *bias_s = reinterpret_cast<float *>(smem + S::off_bias);
    float *skip_s = reinterpret_cast<float *>(smem + S::off_skip);
    uint64_t *bar = reinterpret_cast<uint64_t *>(smem + S::off_bar);

    const int tid = threadIdx.x;
    const int c = tid / NG;          // channel within the CTA
    const int g = tid % NG;          // state group: states 4g .. 4g+3
    const int d0 = blockIdx.x * CH;
    const int b = blockIdx.y;
    const int k = blockIdx.z;        // chunk
    const int D = a.dim, N = a.dstate, L = a.seqlen;
    const int d = d0 + c;
    const bool live = d < D;
    const int t_begin = k * a.chunk_len;
    const int t_end = min(L, t_begin + a.chunk_len);
    const int ntiles = (t_end - t_begin + TT - 1) / TT;

    // ---- per-thread constants: A·log2e for the four states, initial state
    float2 A2[2] = {make_float2(0.f, 0.f), make_float2(0.f, 0.f)};
    float2 h[2] = {make_float2(0.f, 0.f), make_float2(0.f, 0.f)};
    {
        float av[4], hv[4];
#pragma unroll
        for (int j = 0; j < 4; ++j) {
            const int n = 4 * g + j;
            av[j] = 0.f;
            hv[j] = 0.f;
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
        A2[0] = make_float2(av[0], av[1]);
        A2[1] = make_float2(av[2], av[3]);
        h[0] = make_float2(hv[0], hv[1]);
        h[1] = make_float2(hv[2], hv[3]);
    }
    for (int i = tid; i < CH; i += NT) {
        const int dd = d0 + i;
        bias_s[i] = (dd < D && a.bias) ? a.bias[dd] : 0.f;
        skip_s[i] = (dd < D && a.Dskip) ? a.Dskip[dd] : 0.f;
    }
    // Padded state rows of the fp32 B/C tiles stay zero for the whole launch.
    for (int i = tid; i < TT * NP; i += NT) {
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
        const T *gu = static_cast<const T *>(a.u), *gd = static_cast<const T *>(a.delta);
        const T *gz = static_cast<const T *>(a.z);
        for (int i = tid; i < CH * TT; i += NT) {
            const int cc = i / TT, tt = i % TT, dd = d0 + cc, t = t0 + tt;
            const bool in = dd < D && t < L;
            const size_t off = ((size_t)b * D + dd) * L + t;
            u_s[i] = in ? gu[off] : T(0.f);
            d_s[i] = in ? gd[off] : T(0.f);
            if (MODE == 0 && HAS_Z) z_s[i] = in ? gz[off] : T(0.f);
        }
        const T *gB = static_cast<const T *>(a.B), *gC = static_cast<const T *>(a.C);
        for (int i = tid; i < N * TT; i += NT) {
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

        // ---- pre-pass: once per (channel, token)
        for (int i = tid; i < CH * TT; i += NT) {
            const int cc = i / TT, tt = i % TT;
            const bool valid = (t0 + tt) < t_end && (d0 + cc) < D;
            const float uv = IO<T>::to_f(u_s[i]);
            float dv = IO<T>::to_f(d_s[i]) + bias_s[cc];
            if (a.delta_softplus) dv = softplus(dv);
            if (!valid) dv = 0.f;  // Δ = 0 keeps the state: Ā = 1, B̄u = 0
            dt2[cc * S::kRow2 + tt] = make_float2(dv, dv * uv);
            if (MODE == 0) {
                const float gate = HAS_Z ? gate_of<T>(IO<T>::to_f(z_s[i])) : 1.f;
                gd2[cc * S::kRow2 + tt] = make_float2(gate, skip_s[cc] * uv);
            }
        }
        for (int i = tid; i < N * TT; i += NT) {
            const int n = i / TT, tt = i % TT;
            Bf[tt * NP + n] = IO<T>::to_f(B_s[i]);
            if (MODE == 0) Cf[tt * NP + n] = IO<T>::to_f(C_s[i]);
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

        // ---- the scan over this tile, NG tokens per reduction block
        const float2 *dtrow = dt2 + c * S::kRow2;
#pragma unroll 2
        for (int tb = 0; tb < TT; tb += NG) {
            float part[NG];
#pragma unroll
            for (int j = 0; j < NG; ++j) {
                const int tt = tb + j;
                const float2 dd = dtrow[tt];
                const float4 bv = *reinterpret_cast<const float4 *>(Bf + tt * NP + 4 * g);
                const float2 dd2 = make_float2(dd.x, dd.x);
                const float2 x01 = __fmul2_rn(dd2, A2[0]);
                const float2 x23 = __fmul2_rn(dd2, A2[1]);
                const float2 a01 = make_float2(ex2(x01.x), ex2(x01.y));
                const float2 a23 = make_float2(ex2(x23.x), ex2(x23.y));
                const float2 du2 = make_float2(dd.y, dd.y);
                const float2 bu01 = __fmul2_rn(make_float2(bv.x, bv.y), du2);
                const float2 bu23 = __fmul2_rn(make_float2(bv.z, bv.w), du2);
                h[0] = __ffma2_rn(a01, h[0], bu01);
                h[1] = __ffma2_rn(a23, h[1], bu23);
                if (MODE == 0) {
                    const float4 cv = *reinterpret_cast<const float4 *>(Cf + tt * NP + 4 * g);
                    float2 acc = __fmul2_rn(make_float2(cv.x, cv.y), h[0]);
                    acc = __ffma2_rn(make_float2(cv.z, cv.w), h[1], acc);
                    part[j] = acc.x + acc.y;
                } else {
                    dsum += dd.x;
                }
            }
            if (MODE == 0) {
                // Transposed reduction: afterwards lane g holds the full C·h of token tb+g.
                float s;
                if (NG == 1) {
                    s = part[0];
                } else if (NG == 2) {
                    const float send = g ? part[0] : part[1];
                    const float keep = g ? part[1] : part[0];
                    s = keep + __shfl_xor_sync(0xffffffffu, send, 1);
                } else {
                    const bool hi = g & 2;
                    const float s0 = hi ? part[0] : part[2], s1 = hi ? part[1] : part[3];
                    float k0 = hi ? part[2] : part[0], k1 = hi ? part[3] : part[1];
                    k0 += __shfl_xor_sync(0xffffffffu, s0, 2);
                    k1 += __shfl_xor_sync(0xffffffffu, s1, 2);
                    const bool odd = g & 1;
                    const float s2 = odd ? k0 : k1;
                    s = (odd ? k1 : k0) + __shfl_xor_sync(0xffffffffu, s2, 1);
                }
                const int tt = tb + g;
                const float2 gd = gd2[c * S::kRow2 + tt];
                out_s[c * TT + tt] = IO<T>::from_f((s + gd.y) * gd.x);
            }
        }

        if (MODE == 0) {
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
                for (int i = tid; i < CH * TT; i += NT) {
                    const int cc = i / TT, tt = i % TT, dd = d0 + cc, t = t0 + tt;
                    if (dd < D && t < t_end) gy[((size_t)b * D + dd) * L + t] = out_s[i];
                }
            }
        }
        if (MODE == 1) __syncthreads();  // pre-pass tiles are rewritten by the next tile
    }
    if (TMA && MODE == 0 && tid == 0) bulk_wait0();

    const float hv[4] = {h[0].x, h[0].y, h[1].x, h[1].y};
    if (MODE == 0) {
        if (k == a.nchunks - 1 && a.hL && live) {
#pragma unroll
            for (int j = 0; j < 4; ++j)
                if (4 * g + j < N) a.hL[((size_t)b * D + d) * N + 4 * g + j] = hv[j];
        }
    } else if (live) {
        const float av[4] = {A2[0].x, A2[0].y, A2[1].x, A2[1].y};
#pragma unroll
        for (int j = 0; j < 4; ++j) {
            const int n = 4 * g + j;
            if (n < N)
                a.agg[(((size_t)b * D + d) * (a.nchunks - 1) + k) * N + n] =
                    make_float2(ex2(av[j] * dsum), hv[j]);
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

template <typename T, int NG, bool HAS_Z, bool TMA, int MODE>
cudaError_t launch_one(const Maps &maps, const ScanArgs &a, dim3 grid, cudaStream_t st) {
    using S = Smem<T, NG>;
    auto kern = scan_kernel<T, NG, HAS_Z, TMA, MODE>;
    static bool attr_set = false;
    if (!attr_set) {
        cudaError_t e = cudaFuncSetAttribute(kern, cudaFuncAttributeMaxDynamicSharedMemorySize, S::bytes);
        if (e != cudaSuccess) return e;
        attr_set = true;
    }
    kern<<<grid, Shape<NG>::kThreads, S::bytes, st>>>(maps, a);
    return cudaGetLastError();
}

template <typename T, int NG, bool HAS_Z, bool TMA>
cudaError_t launch_all(const Maps &maps, const ScanArgs &a, cudaStream_t st) {
    const int CH = Shape<NG>::kCH;
    const unsigned gx = (unsigned)((a.dim + CH - 1) / CH);
    cudaError_t e;
    if (a.nchunks > 1) {
        e = launch_one<T, NG, false, TMA, 1>(maps, a, dim3(gx, a.batch, a.nchunks - 1), st);
        if (e != cudaSuccess) return e;
        const size_t total = (size_t)a.batch * a.dim * a.dstate;
        carry_kernel<<<(unsigned)((total + 255) / 256), 256, 0, st>>>(a);
        e = cudaGetLastError();
        if (e != cudaSuccess) return e;
    }
    return launch_one<T, NG, HAS_Z, TMA, 0>(maps, a, dim3(gx, a.batch, a.nchunks), st);
}

template <typename T, int NG>
cudaError_t dispatch_z_tma(const Maps &maps, const ScanArgs &a, bool tma, cudaStream_t st) {
    const bool z = a.z != nullptr;
    if (tma) return z ? launch_all<T, NG, true, true>(maps, a, st) : launch_all<T, NG, false, true>(maps, a, st);
    return z ? launch_all<T, NG, true, false>(maps, a, st) : launch_all<T, NG, false, false>(maps, a, st);
}

template <typename T>
cudaError_t dispatch_ng(const Maps &maps, const ScanArgs &a, int ng, bool tma, cudaStream_t st) {
    switch (ng) {
        case 1: return dispatch_z_tma<T, 1>(maps, a, tma, st);
        case 2: return dispatch_z_tma<T, 2>(maps, a, tma, st);
        default: return dispatch_z_tma<T, 4>(maps, a, tma, st);
    }
}

int channels_per_cta(int ng) {
    switch (ng) {
        case 1: return Shape<1>::kCH;
        case 2: return Shape<2>::kCH;
        default: return Shape<4>::kCH;
    }
}

}  // namespace

int scan_groups(int64_t dstate) { return dstate <= 4 ? 1 : (dstate <= 8 ? 2 : 4); }

int64_t scan_chunk_len(int64_t batch, int64_t dim, int64_t dstate, int64_t seqlen, int64_t requested) {
    if (requested > 0) return std::min<int64_t>(requested, ((seqlen + 63) / 64) * 64);
    // Enough resident threads to keep every SM's MUFU and FMA pipes busy.
    const int64_t threads = batch * dim * scan_groups(dstate);
    const int64_t want = 148LL * 512;
    int64_t K = (want + threads - 1) / threads;
    K = std::max<int64_t>(1, std::min<int64_t>(K, (seqlen + 511) / 512));
    const int64_t len = (seqlen + K - 1) / K;
    return ((len + 63) / 64) * 64;
}

cudaError_t scan_launch(const ScanArgs &a, bool bf16, cudaStream_t st) {
    const int ng = scan_groups(a.dstate);
    const int CH = channels_per_cta(ng);
    const size_t es = bf16 ? 2 : 4;
    // TMA needs a row pitch that is a multiple of 16 bytes.
    const bool tma = ((size_t)a.seqlen * es) % 16 == 0;
    Maps maps;
    memset(&maps, 0, sizeof(maps));
    if (tma) {
        const CUtensorMapDataType dt = bf16 ? CU_TENSOR_MAP_DATA_TYPE_BFLOAT16 : CU_TENSOR_MAP_DATA_TYPE_FLOAT32;
        bool ok = make_map(&maps.u, dt, es, a.u, a.seqlen, a.dim, a.batch, TT, CH) &&
                  make_map(&maps.d, dt, es, a.delta, a.seqlen, a.dim, a.batch, TT, CH) &&
                  make_map(&maps.B, dt, es, a.B, a.seqlen, a.dstate, a.batch, TT, a.dstate) &&
                  make_map(&maps.C, dt, es, a.C, a.seqlen, a.dstate, a.batch, TT, a.dstate) &&
                  make_map(&maps.y, dt, es, a.y, a.seqlen, a.dim, a.batch, TT, CH);
        if (ok && a.z) ok = make_map(&maps.z, dt, es, a.z, a.seqlen, a.dim, a.batch, TT, CH);
        if (!ok) return cudaErrorInvalidValue;
    }
    return bf16 ? dispatch_ng<__nv_bfloat16>(maps, a, ng, tma, st) : dispatch_ng<float>(maps, a, ng, tma, st);
}

}  // namespace ssm
