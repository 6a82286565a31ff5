// ssd.cu — the Mamba-2 layer scan (state space duality) for sm_103a.
//
// "Mamba and selective state spaces, from first principles", section
// "Mamba-2: state space duality": A_t is a scalar times the identity per head,
// a_t = exp(Δ_t A_h); the P channels of a head share a_t, B_t and C_t, and the
// head's state is an N × P matrix,
//   S_t = a_t S_{t−1} + Δ_t B_t x_tᵀ,   y_t = S_tᵀ C_t + D_h x_t.
// The SSD algorithm on that page cuts the sequence into chunks of Q tokens; a
// chunk's output is a masked matrix product inside the chunk plus the state it
// inherits read through the decay, and its final state is one more product.
//
// Per chunk of Q = 64 tokens (cum_i = Σ_{k<=i} Δ_k A_h within the chunk):
//   Y   = diag(e^{cum}) · C · S_inᵀ                  (the inherited state)
//       + (C Bᵀ ∘ Λ) · X,  Λ_ij = e^{cum_i − cum_j}·Δ_j for j <= i, else 0
//       + D_h · X
//   S_out = e^{cum_{Q−1}} · S_in + Xᵀ · diag(e^{cum_{Q−1} − cum_j}·Δ_j) · B
// All four products run on the tensor cores (mma.sync m16n8k16, bf16 operands,
// fp32 accumulators); the state stays in fp32 registers across chunks.  The
// operands that are not inputs — the inherited state, the decay-masked C·Bᵀ
// block and the weighted B — enter as a pair of bf16 values (the rounded value
// and the rounded remainder) and are multiplied twice, so they carry ~16 bits
// instead of bf16's 8 whatever the input range.  The weighted B's remainder
// lives in the C tile, free by then.
//
// One CTA of four warps owns one (sequence, head) and walks its chunks in
// order; warp w owns rows 16w .. 16w+15 of the chunk's outputs and of the state.
// Shared tiles are unpadded, with the 16-byte chunks of row r stored at chunk
// position c ^ (r & 7), so the eight rows an ldmatrix reads hit eight
// different bank groups; three CTAs fit on an SM.
// Shapes built: P = 64, N = 128, bf16 I/O.
#include <algorithm>

#include "ssm_device.cuh"
#include "ssm_internal.h"

namespace ssm {
namespace {

constexpr int Q = 64;                  // tokens per chunk
constexpr int P = 64;                  // head dimension
constexpr int NS = 128;                // state size
constexpr int XS = P;                  // row (bf16 elements) of the x tile
constexpr int BS = NS;                 // row of the B, C and state tiles
constexpr int kThreads = 128;

// Element (row, col) of a swizzled tile with `stride` elements per row.
__device__ __forceinline__ int swz(int row, int col, int stride) {
    return row * stride + ((((col >> 3) ^ (row & 7))) << 3) + (col & 7);
}

struct __align__(16) SsdSmem {
    __nv_bfloat16 x[Q * XS];           // x chunk, [token][p]
    __nv_bfloat16 B[Q * BS];           // B chunk, [token][n] (scaled by w_j for the state product)
    __nv_bfloat16 C[Q * BS];           // C chunk, [token][n]; then the weighted B's remainder
    __nv_bfloat16 S[P * BS];           // inherited state, [p][n]: bf16 value ...
    __nv_bfloat16 Sl[P * BS];          // ... and bf16 remainder
    float cum[Q], delta[Q], wsc[Q];    // prefix sums of Δ·A, Δ, and the state weights w_j
};

__device__ __forceinline__ uint32_t pack_bf16(float lo, float hi) {
    const __nv_bfloat162 v = __floats2bfloat162_rn(lo, hi);
    return *reinterpret_cast<const uint32_t *>(&v);
}
// (v0, v1) as two bf16 pairs: the rounded values and the rounded remainders.
__device__ __forceinline__ void split_bf16(float v0, float v1, uint32_t &hi, uint32_t &lo) {
    const __nv_bfloat162 h = __floats2bfloat162_rn(v0, v1);
    const float2 hf = __bfloat1622float2(h);
    hi = *reinterpret_cast<const uint32_t *>(&h);
    lo = pack_bf16(v0 - hf.x, v1 - hf.y);
}

__device__ __forceinline__ void ldsm_x4(uint32_t *r, const void *p) {
    asm volatile("ldmatrix.sync.aligned.m8n8.x4.shared.b16 {%0, %1, %2, %3}, [%4];"
                 : "=r"(r[0]), "=r"(r[1]), "=r"(r[2]), "=r"(r[3])
                 : "r"(smem_u32(p)));
}
__device__ __forceinline__ void ldsm_x4_t(uint32_t *r, const void *p) {
    asm volatile("ldmatrix.sync.aligned.m8n8.x4.trans.shared.b16 {%0, %1, %2, %3}, [%4];"
                 : "=r"(r[0]), "=r"(r[1]), "=r"(r[2]), "=r"(r[3])
                 : "r"(smem_u32(p)));
}
// d += a · b, m16n8k16, bf16 operands, fp32 accumulators
__device__ __forceinline__ void mma16816(float *d, const uint32_t *a, uint32_t b0, uint32_t b1) {
    asm volatile(
        "mma.sync.aligned.m16n8k16.row.col.f32.bf16.bf16.f32 {%0, %1, %2, %3}, {%4, %5, %6, %7}, {%8, %9}, "
        "{%0, %1, %2, %3};"
        : "+f"(d[0]), "+f"(d[1]), "+f"(d[2]), "+f"(d[3])
        : "r"(a[0]), "r"(a[1]), "r"(a[2]), "r"(a[3]), "r"(b0), "r"(b1));
}

// A fragment (16 × 16) of a row-major tile: rows r0.., columns k0.. (stride in elements).
__device__ __forceinline__ void frag_a(uint32_t *a, const __nv_bfloat16 *base, int stride, int r0, int k0, int lane) {
    const int m = lane >> 3, r = lane & 7;
    ldsm_x4(a, base + swz(r0 + r + 8 * (m & 1), k0 + 8 * (m >> 1), stride));
}
// A fragment of the transpose of a row-major tile: A[m][k] = tile[k][m].
__device__ __forceinline__ void frag_a_t(uint32_t *a, const __nv_bfloat16 *base, int stride, int m0, int k0, int lane) {
    const int mi = lane >> 3, r = lane & 7;
    ldsm_x4_t(a, base + swz(k0 + r + 8 * (mi >> 1), m0 + 8 * (mi & 1), stride));
}
// B fragments of two adjacent n-tiles (n0, n0 + 8) for one k-step, from a tile
// stored [n][k] (k contiguous): b[0..1] for n-tile n0, b[2..3] for n0 + 8.
__device__ __forceinline__ void frag_b_nk(uint32_t *b, const __nv_bfloat16 *base, int stride, int n0, int k0, int lane) {
    const int m = lane >> 3, r = lane & 7;
    ldsm_x4(b, base + swz(n0 + r + 8 * (m >> 1), k0 + 8 * (m & 1), stride));
}
// The same from a tile stored [k][n] (n contiguous).
__device__ __forceinline__ void frag_b_kn(uint32_t *b, const __nv_bfloat16 *base, int stride, int n0, int k0, int lane) {
    const int m = lane >> 3, r = lane & 7;
    ldsm_x4_t(b, base + swz(k0 + r + 8 * (m & 1), n0 + 8 * (m >> 1), stride));
}

__global__ void __launch_bounds__(kThreads, 3)
ssd_kernel(const SsdArgs a) {
    extern __shared__ __align__(16) unsigned char smem_raw[];
    SsdSmem &sm = *reinterpret_cast<SsdSmem *>(smem_raw);
    const int tid = threadIdx.x, lane = tid & 31, w = tid >> 5;
    const int gid = lane >> 2, tig = lane & 3;
    const int bh = blockIdx.x, b = bh / a.nheads, h = bh % a.nheads;
    const int L = a.seqlen, H = a.nheads;
    const __nv_bfloat16 *xg = static_cast<const __nv_bfloat16 *>(a.x);
    const __nv_bfloat16 *dtg = static_cast<const __nv_bfloat16 *>(a.dt);
    const __nv_bfloat16 *Bg = static_cast<const __nv_bfloat16 *>(a.B);
    const __nv_bfloat16 *Cg = static_cast<const __nv_bfloat16 *>(a.C);
    __nv_bfloat16 *yg = static_cast<__nv_bfloat16 *>(a.y);
    const float Ah = a.A[h];
    const float Dh = a.Dskip ? a.Dskip[h] : 0.f;
    const float bias = a.dt_bias ? a.dt_bias[h] : 0.f;

    // the state S[p][n] in fp32: warp w owns columns n = 32w .. 32w+31 for all
    // P rows; Sacc[mt][nt][0..3] holds (p = 16mt+gid, n = 32w+8nt+2tig, +1)
    // and (p + 8, same n)
    float Sacc[P / 16][4][4];
#pragma unroll
    for (int mt = 0; mt < P / 16; ++mt) {
#pragma unroll
        for (int nt = 0; nt < 4; ++nt) {
#pragma unroll
            for (int e = 0; e < 4; ++e) {
                const int p = 16 * mt + gid + 8 * (e >> 1), n = 32 * w + 8 * nt + 2 * tig + (e & 1);
                Sacc[mt][nt][e] = a.h0 ? a.h0[(((size_t)b * H + h) * P + p) * NS + n] : 0.f;
            }
        }
    }

    // the inherited state as its bf16 operand pair, [p][n] in S (value) and Sl
    auto store_state = [&]() {
#pragma unroll
        for (int mt = 0; mt < P / 16; ++mt) {
#pragma unroll
            for (int nt = 0; nt < 4; ++nt) {
                const int p = 16 * mt + gid, n = 32 * w + 8 * nt + 2 * tig;
                uint32_t hi, lo;
                split_bf16(Sacc[mt][nt][0], Sacc[mt][nt][1], hi, lo);
                *reinterpret_cast<uint32_t *>(sm.S + swz(p, n, BS)) = hi;
                *reinterpret_cast<uint32_t *>(sm.Sl + swz(p, n, BS)) = lo;
                split_bf16(Sacc[mt][nt][2], Sacc[mt][nt][3], hi, lo);
                *reinterpret_cast<uint32_t *>(sm.S + swz(p + 8, n, BS)) = hi;
                *reinterpret_cast<uint32_t *>(sm.Sl + swz(p + 8, n, BS)) = lo;
            }
        }
    };
    store_state();
    __syncthreads();

    // the decay-masked block Λ ∘ C·Bᵀ lives, as a bf16 value / remainder pair
    // [i][j], in the state buffers while they are free (after the read-out of
    // the inherited state, before the new state is stored)
    __nv_bfloat16 *Mh = sm.S, *Ml = sm.Sl;
    constexpr int MS = Q;                           // row of the masked block

    const int nchunks = (L + Q - 1) / Q;
    for (int ck = 0; ck < nchunks; ++ck) {
        const int t0 = ck * Q;
        // ---- stage the chunk: x, B, C rows as 16-byte words; Δ and its prefix sum
#pragma unroll
        for (int i = tid; i < Q * (P / 8); i += kThreads) {
            const int r = i / (P / 8), q = i % (P / 8), t = t0 + r;
            uint4 v = make_uint4(0u, 0u, 0u, 0u);
            if (t < L) v = __ldg(reinterpret_cast<const uint4 *>(xg + (((size_t)b * L + t) * H + h) * P) + q);
            *reinterpret_cast<uint4 *>(sm.x + swz(r, 8 * q, XS)) = v;
        }
#pragma unroll
        for (int i = tid; i < Q * (NS / 8); i += kThreads) {
            const int r = i / (NS / 8), q = i % (NS / 8), t = t0 + r;
            uint4 vb = make_uint4(0u, 0u, 0u, 0u), vc = vb;
            if (t < L) {
                vb = __ldg(reinterpret_cast<const uint4 *>(Bg + ((size_t)b * L + t) * NS) + q);
                vc = __ldg(reinterpret_cast<const uint4 *>(Cg + ((size_t)b * L + t) * NS) + q);
            }
            *reinterpret_cast<uint4 *>(sm.B + swz(r, 8 * q, BS)) = vb;
            *reinterpret_cast<uint4 *>(sm.C + swz(r, 8 * q, BS)) = vc;
        }
        if (w < 2) {
            const int i = tid, t = t0 + i;
            float d = 0.f;
            if (t < L) {
                const float x = __bfloat162float(dtg[((size_t)b * L + t) * H + h]) + bias;
                d = a.dt_softplus ? softplus_poly(x) : x;
            }
            sm.delta[i] = d;
            // inclusive prefix sum of Δ·A over the chunk: a scan in each of the
            // two warps, then warp 1 adds warp 0's total
            float v = d * Ah;
#pragma unroll
            for (int o = 1; o < 32; o <<= 1) {
                const float u = __shfl_up_sync(0xffffffffu, v, o);
                if (lane >= o) v += u;
            }
            sm.cum[i] = v;
        }
        __syncthreads();
        if (w == 1) sm.cum[tid] += sm.cum[31];
        __syncthreads();
        if (tid < Q) sm.wsc[tid] = ex2((sm.cum[Q - 1] - sm.cum[tid]) * kLog2e) * sm.delta[tid];

        // ---- Y = diag(e^cum) · C · S_inᵀ: all 64 rows, columns p = 16w .. 16w+15
        float Y[Q / 16][2][4];
#pragma unroll
        for (int mt = 0; mt < Q / 16; ++mt)
#pragma unroll
            for (int nt = 0; nt < 2; ++nt) Y[mt][nt][0] = Y[mt][nt][1] = Y[mt][nt][2] = Y[mt][nt][3] = 0.f;
#pragma unroll
        for (int ks = 0; ks < NS / 16; ++ks) {
            uint32_t bf[4], bl[4];
            frag_b_nk(bf, sm.S, BS, 16 * w, 16 * ks, lane);
            frag_b_nk(bl, sm.Sl, BS, 16 * w, 16 * ks, lane);
#pragma unroll
            for (int mt = 0; mt < Q / 16; ++mt) {
                uint32_t af[4];
                frag_a(af, sm.C, BS, 16 * mt, 16 * ks, lane);
                mma16816(Y[mt][0], af, bf[0], bf[1]);
                mma16816(Y[mt][1], af, bf[2], bf[3]);
                mma16816(Y[mt][0], af, bl[0], bl[1]);
                mma16816(Y[mt][1], af, bl[2], bl[3]);
            }
        }
#pragma unroll
        for (int mt = 0; mt < Q / 16; ++mt) {
            const float e0 = ex2(sm.cum[16 * mt + gid] * kLog2e), e1 = ex2(sm.cum[16 * mt + gid + 8] * kLog2e);
#pragma unroll
            for (int nt = 0; nt < 2; ++nt) {
                Y[mt][nt][0] *= e0;
                Y[mt][nt][1] *= e0;
                Y[mt][nt][2] *= e1;
                Y[mt][nt][3] *= e1;
            }
        }

        // ---- G = C · Bᵀ for rows 16w .. 16w+15 on the causal part (columns
        // j <= 16w + 15), masked by Λ into the shared value / remainder pair
        {
            const int r0 = 16 * w;
            const int njt = 2 * (w + 1);
            float G[Q / 8][4];
#pragma unroll
            for (int nt = 0; nt < Q / 8; ++nt) G[nt][0] = G[nt][1] = G[nt][2] = G[nt][3] = 0.f;
#pragma unroll
            for (int ks = 0; ks < NS / 16; ++ks) {
                uint32_t af[4];
                frag_a(af, sm.C, BS, r0, 16 * ks, lane);
#pragma unroll
                for (int np = 0; np < Q / 16; ++np) {
                    if (2 * np < njt) {
                        uint32_t bf[4];
                        frag_b_nk(bf, sm.B, BS, 16 * np, 16 * ks, lane);
                        mma16816(G[2 * np], af, bf[0], bf[1]);
                        mma16816(G[2 * np + 1], af, bf[2], bf[3]);
                    }
                }
            }
            __syncthreads();                         // every warp is done reading S, Sl
            const float cr0 = sm.cum[r0 + gid], cr1 = sm.cum[r0 + gid + 8];
#pragma unroll
            for (int nt = 0; nt < Q / 8; ++nt) {
                if (nt < njt) {
                    const int j0 = 8 * nt + 2 * tig;
                    float v[4];
#pragma unroll
                    for (int e = 0; e < 4; ++e) {
                        const int i = r0 + gid + 8 * (e >> 1), j = j0 + (e & 1);
                        const float ci = (e >> 1) ? cr1 : cr0;
                        v[e] = j <= i ? G[nt][e] * ex2((ci - sm.cum[j]) * kLog2e) * sm.delta[j] : 0.f;
                    }
                    uint32_t hi, lo;
                    split_bf16(v[0], v[1], hi, lo);
                    *reinterpret_cast<uint32_t *>(Mh + swz(r0 + gid, j0, MS)) = hi;
                    *reinterpret_cast<uint32_t *>(Ml + swz(r0 + gid, j0, MS)) = lo;
                    split_bf16(v[2], v[3], hi, lo);
                    *reinterpret_cast<uint32_t *>(Mh + swz(r0 + gid + 8, j0, MS)) = hi;
                    *reinterpret_cast<uint32_t *>(Ml + swz(r0 + gid + 8, j0, MS)) = lo;
                }
            }
        }
        __syncthreads();

        // ---- Y += (Λ ∘ C·Bᵀ) · X on the causal blocks (row block mt, column block ks <= mt)
#pragma unroll
        for (int ks = 0; ks < Q / 16; ++ks) {
            uint32_t bf[4];
            frag_b_kn(bf, sm.x, XS, 16 * w, 16 * ks, lane);
#pragma unroll
            for (int mt = 0; mt < Q / 16; ++mt) {
                if (ks <= mt) {
                    uint32_t mh[4], ml[4];
                    frag_a(mh, Mh, MS, 16 * mt, 16 * ks, lane);
                    frag_a(ml, Ml, MS, 16 * mt, 16 * ks, lane);
                    mma16816(Y[mt][0], mh, bf[0], bf[1]);
                    mma16816(Y[mt][1], mh, bf[2], bf[3]);
                    mma16816(Y[mt][0], ml, bf[0], bf[1]);
                    mma16816(Y[mt][1], ml, bf[2], bf[3]);
                }
            }
        }

        // ---- y = Y + D·x, to memory
#pragma unroll
        for (int mt = 0; mt < Q / 16; ++mt) {
#pragma unroll
            for (int nt = 0; nt < 2; ++nt) {
#pragma unroll
                for (int hr = 0; hr < 2; ++hr) {
                    const int i = 16 * mt + gid + 8 * hr, t = t0 + i, p = 16 * w + 8 * nt + 2 * tig;
                    if (t < L) {
                        const __nv_bfloat162 xv = *reinterpret_cast<const __nv_bfloat162 *>(sm.x + swz(i, p, XS));
                        const float y0 = fmaf(Dh, __low2float(xv), Y[mt][nt][2 * hr]);
                        const float y1 = fmaf(Dh, __high2float(xv), Y[mt][nt][2 * hr + 1]);
                        *reinterpret_cast<uint32_t *>(yg + (((size_t)b * L + t) * H + h) * P + p) = pack_bf16(y0, y1);
                    }
                }
            }
        }

        // ---- S_out = e^{cum_{Q−1}} S_in + Xᵀ · diag(w) · B,  w_j = e^{cum_{Q−1} − cum_j}·Δ_j
        __syncthreads();                            // every warp is done reading B, C and the masked block
        const float clast = sm.cum[Q - 1];
        for (int i = tid; i < Q * (NS / 2); i += kThreads) {
            const int r = i / (NS / 2), q = i % (NS / 2);
            const float wj = sm.wsc[r];
            uint32_t *pb = reinterpret_cast<uint32_t *>(sm.B + r * BS) + q;
            const float2 f = __bfloat1622float2(*reinterpret_cast<const __nv_bfloat162 *>(pb));
            uint32_t hi, lo;
            split_bf16(f.x * wj, f.y * wj, hi, lo);
            *pb = hi;
            reinterpret_cast<uint32_t *>(sm.C + r * BS)[q] = lo;   // same swizzled position as in B
        }
        __syncthreads();
        {
            const float et = ex2(clast * kLog2e);
#pragma unroll
            for (int mt = 0; mt < P / 16; ++mt)
#pragma unroll
                for (int nt = 0; nt < 4; ++nt)
#pragma unroll
                    for (int e = 0; e < 4; ++e) Sacc[mt][nt][e] *= et;
#pragma unroll
            for (int ks = 0; ks < Q / 16; ++ks) {
                uint32_t bh0[4], bl0[4], bh1[4], bl1[4];
                frag_b_kn(bh0, sm.B, BS, 32 * w, 16 * ks, lane);
                frag_b_kn(bl0, sm.C, BS, 32 * w, 16 * ks, lane);
                frag_b_kn(bh1, sm.B, BS, 32 * w + 16, 16 * ks, lane);
                frag_b_kn(bl1, sm.C, BS, 32 * w + 16, 16 * ks, lane);
#pragma unroll
                for (int mt = 0; mt < P / 16; ++mt) {
                    uint32_t af[4];
                    frag_a_t(af, sm.x, XS, 16 * mt, 16 * ks, lane);   // A[p][j] = x[j][p]
                    mma16816(Sacc[mt][0], af, bh0[0], bh0[1]);
                    mma16816(Sacc[mt][1], af, bh0[2], bh0[3]);
                    mma16816(Sacc[mt][2], af, bh1[0], bh1[1]);
                    mma16816(Sacc[mt][3], af, bh1[2], bh1[3]);
                    mma16816(Sacc[mt][0], af, bl0[0], bl0[1]);
                    mma16816(Sacc[mt][1], af, bl0[2], bl0[3]);
                    mma16816(Sacc[mt][2], af, bl1[0], bl1[1]);
                    mma16816(Sacc[mt][3], af, bl1[2], bl1[3]);
                }
            }
        }
        // the next chunk's inherited state, as its bf16 operand pair (the
        // masked block in the same buffers is no longer read)
        store_state();
        __syncthreads();
    }

    if (a.hL) {
#pragma unroll
        for (int mt = 0; mt < P / 16; ++mt) {
#pragma unroll
            for (int nt = 0; nt < 4; ++nt) {
#pragma unroll
                for (int e = 0; e < 4; ++e) {
                    const int p = 16 * mt + gid + 8 * (e >> 1), n = 32 * w + 8 * nt + 2 * tig + (e & 1);
                    a.hL[(((size_t)b * H + h) * P + p) * NS + n] = Sacc[mt][nt][e];
                }
            }
        }
    }
}

}  // namespace

bool ssd_supported(int64_t headdim, int64_t dstate) { return headdim == P && dstate == NS; }

cudaError_t ssd_launch(const SsdArgs &a, cudaStream_t st) {
    constexpr size_t smem = sizeof(SsdSmem);
    static PerDevice attr;  // the shared-memory limit is raised once per device
    int done = 0;
    const cudaError_t e = attr.get(
        [&](int *v) {
            *v = 1;
            return cudaFuncSetAttribute(ssd_kernel, cudaFuncAttributeMaxDynamicSharedMemorySize, (int)smem);
        },
        &done);
    if (e != cudaSuccess) return e;
    ssd_kernel<<<a.batch * a.nheads, kThreads, smem, st>>>(a);
    return cudaGetLastError();
}

}  // namespace ssm
