// ssd.cu — the Mamba-2 layer scan (state space duality) for sm_103a, on the
// tcgen05 tensor cores.
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
// Per chunk of Q = 128 tokens (cum_i = Σ_{k<=i} Δ_k A_h within the chunk,
// w_j = e^{cum_{Q−1} − cum_j}·Δ_j):
//   G     = C · Bᵀ                                        (Q × Q, K = N)
//   M     = G ∘ Λ,  Λ_ij = e^{cum_i − cum_j}·Δ_j for j <= i, else 0
//   Y     = M · X  +  diag(e^{cum}) · C · S_in  +  D_h · X   (Q × P)
//   S_out = e^{cum_{Q−1}} · S_in  +  Bᵀ · diag(w) · X         (N × P)
// Every product is a chain of tcgen05 MMAs (kind::f16, bf16 operands, fp32
// accumulators in tensor memory, M = 128 rows).  C, B and X arrive by TMA as
// 128-byte-swizzled tiles and the MMAs read them where they lie: C and B
// K-major for G, C K-major for the state read-out, B along its token rows
// (MN-major) for the chunk state, X MN-major.  The operands that are not
// inputs — M, the inherited state and the weighted X — are written by the
// math warps as a bf16 value and a bf16 remainder, so they carry ~16 bits
// instead of bf16's 8: M into tensor memory in place of G (the A operand of
// M · X), the other two into shared memory stacked along N (one MMA of
// N = 128 gives both halves, which the epilogue adds).
//
// One CTA per (sequence, head) walks its chunks in order (the state is the
// chain).  Warp 0 issues the TMA copies and the MMAs from one lane; eight math
// warps (warps 4 .. 11) — two per TMEM lane quarter, each taking half the
// columns — form Δ and its prefix sums, the weighted X, the masked block, y and
// the next state, and hand each operand to warp 0 through an mbarrier.  Warps
// 1 .. 3 only complete warp 0's warpgroup, so that setmaxnreg can move their
// registers to the math warpgroups (the control code needs ~110 registers
// without spilling, the math code more than the 168 a 12-warp launch gives
// every thread).  Inputs are double-buffered, so chunk k+2's tiles load while
// chunk k+1 runs.  Shapes built: P = 64, N = 128, bf16 I/O.
#include <algorithm>
#include <cstring>

#include "ssm_device.cuh"
#include "ssm_internal.h"
#include "tcgen05.cuh"

namespace ssm {
namespace {

constexpr int Q = 128;                 // tokens per chunk (MMA rows)
constexpr int P = 64;                  // head dimension
constexpr int NS = 128;                // state size
constexpr int kMath = 8;               // math warps: warps 4 .. 11, two warpgroups
constexpr int kCtrl = 0;               // the control warp: MMAs from its lane 0
constexpr int kFirstMath = 4;          // warps 1 .. 3 only make up the control warpgroup
constexpr int kThreads = 32 * (kFirstMath + kMath);
// Registers per thread after the split: the control warpgroup gives up what the
// math warpgroups take (launch: 384 threads × 168; 128 × 40 + 256 × 232 = 384 × 168).
constexpr int kCtrlRegs = 112, kMathRegs = 192;
static_assert(4 * 32 * kCtrlRegs + kMath * 32 * kMathRegs <= kThreads * 168, "register split");
constexpr uint32_t kWaitLimit = 1u << 22;
constexpr int kStatusTimeout = 4;      // SSM_ERR_TIMEOUT
constexpr int kFlagLimit = 1 << 24;    // polls of the previous segment's flag (≈1 µs each)

// Shared memory: 128-byte-swizzled slabs of 128 rows × 128 bytes (1024-byte aligned).
constexpr int kSlab = 128 * 128;
constexpr int kBufC = 0, kBufB = 2 * kSlab, kBufX = 4 * kSlab;  // within one input buffer:
constexpr int kBuf = 5 * kSlab;        // C [token][n] and B [token][n] (2 slabs each), X [token][p]
constexpr int kOffW = 2 * kBuf;        // weighted X [j][p]: value slab, remainder slab
constexpr int kOffS = kOffW + 2 * kSlab;   // inherited state [n][p]: value slab, remainder slab
constexpr int kOffF = kOffS + 2 * kSlab;   // floats: Δ[Q], cum[Q] (log2 units)
constexpr int kOffBar = kOffF + 2 * Q * 4;
constexpr int kNumBars = 9;
constexpr int kOffMisc = kOffBar + kNumBars * 8;   // TMEM base, failure flag
constexpr int kSmemUsed = kOffMisc + 16;
constexpr int kSmemBytes = kSmemUsed + 1024;   // slack to align the base to 1024 bytes
static_assert(kSmemBytes <= 232448, "shared memory per CTA");

// TMEM columns (fp32 accumulators, lane = row).  G is overwritten in place by
// the masked block's bf16 value / remainder pairs.
constexpr uint32_t kColG = 0, kColY1 = 128, kColY2 = 256, kColS = 384, kTmemCols = 512;

struct Maps {
    CUtensorMap x, B, C, y;
};

// Byte offset of 16-byte chunk c (elements 8c .. 8c+7) of row r in a swizzled slab.
__device__ __forceinline__ int sw128(int r, int c) { return r * 128 + ((c ^ (r & 7)) << 4); }

__device__ __forceinline__ uint32_t pack_bf16(float lo, float hi) {
    const __nv_bfloat162 v = __floats2bfloat162_rn(lo, hi);
    return *reinterpret_cast<const uint32_t *>(&v);
}
// (v0, v1) as two bf16 pairs: the values cut to bf16 and the remainders rounded
// to bf16 (value + remainder is within 2^-16 of v, relatively).
__device__ __forceinline__ void split_bf16(float v0, float v1, uint32_t &hi, uint32_t &lo) {
    const uint32_t b0 = __float_as_uint(v0) & 0xffff0000u, b1 = __float_as_uint(v1) & 0xffff0000u;
    hi = __byte_perm(b0, b1, 0x7632);
    lo = pack_bf16(v0 - __uint_as_float(b0), v1 - __uint_as_float(b1));
}
// Eight values as a 16-byte value chunk and a 16-byte remainder chunk.
__device__ __forceinline__ void split8(const float *v, uint4 &hi, uint4 &lo) {
    split_bf16(v[0], v[1], hi.x, lo.x);
    split_bf16(v[2], v[3], hi.y, lo.y);
    split_bf16(v[4], v[5], hi.z, lo.z);
    split_bf16(v[6], v[7], hi.w, lo.w);
}
__device__ __forceinline__ void unpack8(uint4 w, float *o) {
    const uint32_t ws[4] = {w.x, w.y, w.z, w.w};
#pragma unroll
    for (int k = 0; k < 4; ++k) {
        o[2 * k] = __uint_as_float(ws[k] << 16);
        o[2 * k + 1] = __uint_as_float(ws[k] & 0xffff0000u);
    }
}

// 32 consecutive columns of this warp's TMEM lane quarter, one register each.
__device__ __forceinline__ void ld32(uint32_t ta, float *v) {
    uint32_t r[32];
    asm volatile(
        "tcgen05.ld.sync.aligned.32x32b.x32.b32 {%0, %1, %2, %3, %4, %5, %6, %7, %8, %9, %10, %11, %12, %13, %14, "
        "%15, %16, %17, %18, %19, %20, %21, %22, %23, %24, %25, %26, %27, %28, %29, %30, %31}, [%32];"
        : "=r"(r[0]), "=r"(r[1]), "=r"(r[2]), "=r"(r[3]), "=r"(r[4]), "=r"(r[5]), "=r"(r[6]), "=r"(r[7]),
          "=r"(r[8]), "=r"(r[9]), "=r"(r[10]), "=r"(r[11]), "=r"(r[12]), "=r"(r[13]), "=r"(r[14]), "=r"(r[15]),
          "=r"(r[16]), "=r"(r[17]), "=r"(r[18]), "=r"(r[19]), "=r"(r[20]), "=r"(r[21]), "=r"(r[22]), "=r"(r[23]),
          "=r"(r[24]), "=r"(r[25]), "=r"(r[26]), "=r"(r[27]), "=r"(r[28]), "=r"(r[29]), "=r"(r[30]), "=r"(r[31])
        : "r"(ta)
        : "memory");
    asm volatile("tcgen05.wait::ld.sync.aligned;" ::: "memory");
#pragma unroll
    for (int i = 0; i < 32; ++i) v[i] = __uint_as_float(r[i]);
}
__device__ __forceinline__ void st16(uint32_t ta, const uint32_t *r) {
    asm volatile(
        "tcgen05.st.sync.aligned.32x32b.x16.b32 [%0], {%1, %2, %3, %4, %5, %6, %7, %8, %9, %10, %11, %12, %13, "
        "%14, %15, %16};" ::"r"(ta),
        "r"(r[0]), "r"(r[1]), "r"(r[2]), "r"(r[3]), "r"(r[4]), "r"(r[5]), "r"(r[6]), "r"(r[7]), "r"(r[8]),
        "r"(r[9]), "r"(r[10]), "r"(r[11]), "r"(r[12]), "r"(r[13]), "r"(r[14]), "r"(r[15])
        : "memory");
}

// Instruction descriptor: fp32 accumulator, bf16 A and B, M × N; a_mn / b_mn
// set when that operand is MN-major (its M or N index runs along the rows).
__host__ __device__ constexpr uint32_t idesc_bf16(uint32_t M, uint32_t N, uint32_t a_mn, uint32_t b_mn) {
    return (1u << 4) | (1u << 7) | (1u << 10) | (a_mn << 15) | (b_mn << 16) | ((N >> 3) << 17) | ((M >> 4) << 24);
}
// Operand descriptor of a 128-byte-swizzled tile, 8-row groups 1024 bytes
// apart.  K-major (K along the 128-byte rows): a K-step of 16 elements starts
// 32 bytes on.  MN-major (K down the rows): a K-step of 16 rows starts 2048
// bytes on, and 64-element blocks of M or N lie `lbo` bytes apart.
__device__ __forceinline__ uint64_t desc_sw128(uint32_t addr, uint32_t lbo) {
    return (uint64_t)((addr & 0x3FFFF) >> 4) | ((uint64_t)(lbo >> 4) << 16) | ((uint64_t)(1024 >> 4) << 32) |
           (1ull << 46) | (2ull << 61);
}
// D (TMEM) (+)= A · B, both from shared memory, issued by one thread.
__device__ __forceinline__ void mma_ss(uint32_t d, uint64_t ad, uint64_t bd, uint32_t idesc, bool acc) {
    asm volatile(
        "{\n\t.reg .pred p;\n\tsetp.ne.b32 p, %4, 0;\n\t"
        "tcgen05.mma.cta_group::1.kind::f16 [%0], %1, %2, %3, p;\n\t}" ::"r"(d),
        "l"(ad), "l"(bd), "r"(idesc), "r"((uint32_t)acc)
        : "memory");
}
// D (TMEM) (+)= A (TMEM) · B (shared memory), issued by one thread.
__device__ __forceinline__ void mma_ts(uint32_t d, uint32_t a, uint64_t bd, uint32_t idesc, bool acc) {
    asm volatile(
        "{\n\t.reg .pred p;\n\tsetp.ne.b32 p, %4, 0;\n\t"
        "tcgen05.mma.cta_group::1.kind::f16 [%0], [%1], %2, %3, p;\n\t}" ::"r"(d),
        "r"(a), "l"(bd), "r"(idesc), "r"((uint32_t)acc)
        : "memory");
}
__device__ __forceinline__ void tma_load_4d(void *dst, const CUtensorMap *map, uint64_t *bar, int c0, int c1, int c2,
                                            int c3) {
    asm volatile(
        "cp.async.bulk.tensor.4d.shared::cluster.global.tile.mbarrier::complete_tx::bytes"
        " [%0], [%1, {%2, %3, %4, %5}], [%6];" ::"r"(smem_u32(dst)),
        "l"(reinterpret_cast<uint64_t>(map)), "r"(c0), "r"(c1), "r"(c2), "r"(c3), "r"(smem_u32(bar))
        : "memory");
}
__device__ __forceinline__ void tma_store_4d(const CUtensorMap *map, const void *src, int c0, int c1, int c2, int c3) {
    asm volatile("cp.async.bulk.tensor.4d.global.shared::cta.tile.bulk_group [%0, {%1, %2, %3, %4}], [%5];" ::"l"(
                     reinterpret_cast<uint64_t>(map)),
                 "r"(c0), "r"(c1), "r"(c2), "r"(c3), "r"(smem_u32(src))
                 : "memory");
}
__device__ __forceinline__ void mbar_arrive(uint64_t *bar) {
    asm volatile("mbarrier.arrive.shared::cta.b64 _, [%0];" ::"r"(smem_u32(bar)) : "memory");
}
// Barrier 1 among the 256 math threads (the control warp does not take part);
// the second form returns whether `p` held on any of them.
__device__ __forceinline__ void math_sync() { asm volatile("bar.sync 1, 256;" ::: "memory"); }
__device__ __forceinline__ bool math_sync_or(bool p) {
    uint32_t r;
    asm volatile(
        "{\n\t.reg .pred p, q;\n\tsetp.ne.u32 p, %1, 0;\n\tbar.red.or.pred q, 1, 256, p;\n\t"
        "selp.u32 %0, 1, 0, q;\n\t}"
        : "=r"(r)
        : "r"((uint32_t)p)
        : "memory");
    return r != 0;
}

// Per chunk k of a (sequence, head):
//   math:    the weighted X (→ w_ready), the masked block from G_k into TMEM
//            (→ m_ready); warp 0 then forms Δ and the prefix sums of Δ·A for
//            chunk k+1 while Y1_k runs; once every product is in, y over X_k in
//            shared memory and the next state, whose bf16 pair goes to shared
//            memory (→ s_ready);
//   control: on s_ready, chunk k−1's y leaves by TMA and chunk k+1's tiles load
//            into its buffer, and Y2_k = C_k · [S_hi | S_lo] is issued; the chunk
//            state [Bᵀ W_hi | Bᵀ W_lo] on w_ready; Y1_k = M_k · X_k on m_ready;
//            then, once Y1_k has read the masked block, G_{k+1} = C_{k+1} B_{k+1}ᵀ.
__global__ void __launch_bounds__(kThreads, 1) ssd_kernel(const __grid_constant__ Maps maps, const SsdArgs a) {
    extern __shared__ unsigned char smem_raw[];
    unsigned char *sm =
        reinterpret_cast<unsigned char *>((reinterpret_cast<uintptr_t>(smem_raw) + 1023) & ~uintptr_t(1023));
    const int tid = threadIdx.x, warp = tid >> 5, lane = tid & 31;
    const int L = a.seqlen, H = a.nheads;
    float *delta = reinterpret_cast<float *>(sm + kOffF), *cum = delta + Q;
    uint64_t *bars = reinterpret_cast<uint64_t *>(sm + kOffBar);
    uint64_t *full = bars, *g_done = bars + 2, *y2_done = bars + 3, *ys_done = bars + 4, *drain = bars + 5;
    uint64_t *w_ready = bars + 6, *m_ready = bars + 7, *s_ready = bars + 8;
    uint32_t *tmem_slot = reinterpret_cast<uint32_t *>(sm + kOffMisc);
    volatile int *fail_flag = reinterpret_cast<volatile int *>(sm + kOffMisc + 4);
    int *item_slot = reinterpret_cast<int *>(sm + kOffMisc + 8);
    if (tid == 0) *item_slot = a.ticket ? atomicAdd(a.ticket, 1) : (int)blockIdx.x;
    __syncthreads();
    // the work item: segment `seg` (chunks c0 .. c0 + nchunks − 1) of the chain
    // (b, h); segments are taken in order, every chain's first segment first
    const int item = *item_slot, chains = a.batch * H;
    const int seg = item / chains, chain = item % chains;
    const int b = chain / H, h = chain % H;
    const int c0 = seg * a.seg_chunks;
    const int nchunks = min((L + Q - 1) / Q - c0, a.seg_chunks);
    const float Ah2 = a.A[h] * kLog2e;     // Δ·A in log2 units
    const float Dh = a.Dskip ? a.Dskip[h] : 0.f;
    const float dbias = a.dt_bias ? a.dt_bias[h] : 0.f;
    const unsigned short *dtg = static_cast<const unsigned short *>(a.dt) + (size_t)b * L * H + h;
    const bool math = warp >= kFirstMath;
    const bool ctrl = tid == 32 * kCtrl;
    const int lead = 32 * kFirstMath;      // the first math thread

    // math warp w: TMEM lane quarter w % 4 (rows 32·(w%4) ..), column half w / 4
    const int qr = warp & 3, hf = ((warp - kFirstMath) >> 2) & 1;
    const int row = 32 * qr + lane;

    if (tid == 0) {
        for (int i = 0; i < 6; ++i) mbar_init(&bars[i], 1);
        for (int i = 6; i < kNumBars; ++i) mbar_init(&bars[i], kMath);
        *fail_flag = 0;
        fence_mbar_init();
    }
    if (warp == kCtrl) tc::alloc(tmem_slot, kTmemCols);
    fence_proxy_async_smem();
    tc::fence_before_sync();
    __syncthreads();
    tc::fence_after_sync();
    const uint32_t tmem = *tmem_slot;
    if (math) asm volatile("setmaxnreg.inc.sync.aligned.u32 %0;" ::"n"(kMathRegs));
    else asm volatile("setmaxnreg.dec.sync.aligned.u32 %0;" ::"n"(kCtrlRegs));
    bool ok = true;
    int issued = 0, seen = 0;   // control thread: chunk loads issued / seen complete

    if (ctrl) {
        // ---------------------------------------------------------------- control
        auto issue_loads = [&](int ck) {
            const int bi = ck & 1;
            unsigned char *buf = sm + bi * kBuf;
            const int t0 = (c0 + ck) * Q;
            mbar_arrive_expect_tx(&full[bi], 5u * kSlab);
            tma_load_4d(buf + kBufX, &maps.x, &full[bi], 0, h, t0, b);
            for (int s = 0; s < 2; ++s) {
                tma_load_3d(buf + kBufC + s * kSlab, &maps.C, &full[bi], 64 * s, t0, b);
                tma_load_3d(buf + kBufB + s * kSlab, &maps.B, &full[bi], 64 * s, t0, b);
            }
            issued = ck + 1;
        };
        // buffer k & 1 takes chunk k, so its barrier completes phase (k >> 1) & 1
        auto wait_loads = [&](int ck) {
            if (mbar_wait_bounded(&full[ck & 1], (ck >> 1) & 1, kWaitLimit)) seen = ck + 1;
            else ok = false;
        };
        auto issue_g = [&](int ck) {   // G = C · Bᵀ (K = n), both K-major
            const uint32_t base = smem_u32(sm + (ck & 1) * kBuf);
            constexpr uint32_t id = idesc_bf16(Q, Q, 0, 0);
#pragma unroll
            for (int ks = 0; ks < NS / 16; ++ks) {
                const uint32_t off = (ks / 4) * kSlab + (ks % 4) * 32;
                mma_ss(tmem + kColG, desc_sw128(base + kBufC + off, 16), desc_sw128(base + kBufB + off, 16), id,
                       ks > 0);
            }
            tc::commit(g_done);
        };
        // chunk ck's y (over its X tile) leaves; ck + 2 then loads into that buffer
        auto store_y = [&](int ck) {
            tma_store_4d(&maps.y, sm + (ck & 1) * kBuf + kBufX, 0, h, (c0 + ck) * Q, b);   // rows past L are clipped
            bulk_commit();
        };
        issue_loads(0);
        if (nchunks > 1) issue_loads(1);
        wait_loads(0);
        tc::fence_after_sync();
        issue_g(0);
        int ck = 0;
        for (; ck < nchunks && ok && !*fail_flag; ++ck) {
            const uint32_t par = ck & 1;
            const uint32_t bufa = smem_u32(sm + (ck & 1) * kBuf);
            // s_ready: the inherited state's pair is written, and chunk k−1's y with it
            if (!mbar_wait_bounded(s_ready, par, kWaitLimit)) ok = false;
            tc::fence_after_sync();
            if (ck > 0) store_y(ck - 1);
            {   // Y2 = C · [S_hi | S_lo] (K = n)
                constexpr uint32_t id = idesc_bf16(Q, 2 * P, 0, 1);
                const uint32_t sb = smem_u32(sm + kOffS);
#pragma unroll
                for (int ks = 0; ks < NS / 16; ++ks) {
                    const uint32_t aoff = (ks / 4) * kSlab + (ks % 4) * 32;
                    mma_ss(tmem + kColY2, desc_sw128(bufa + kBufC + aoff, 16), desc_sw128(sb + ks * 2048, kSlab),
                           id, ks > 0);
                }
                tc::commit(y2_done);
            }
            if (ck > 0 && ck + 1 < nchunks) {
                bulk_wait_read0();      // chunk k−1's y has left its buffer
                issue_loads(ck + 1);
            }
            // [Bᵀ W_hi | Bᵀ W_lo] (K = j): A is the B tile read down its token rows
            if (!mbar_wait_bounded(w_ready, par, kWaitLimit)) ok = false;
            tc::fence_after_sync();
            {
                constexpr uint32_t id = idesc_bf16(NS, 2 * P, 1, 1);
                const uint32_t wb = smem_u32(sm + kOffW);
#pragma unroll
                for (int ks = 0; ks < Q / 16; ++ks)
                    mma_ss(tmem + kColS, desc_sw128(bufa + kBufB + ks * 2048, kSlab),
                           desc_sw128(wb + ks * 2048, kSlab), id, ks > 0);
            }
            // Y1 = M · X (K = j; M from TMEM): the value half of M, then the remainder
            if (!mbar_wait_bounded(m_ready, par, kWaitLimit)) ok = false;
            tc::fence_after_sync();
            {
                constexpr uint32_t id = idesc_bf16(Q, P, 0, 1);
#pragma unroll
                for (int ks = 0; ks < 2 * (Q / 16); ++ks) {
                    const int k = ks % (Q / 16);
                    const uint32_t acol = kColG + 32 * (k / 2) + 8 * (k % 2) + (ks < Q / 16 ? 0 : 16);
                    mma_ts(tmem + kColY1, tmem + acol, desc_sw128(bufa + kBufX + k * 2048, kSlab), id, ks > 0);
                }
                tc::commit(ys_done);
            }
            if (ck + 1 < nchunks) {
                // G_{k+1} overwrites the masked block: wait until Y1_k has read it
                if (!mbar_wait_bounded(ys_done, par, kWaitLimit)) ok = false;
                wait_loads(ck + 1);
                tc::fence_after_sync();
                issue_g(ck + 1);
            }
        }
        // the last chunk's y
        if (ok && ck == nchunks) {
            if (mbar_wait_bounded(s_ready, nchunks & 1, kWaitLimit)) store_y(nchunks - 1);
            else ok = false;
        }
        if (!ok) *fail_flag = 1;
        bulk_wait0();
    } else if (math) {
        // ---------------------------------------------------------------- math
        // the state S[n][p], fp32: thread (row n, half hf) holds p = 32·hf .. 32·hf+31
        float S[32];
        auto store_state = [&]() {   // S as its bf16 value / remainder slabs, rows n
#pragma unroll
            for (int c = 0; c < 4; ++c) {
                uint4 vh, vl;
                split8(S + 8 * c, vh, vl);
                const int off = sw128(row, 4 * hf + c);
                *reinterpret_cast<uint4 *>(sm + kOffS + off) = vh;
                *reinterpret_cast<uint4 *>(sm + kOffS + kSlab + off) = vl;
            }
        };
        // warp 0: Δ and the prefix sums of Δ·A (log2 units) of chunk ck from the
        // raw bf16 dt its lanes hold (tokens 4·lane .. 4·lane+3), then the next
        // chunk's dt, widened only when used so that the loads overlap a chunk
        unsigned short dtr[4] = {0, 0, 0, 0};
        auto fetch_dt = [&](int ck) {
#pragma unroll
            for (int e = 0; e < 4; ++e) {
                const int t = (c0 + ck) * Q + 4 * lane + e;
                if (t < L) dtr[e] = dtg[(size_t)t * H];
            }
        };
        // scan_dt forms the chunk's values in registers; put_dt stores them
        float4 dnext, cnext;
        auto scan_dt = [&](int ck) {
            float d[4], c[4];
            float run = 0.f;
#pragma unroll
            for (int e = 0; e < 4; ++e) {
                const float x = __uint_as_float((uint32_t)dtr[e] << 16) + dbias;
                d[e] = 4 * lane + e + (c0 + ck) * Q < L ? (a.dt_softplus ? softplus_poly(x) : x) : 0.f;
                run = fmaf(d[e], Ah2, run);
                c[e] = run;
            }
            if (ck + 1 < nchunks) fetch_dt(ck + 1);
            float v = run;   // inclusive scan of the lane totals
#pragma unroll
            for (int o = 1; o < 32; o <<= 1) {
                const float u = __shfl_up_sync(0xffffffffu, v, o);
                if (lane >= o) v += u;
            }
            const float before = v - run;
            dnext = make_float4(d[0], d[1], d[2], d[3]);
            cnext = make_float4(before + c[0], before + c[1], before + c[2], before + c[3]);
        };
        auto put_dt = [&]() {
            *reinterpret_cast<float4 *>(delta + 4 * lane) = dnext;
            *reinterpret_cast<float4 *>(cum + 4 * lane) = cnext;
        };
        if (warp == kFirstMath) {
            fetch_dt(0);
            scan_dt(0);
            put_dt();
        }
        // the state entering the segment: h0 (or zero) for a chain's first, else
        // what the previous segment left in the carry once its flag is up
        const float *sin = seg == 0 ? a.h0 : a.carry;
        if (seg > 0) {
            if (tid == lead && !wait_flag(a.flags + chain, seg, kFlagLimit)) ok = false;
            math_sync();
            (void)flag_acquire(a.flags + chain);
        }
#pragma unroll
        for (int j = 0; j < 32; ++j)
            S[j] = sin ? __ldcg(sin + (((size_t)b * H + h) * P + 32 * hf + j) * NS + row) : 0.f;
        store_state();
        fence_proxy_async_smem();
        __syncwarp();
        if (lane == 0) mbar_arrive(s_ready);
        math_sync();   // chunk 0's Δ and prefix sums

        for (int ck = 0; ck < nchunks; ++ck) {
            const uint32_t par = ck & 1;
            unsigned char *buf = sm + (ck & 1) * kBuf;
            const float ci = cum[row], clast = cum[Q - 1], drow = delta[row];

            // ---- the weighted X: w_j · x_j, w_j = e^{cum_last − cum_j}·Δ_j (row j)
            if (!mbar_wait_bounded(&full[ck & 1], (ck >> 1) & 1, kWaitLimit)) ok = false;
            {
                const float wj = ex2(clast - ci) * drow;
#pragma unroll
                for (int c = 0; c < 4; ++c) {
                    const int off = sw128(row, 4 * hf + c);
                    float xv[8];
                    unpack8(*reinterpret_cast<const uint4 *>(buf + kBufX + off), xv);
#pragma unroll
                    for (int e = 0; e < 8; ++e) xv[e] *= wj;
                    uint4 vh, vl;
                    split8(xv, vh, vl);
                    *reinterpret_cast<uint4 *>(sm + kOffW + off) = vh;
                    *reinterpret_cast<uint4 *>(sm + kOffW + kSlab + off) = vl;
                }
                fence_proxy_async_smem();
                __syncwarp();
                if (lane == 0) mbar_arrive(w_ready);
            }

            // ---- the masked block M (rows i) into TMEM over G
            if (!mbar_wait_bounded(g_done, par, kWaitLimit)) ok = false;
            __syncwarp();
            tc::fence_after_sync();
#pragma unroll 1
            for (int cb = 0; cb < 2; ++cb) {   // this warp's 64 columns, 32 at a time
                const int j0 = 64 * hf + 32 * cb;
                uint32_t mh[16], ml[16];
                if (j0 >= 32 * qr) {           // on or above the diagonal: zero for j > i
                    if (j0 > 32 * qr) {
#pragma unroll
                        for (int e = 0; e < 16; ++e) mh[e] = ml[e] = 0u;
                    } else {
                        float g[32];
                        ld32(tc::taddr(tmem, 32 * qr, kColG + j0), g);
#pragma unroll
                        for (int e = 0; e < 8; ++e) {
                            const int j = j0 + 4 * e;
                            const float4 cj = *reinterpret_cast<const float4 *>(cum + j);
                            const float4 dj = *reinterpret_cast<const float4 *>(delta + j);
                            const float m0 = j <= row ? g[4 * e] * dj.x * ex2(ci - cj.x) : 0.f;
                            const float m1 = j + 1 <= row ? g[4 * e + 1] * dj.y * ex2(ci - cj.y) : 0.f;
                            const float m2 = j + 2 <= row ? g[4 * e + 2] * dj.z * ex2(ci - cj.z) : 0.f;
                            const float m3 = j + 3 <= row ? g[4 * e + 3] * dj.w * ex2(ci - cj.w) : 0.f;
                            split_bf16(m0, m1, mh[2 * e], ml[2 * e]);
                            split_bf16(m2, m3, mh[2 * e + 1], ml[2 * e + 1]);
                        }
                    }
                } else {                       // entirely below the diagonal
                    float g[32];
                    ld32(tc::taddr(tmem, 32 * qr, kColG + j0), g);
#pragma unroll
                    for (int e = 0; e < 8; ++e) {
                        const int j = j0 + 4 * e;
                        const float4 cj = *reinterpret_cast<const float4 *>(cum + j);
                        const float4 dj = *reinterpret_cast<const float4 *>(delta + j);
                        split_bf16(g[4 * e] * dj.x * ex2(ci - cj.x), g[4 * e + 1] * dj.y * ex2(ci - cj.y), mh[2 * e],
                                   ml[2 * e]);
                        split_bf16(g[4 * e + 2] * dj.z * ex2(ci - cj.z), g[4 * e + 3] * dj.w * ex2(ci - cj.w),
                                   mh[2 * e + 1], ml[2 * e + 1]);
                    }
                }
                st16(tc::taddr(tmem, 32 * qr, kColG + j0), mh);
                st16(tc::taddr(tmem, 32 * qr, kColG + j0 + 16), ml);
            }
            asm volatile("tcgen05.wait::st.sync.aligned;" ::: "memory");
            tc::fence_before_sync();
            __syncwarp();
            if (lane == 0) mbar_arrive(m_ready);

            // ---- warp 0: the next chunk's Δ and prefix sums while Y1 runs, stored
            // once every math warp is past its masked block (the last reader)
            if (warp == kFirstMath && ck + 1 < nchunks) {
                scan_dt(ck + 1);
                if (!mbar_wait_bounded(m_ready, par, kWaitLimit)) ok = false;
                __syncwarp();
                put_dt();
            }

            // ---- y = Y1 + e^{cum_i}·Y2 + D·x (rows i, over X), S = e^{cum_last}·S + chunk state (rows n)
            {
                const float ei = ex2(ci), el = ex2(clast);
                if (!mbar_wait_bounded(y2_done, par, kWaitLimit)) ok = false;
                if (!mbar_wait_bounded(ys_done, par, kWaitLimit)) ok = false;
                __syncwarp();
                tc::fence_after_sync();
#pragma unroll
                for (int c = 0; c < 4; ++c) {   // 8 columns p = 32·hf + 8c .. at a time
                    const int col = 32 * hf + 8 * c;
                    uint32_t y1[8], yh[8], yl[8], sh[8], sl[8];
                    tc::ld8_nowait(tc::taddr(tmem, 32 * qr, kColY1 + col), y1);
                    tc::ld8_nowait(tc::taddr(tmem, 32 * qr, kColY2 + col), yh);
                    tc::ld8_nowait(tc::taddr(tmem, 32 * qr, kColY2 + P + col), yl);
                    tc::ld8_nowait(tc::taddr(tmem, 32 * qr, kColS + col), sh);
                    tc::ld8_nowait(tc::taddr(tmem, 32 * qr, kColS + P + col), sl);
                    tc::wait_ld();
                    const int off = sw128(row, col / 8);
                    float xv[8], yv[8];
                    unpack8(*reinterpret_cast<const uint4 *>(buf + kBufX + off), xv);
#pragma unroll
                    for (int e = 0; e < 8; ++e) {
                        const float y2 = __uint_as_float(yh[e]) + __uint_as_float(yl[e]);
                        yv[e] = fmaf(ei, y2, fmaf(Dh, xv[e], __uint_as_float(y1[e])));
                        S[8 * c + e] = fmaf(el, S[8 * c + e], __uint_as_float(sh[e]) + __uint_as_float(sl[e]));
                    }
                    *reinterpret_cast<uint4 *>(buf + kBufX + off) = make_uint4(
                        pack_bf16(yv[0], yv[1]), pack_bf16(yv[2], yv[3]), pack_bf16(yv[4], yv[5]), pack_bf16(yv[6], yv[7]));
                }
                tc::fence_before_sync();
                store_state();   // Y2_k has completed: the slabs are free
                fence_proxy_async_smem();
                __syncwarp();
                if (lane == 0) mbar_arrive(s_ready);   // the next state's pair and this chunk's y
            }
            // the next chunk's Δ and prefix sums are visible; stop together on a failure
            if (math_sync_or(!ok)) {
                if (tid == lead) *fail_flag = 1;
                break;
            }
        }
        // a chain's last segment writes hL; the others hand the state on
        const bool last = c0 + nchunks >= (L + Q - 1) / Q;
        float *sout = last ? a.hL : a.carry;
        if (sout && in_range(((int64_t)b * H + h) * P * NS, P * NS, (int64_t)a.batch * H * P * NS)) {
#pragma unroll
            for (int j = 0; j < 32; ++j) sout[(((size_t)b * H + h) * P + 32 * hf + j) * NS + row] = S[j];
        }
        if (!last) {
            // every math thread's state stores precede the flag (barrier, then a
            // release at device scope by one thread)
            math_sync();
            if (tid == lead) {
                __threadfence();
                flag_release(a.flags + chain, seg + 1);
            }
        }
    }
    __syncwarp();
    __syncthreads();   // both roles are done: every load that will be issued is issued
    if (ctrl && (!ok || *fail_flag || seen < issued)) {
        // a bounded wait ran out: let this CTA's copies and products in flight
        // finish (again bounded) before the tensor memory goes
        for (int c = seen; c < issued; ++c) mbar_wait_bounded(&full[c & 1], (c >> 1) & 1, kWaitLimit);
        tc::commit(drain);
        mbar_wait_bounded(drain, 0, kWaitLimit);
    }
    if (!ok && a.status) record_error(a.status, kStatusTimeout);
    tc::fence_before_sync();
    __syncthreads();
    tc::fence_after_sync();
    if (warp == kCtrl) tc::dealloc(tmem, kTmemCols);
}

// A bf16 tensor map with 128-byte swizzle: `rank` dims innermost first, the
// byte strides of dims 1.., the box.
bool make_map(CUtensorMap *m, const void *ptr, int rank, const cuuint64_t *dims, const cuuint64_t *strides,
              const cuuint32_t *box) {
    TensorMapEncodeFn fn = tensor_map_encoder();
    if (!fn) return false;
    const cuuint32_t estr[4] = {1, 1, 1, 1};
    return fn(m, CU_TENSOR_MAP_DATA_TYPE_BFLOAT16, rank, const_cast<void *>(ptr), dims, strides, box, estr,
              CU_TENSOR_MAP_INTERLEAVE_NONE, CU_TENSOR_MAP_SWIZZLE_128B, CU_TENSOR_MAP_L2_PROMOTION_L2_256B,
              CU_TENSOR_MAP_FLOAT_OOB_FILL_NONE) == CUDA_SUCCESS;
}

}  // namespace

bool ssd_supported(int64_t headdim, int64_t dstate) { return headdim == P && dstate == NS; }

// Segments per chain.  One CTA per SM runs a segment at a time, so the launch
// takes ⌈segments × chains / SMs⌉ rounds, each as long as a segment plus its
// start: ≈2.5 chunk-times (CTA start, TMEM allocation, the first tiles' load
// from memory and G before the pipeline is full), fitted to B300 timings of the
// 4 × 2048 and 8 × 4096 token, 80-head layers split into 1, 2 and 4 segments.
// The split with the fewest chunk-times wins, up to four segments.
SsdPlan ssd_plan(int64_t batch, int64_t seqlen, int64_t nheads, bool split) {
    const int64_t nch = (seqlen + Q - 1) / Q, chains = batch * nheads;
    SsdPlan p{(int)nch, 1};
    if (!split) return p;
    const int64_t sms = sm_count();
    double best = 1e300;
    for (int64_t s = 1; s <= std::min<int64_t>(4, nch); ++s) {
        const int64_t per = (nch + s - 1) / s, nseg = (nch + per - 1) / per;
        const double t = (double)((nseg * chains + sms - 1) / sms) * ((double)per + 2.5);
        if (t < best * 0.999) {
            best = t;
            p = SsdPlan{(int)per, (int)nseg};
        }
    }
    return p;
}

cudaError_t ssd_launch(const SsdArgs &a, int nseg, cudaStream_t st) {
    Maps maps;
    memset(&maps, 0, sizeof(maps));
    const cuuint64_t Lb = (cuuint64_t)a.seqlen, Bb = (cuuint64_t)a.batch, Hh = (cuuint64_t)a.nheads;
    // x, y: (batch, L, H, P) as dims (P, H, L, batch); a box is one head × Q tokens
    const cuuint64_t xd[4] = {P, Hh, Lb, Bb}, xs[3] = {P * 2, Hh * P * 2, Lb * Hh * P * 2};
    const cuuint32_t xbox[4] = {P, 1, Q, 1};
    // B, C: (batch, L, N) as dims (N, L, batch); a box is 64 states × Q tokens
    const cuuint64_t bd[3] = {NS, Lb, Bb}, bs[2] = {NS * 2, Lb * NS * 2};
    const cuuint32_t bbox[3] = {64, Q, 1};
    const bool ok = make_map(&maps.x, a.x, 4, xd, xs, xbox) && make_map(&maps.y, a.y, 4, xd, xs, xbox) &&
                    make_map(&maps.B, a.B, 3, bd, bs, bbox) && make_map(&maps.C, a.C, 3, bd, bs, bbox);
    if (!ok) return cudaErrorInvalidValue;
    static PerDevice attr;  // the shared-memory limit is raised once per device
    int done = 0;
    const cudaError_t e = attr.get(
        [&](int *v) {
            *v = 1;
            return cudaFuncSetAttribute(ssd_kernel, cudaFuncAttributeMaxDynamicSharedMemorySize, kSmemBytes);
        },
        &done);
    if (e != cudaSuccess) return e;
    ssd_kernel<<<nseg * a.batch * a.nheads, kThreads, kSmemBytes, st>>>(maps, a);
    return cudaGetLastError();
}

SSM_DEBUG_WORD_READER(debug_word_ssd)

}  // namespace ssm
