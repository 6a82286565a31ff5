// scan_fwd.cu — the fused Mamba selective scan for sm_103a.
//
// What one launch computes is the recurrence of "Mamba and selective state
// spaces, from first principles" ("Selection", "Discretisation: zero-order
// hold", "The hardware-aware scan"): for every channel (b, d) and state n,
//   Δ = softplus(Δraw + bias), Ā = exp(Δ·A), h = Ā·h + Δ·B·u,
//   y = (C·h + D·u)·silu(z),
// writing only y (b × D × L) and the final state — never Ā, B̄ or any h_t.
//
// Design (B300-first, not the pages' kernel).  One state update costs one
// MUFU exponential and four FP32 operations (Δ·A, B·Δu, Ā·h + B̄u, C·h).  On
// this part the FP32 pipe and the MUFU are both busy at the same rate, and a
// scheduler needs at least two resident warps to keep them fed, so:
//   * A warp owns a group of CPW channels; NG = 1 or 2 lanes share a channel
//     and each lane keeps SPT of its states in registers (scalar fp32 math,
//     Ā = ex2.approx of Δ·A·log2e) while walking the time axis in order.
//     With two lanes per channel the per-token partial sums C·h are combined
//     with a transposed shuffle over four tokens.
//   * Each lane forms softplus(Δraw + bias), Δ·u, silu(z) and D·u·silu(z) for
//     its channel straight from the staged bf16/fp32 tile in registers; no
//     per-token intermediate goes through shared memory.
//   * Warps are persistent and take work items — (channel group, chunk of the
//     sequence) — from a counter.  Chained mode hands items out chunk-major,
//     and chunk k of a group starts from the state chunk k-1 published
//     (waiting on a flag, with a bounded spin): every warp stays busy until
//     the end whatever the channel count, with no extra pass.  When there are
//     too few groups to fill the GPU, look-back mode cuts the sequence into
//     chunks that run at once, in the same one launch: every warp first takes
//     aggregate items, which walk a chunk (every chunk but the last) from a
//     zero state and publish its pair (Π Ā, h_end), and then main items, which
//     compose their predecessors' pairs from h0 (the affine composition of the
//     first-principles page, "The hardware-aware scan") for the state they
//     start from, publish the state they leave, and scan from there.
//   * Per tile of TT tokens one lane moves u, Δraw, z (as 8-token × CPW-channel
//     boxes) and B, C (N × TT, shared by every channel) into shared memory with
//     TMA on an mbarrier, two stages deep; the next tile — of the same item or
//     of the next item — loads while this one is scanned.  y leaves with TMA
//     stores from a double-buffered tile.
//   * With bf16 I/O and first-order discretisation the main pass runs warp-
//     specialised (scan_ws_kernel): a producer warp issues the loads and forms
//     the per-token terms, and a consumer warp runs only the recurrence.
#include <algorithm>
#include <cstring>

#include "ssm_device.cuh"
#include "ssm_internal.h"

namespace ssm {

#ifndef SSM_SCAN_N16_LANES
#define SSM_SCAN_N16_LANES 2
#endif
#ifndef SSM_SCAN_WARPS_PER_SM
#define SSM_SCAN_WARPS_PER_SM 8
#endif

#ifndef SSM_SCAN_PACKED
#define SSM_SCAN_PACKED 1
#endif
#ifndef SSM_SCAN_SCALAR_X
#define SSM_SCAN_SCALAR_X 0
#endif
#ifndef SSM_SCAN_SCALAR_H
#define SSM_SCAN_SCALAR_H 0
#endif

// Pairwise fp32 arithmetic of the recurrence, packed f32x2 by default.  A
// microbenchmark of the bare update alone (Δ·A, ex2, B·Δu, Ā·h + B̄u, C·h, no
// loads) retires 5.2 T updates/s with scalar FFMA/FMUL against 4.0 T packed at
// 8 warps per SM, but in the whole kernel, where issue slots are the limit, the
// scalar form's extra instructions cost more (290.6 µs against 262 µs on the
// 4 × 5120 × 2048 layer).  SSM_SCAN_SCALAR_X / _H make only the product that
// feeds the exponential, or the state update, scalar.
__device__ __forceinline__ float2 mul2(float2 a, float2 b) {
#if SSM_SCAN_PACKED
    return __fmul2_rn(a, b);
#else
    return make_float2(a.x * b.x, a.y * b.y);
#endif
}
__device__ __forceinline__ float2 fma2(float2 a, float2 b, float2 c) {
#if SSM_SCAN_PACKED
    return __ffma2_rn(a, b, c);
#else
    return make_float2(fmaf(a.x, b.x, c.x), fmaf(a.y, b.y, c.y));
#endif
}
__device__ __forceinline__ float2 add2(float2 a, float2 b) {
#if SSM_SCAN_PACKED
    return __fadd2_rn(a, b);
#else
    return make_float2(a.x + b.x, a.y + b.y);
#endif
}

constexpr int kTT = 32;                // tokens per tile (chunks are multiples of 64)
constexpr int kWarpsPerSM = SSM_SCAN_WARPS_PER_SM;  // resident warps targeted per SM
constexpr int kSMs = 148;              // B300
constexpr int kWaitLimit = 1 << 22;    // mbarrier polls before giving up
constexpr int kFlagLimit = 1 << 24;    // polls of a predecessor's flag before giving up
// Tokens per work item in chained mode.  Each item start costs the consumer a
// hand-off (flag, carried state); on the 4 × 5120 × 16 × 2048 layer 128 / 256 /
// 384 / 512 / 768-token items ran in 256 / 238 / 224 / 228 / 247 µs.
constexpr int kDefaultChunk = 384;

__host__ __device__ constexpr int al128(int x) { return (x + 127) / 128 * 128; }

// Shared-memory layout of one warp's CTA (byte offsets; TMA destinations 128-B
// aligned).  u, Δraw, z and y tiles are stored as [TT/8][CPW channels][8 tokens]:
// a channel's 8 tokens are one contiguous 16-byte (bf16) or 32-byte (fp32) run
// and each [CPW][8] block is one TMA box.
template <typename T, int SPT, int NG> struct WTile {
    static_assert(SPT % 4 == 0 && (NG == 1 || NG == 2), "tile shape");
    static constexpr int CPW = 32 / NG;           // channels per warp
    static constexpr int NP = SPT * NG;           // states covered (>= N)
    static constexpr int ES = (int)sizeof(T);
    static constexpr int NB8 = kTT / 8;           // 8-token blocks per tile
    static constexpr int BLK = CPW * 8 * ES;      // one 8-token block of one input
    static constexpr int SEQ = NB8 * BLK;         // one input tile
    static constexpr int BC = kTT * NP * 4;       // one fp32 B or C tile, token-major rows of NP
    static constexpr int BUF = 3 * al128(SEQ) + 2 * al128(BC);  // one stage: u, Δ, z, B, C
    static constexpr int off_u = 0, off_d = al128(SEQ), off_z = 2 * al128(SEQ);
    static constexpr int off_B = 3 * al128(SEQ), off_C = off_B + al128(BC);
    static constexpr int OUT = al128(SEQ);                       // one y tile
    static constexpr int off_out = 2 * BUF;                      // two y tiles
    static constexpr int off_ex = off_out + 2 * OUT;             // (Δ, Δ·u) of one 8-token block
    static constexpr int off_bar = off_ex + al128(CPW * 5 * 16);  // 5 slots per channel: 4 + 1 pad
    static constexpr int bytes = off_bar + 16;
};

struct Maps {
    CUtensorMap u, d, z, B, C, y;
};

template <typename T> struct Pack;
template <> struct Pack<float> {
    __device__ __forceinline__ static void store8(float *p, const float *v) {
        reinterpret_cast<float4 *>(p)[0] = make_float4(v[0], v[1], v[2], v[3]);
        reinterpret_cast<float4 *>(p)[1] = make_float4(v[4], v[5], v[6], v[7]);
    }
    __device__ __forceinline__ static void store2(float *p, float2 v) { *reinterpret_cast<float2 *>(p) = v; }
    __device__ __forceinline__ static void store4(float *p, float2 a, float2 b) {
        *reinterpret_cast<float4 *>(p) = make_float4(a.x, a.y, b.x, b.y);
    }
};
template <> struct Pack<__nv_bfloat16> {
    __device__ __forceinline__ static uint32_t pk(float a, float b) {
        const __nv_bfloat162 v = __floats2bfloat162_rn(a, b);
        return *reinterpret_cast<const uint32_t *>(&v);
    }
    __device__ __forceinline__ static void store8(__nv_bfloat16 *p, const float *v) {
        *reinterpret_cast<uint4 *>(p) = make_uint4(pk(v[0], v[1]), pk(v[2], v[3]), pk(v[4], v[5]), pk(v[6], v[7]));
    }
    __device__ __forceinline__ static void store2(__nv_bfloat16 *p, float2 v) {
        *reinterpret_cast<uint32_t *>(p) = pk(v.x, v.y);
    }
    __device__ __forceinline__ static void store4(__nv_bfloat16 *p, float2 a, float2 b) {
        *reinterpret_cast<uint2 *>(p) = make_uint2(pk(a.x, a.y), pk(b.x, b.y));
    }
};


// One work item: a group of CPW channels of one sequence, one chunk of tokens.
struct Item {
    int grp, k, b, d0, t_begin, t_end, ntiles;
};

// ---------------------------------------------------------------- look-back carry
// Chunks of one channel group that run at once join up through the affine
// composition of the first-principles page ("The hardware-aware scan"): chunk
// k's pair (P_k, S_k) = (Π Ā, h_end from a zero state) maps the state entering
// it to the state leaving it, h -> P_k·h + S_k.  Per (group, chunk) a flag in
// the workspace says what is out: 0 nothing, 1 the pair (in a.agg, written by
// the chunk's aggregate item), 2 also the state leaving the chunk (in a.carry,
// slot k + 1, written by its main item before it scans).  In a look-back
// launch every warp runs aggregate items (chunks 0 .. K-2) until their counter
// runs out and then main items; main items wait only on aggregate items, which
// wait on nothing and were all taken by running warps before any main item
// was, so every wait ends.  A lane holds states n = SPT·g + 2q + e of channel
// d as h[q].{x, y}.

// End of chunk it.k's aggregate item, with h the state reached from zero and
// dsum = Σ Δ over the chunk: publishes the pair (flag 1).  A2 holds A·log2(e),
// so P = 2^(A2·ΣΔ) = exp(A·ΣΔ).  The warp barrier orders every lane's stores
// before lane 0's release store.
template <int SPT, int NQ>
__device__ __forceinline__ void publish_pair(const ScanArgs &a, const Item &it, int d, bool live, int g, int lane,
                                             const float2 (&A2)[NQ], float dsum, const float2 (&h)[NQ]) {
    const int D = a.dim, N = a.dstate, K = a.nchunks;
    const int64_t at = (((int64_t)it.b * D + d) * (K - 1) + it.k) * N;
    if (live && in_range(at, N, (int64_t)a.batch * D * (K - 1) * N)) {
#pragma unroll
        for (int q = 0; q < NQ; ++q) {
            const int n = SPT * g + 2 * q;
            if (n < N) a.agg[at + n] = make_float2(ex2(A2[q].x * dsum), h[q].x);
            if (n + 1 < N) a.agg[at + n + 1] = make_float2(ex2(A2[q].y * dsum), h[q].y);
        }
    }
    __syncwarp();
    if (lane == 0) flag_release(a.flags + (size_t)it.grp * K + it.k, 1);
}

// Start of chunk it.k's main item: sets h to the state entering the chunk and,
// but for the last chunk, writes the state leaving it to a.carry; the caller
// then releases flag 2 (release_leaving) once the item's first tile is done,
// when those stores have long landed.  The walk goes back along the group's
// flags to the nearest chunk whose leaving state is out (else to h0) and
// carries that state forward through the pairs in between, oldest first, one
// fmaf per chunk and state: whichever chunk the walk stops at, the bits are
// those of h0 carried chunk by chunk.  Lane i reads the flag of the i-th
// predecessor, 32 at a time, so one round trip finds the stop; the warp
// barrier after the walk orders every lane's reads after the acquire loads
// that saw the flags.  A wait that runs out records SSM_ERR_TIMEOUT and the
// walk goes on with what is there.
template <int SPT, int NQ>
__device__ __forceinline__ void enter_chunk(const ScanArgs &a, const Item &it, int d, bool live, int g, int lane,
                                            float2 (&h)[NQ]) {
    constexpr unsigned FULL = 0xffffffffu;
    const int D = a.dim, N = a.dstate, K = a.nchunks, k = it.k;
    const bool leaves = k < K - 1;  // the state leaving the chunk is published
    const int *fl = a.flags + (size_t)it.grp * K;
    bool ok = true;
    int j = -1;                     // the chunk whose leaving state the walk starts from
    int base = k - 1;               // lane i looks at chunk base - i
    bool own = !leaves;             // the chunk's own pair is out
    for (int polls = 1;; ++polls) {
        if (!own) own = __all_sync(FULL, flag_acquire(fl + k) >= 1);
        bool found = base < 0;
        if (!found) {
            const int m = base - lane;
            const int f = m >= 0 ? flag_acquire(fl + m) : 1;  // before chunk 0: h0
            const unsigned two = __ballot_sync(FULL, m >= 0 && f == 2);
            const unsigned none = __ballot_sync(FULL, f == 0);
            const unsigned nearer = two ? (two & (0u - two)) - 1u : FULL;  // lanes before the first 2
            if (!(none & nearer)) {
                if (two) {
                    j = base - (__ffs(two) - 1);
                    found = true;
                } else {
                    base -= 32;  // every pair in this window is out: look further back
                    found = base < 0;
                    if (!found) continue;
                }
            }
        }
        if (found && own) break;
        if (polls >= kFlagLimit) {
            ok = false;
            j = -1;
            break;
        }
        __nanosleep(64);
    }
    __syncwarp();
    const size_t bd = (size_t)it.b * D + d;
    const int64_t agg_size = (int64_t)a.batch * D * (K - 1) * N;
    // the chunk's own pair first: its loads do not wait on the walk's
    float2 P[NQ], S[NQ];
#pragma unroll
    for (int q = 0; q < NQ; ++q) {
        P[q] = make_float2(1.f, 1.f);
        S[q] = make_float2(0.f, 0.f);
    }
    const float2 *own_pair = a.agg + (bd * (K - 1) + k) * N;
    const bool use_own = leaves && live && in_range((int64_t)(bd * (K - 1) + k) * N, N, agg_size);
    if (use_own) {
#pragma unroll
        for (int q = 0; q < NQ; ++q) {
            const int n = SPT * g + 2 * q;
            if (n < N) {
                const float2 ps = __ldcg(own_pair + n);
                P[q].x = ps.x;
                S[q].x = ps.y;
            }
            if (n + 1 < N) {
                const float2 ps = __ldcg(own_pair + n + 1);
                P[q].y = ps.x;
                S[q].y = ps.y;
            }
        }
    }
    const float *src = nullptr;
    if (j >= 0) src = a.carry + (bd * K + j + 1) * N;
    else if (a.h0) src = a.h0 + bd * N;
#pragma unroll
    for (int q = 0; q < NQ; ++q) {
        const int n = SPT * g + 2 * q;
        float hx = 0.f, hy = 0.f;
        if (src && live) {
            if (n < N) hx = __ldcg(src + n);
            if (n + 1 < N) hy = __ldcg(src + n + 1);
        }
        h[q] = make_float2(hx, hy);
    }
#pragma unroll 1
    for (int m = j + 1; m < k; ++m) {  // h <- P_m·h + S_m
        if (!live || !in_range((int64_t)(bd * (K - 1) + m) * N, N, agg_size)) break;
        const float2 *pr = a.agg + (bd * (K - 1) + m) * N;
#pragma unroll
        for (int q = 0; q < NQ; ++q) {
            const int n = SPT * g + 2 * q;
            if (n < N) {
                const float2 ps = __ldcg(pr + n);
                h[q].x = fmaf(ps.x, h[q].x, ps.y);
            }
            if (n + 1 < N) {
                const float2 ps = __ldcg(pr + n + 1);
                h[q].y = fmaf(ps.x, h[q].y, ps.y);
            }
        }
    }
    const int64_t ct = ((int64_t)bd * K + k + 1) * N;
    if (use_own && in_range(ct, N, (int64_t)a.batch * D * K * N)) {
#pragma unroll
        for (int q = 0; q < NQ; ++q) {
            const int n = SPT * g + 2 * q;
            if (n < N) a.carry[ct + n] = fmaf(P[q].x, h[q].x, S[q].x);
            if (n + 1 < N) a.carry[ct + n + 1] = fmaf(P[q].y, h[q].y, S[q].y);
        }
    }
    if (!ok && lane == 0) record_error(a.status, 4 /* SSM_ERR_TIMEOUT */);
}

// Flag 2 for a main item's chunk after enter_chunk wrote its leaving state
// (the warp barrier orders every lane's stores before lane 0's release).
__device__ __forceinline__ void release_leaving(const ScanArgs &a, const Item &it, int lane) {
    if (it.k >= a.nchunks - 1) return;
    __syncwarp();
    if (lane == 0) flag_release(a.flags + (size_t)it.grp * a.nchunks + it.k, 2);
}

// One pass of the single-warp scan over its work items; false if a wait ran out.
// MODE 0: scan writing y (and hL after the last chunk).
// MODE 1: chunk aggregate (Π Ā, h_end from zero) for chunks 0..K-2, each
//         published for the look-back (publish_pair).
// LBK: the pass runs in a look-back launch (scan_lb_kernel): a MODE 0 pass
//      finds every chunk's start state by look-back (enter_chunk).
template <typename T, int SPT, int NG, bool HAS_Z, bool TMA, int MODE, bool ZOH, bool LBK>
__device__ __forceinline__ bool scan_pass(const Maps &maps, const ScanArgs &a) {
    using S = WTile<T, SPT, NG>;
    constexpr int CPW = S::CPW, NB8 = S::NB8, NQ = SPT / 2;
    constexpr unsigned FULL = 0xffffffffu;
    extern __shared__ __align__(128) unsigned char smem[];
    uint64_t *bar = reinterpret_cast<uint64_t *>(smem + S::off_bar);

    const int lane = threadIdx.x;
    const int c = lane / NG;          // channel within the group
    const int g = lane % NG;          // which SPT states of the channel
    const int D = a.dim, N = a.dstate, L = a.seqlen;
    const int gpb = (D + CPW - 1) / CPW;  // groups per sequence
    const int K = a.nchunks;
    const int kitems = MODE == 0 ? K : K - 1;
    const int items = a.groups * kitems;
    int *ticket = a.tickets + (MODE == 0 ? 0 : 1);
    const bool chained = MODE == 0 && a.chained;

    auto item_of = [&](int t) {
        Item it;
        // Chained items go out chunk-major, so a chunk's predecessor was handed
        // out a full round of groups earlier.
        it.k = t / a.groups;
        it.grp = t % a.groups;
        it.b = it.grp / gpb;
        it.d0 = (it.grp % gpb) * CPW;
        it.t_begin = it.k * a.chunk_len;
        it.t_end = min(L, it.t_begin + a.chunk_len);
        it.ntiles = (it.t_end - it.t_begin + kTT - 1) / kTT;
        return it;
    };
    auto grab = [&]() {
        int t = 0;
        if (lane == 0) t = atomicAdd(ticket, 1);
        return __shfl_sync(FULL, t, 0);
    };

    constexpr uint32_t bc_bytes = S::BC;
    auto stage = [&](int s) { return smem + s * S::BUF; };
    auto issue_loads = [&](const Item &it, int tile, int s) {
        const int t0 = it.t_begin + tile * kTT;
        unsigned char *st = stage(s);
        const uint32_t bytes = (MODE == 0 ? (HAS_Z ? 3u : 2u) : 2u) * S::SEQ + (MODE == 0 ? 2u : 1u) * bc_bytes;
        mbar_arrive_expect_tx(&bar[s], bytes);
#pragma unroll
        for (int j = 0; j < NB8; ++j) {
            tma_load_3d(st + S::off_u + j * S::BLK, &maps.u, &bar[s], t0 + 8 * j, it.d0, it.b);
            tma_load_3d(st + S::off_d + j * S::BLK, &maps.d, &bar[s], t0 + 8 * j, it.d0, it.b);
            if (MODE == 0 && HAS_Z) tma_load_3d(st + S::off_z + j * S::BLK, &maps.z, &bar[s], t0 + 8 * j, it.d0, it.b);
        }
        tma_load_3d(st + S::off_B, &maps.B, &bar[s], 0, t0, it.b);
        if (MODE == 0) tma_load_3d(st + S::off_C, &maps.C, &bar[s], 0, t0, it.b);
    };
    // Plain loads for shapes TMA cannot describe (row pitch not a multiple of 16 B).
    auto generic_loads = [&](const Item &it, int tile, int s) {
        const int t0 = it.t_begin + tile * kTT;
        unsigned char *st = stage(s);
        T *us = reinterpret_cast<T *>(st + S::off_u), *ds = reinterpret_cast<T *>(st + S::off_d);
        T *zs = reinterpret_cast<T *>(st + S::off_z);
        const T *gu = static_cast<const T *>(a.u), *gdl = static_cast<const T *>(a.delta);
        const T *gz = static_cast<const T *>(a.z);
        for (int i = lane; i < CPW * kTT; i += 32) {
            const int tt = i / CPW, cc = i % CPW, dch = it.d0 + cc, t = t0 + tt;
            const bool in = dch < D && t < L;
            const size_t off = ((size_t)it.b * D + dch) * L + t;
            const int si = (tt / 8) * (CPW * 8) + cc * 8 + (tt % 8);
            us[si] = in ? gu[off] : T(0.f);
            ds[si] = in ? gdl[off] : T(0.f);
            if (MODE == 0 && HAS_Z) zs[si] = in ? gz[off] : T(0.f);
        }
        float *Bs = reinterpret_cast<float *>(st + S::off_B), *Cs = reinterpret_cast<float *>(st + S::off_C);
        for (int i = lane; i < kTT * S::NP; i += 32) {
            const int tt = i / S::NP, t = t0 + tt;
            const bool in = t < L;
            const size_t off = ((size_t)it.b * L + t) * S::NP + i % S::NP;
            Bs[i] = in ? a.Bt[off] : 0.f;
            if (MODE == 0) Cs[i] = in ? a.Ct[off] : 0.f;
        }
    };

    int cur = grab();
    if (cur >= items) return true;
    int nxt = grab();
    Item it = item_of(cur);
    int s = 0;                 // stage holding the current tile
    uint32_t phase = 0;        // bit s: parity of stage s's next completion
    int ostage = 0;            // y tile being written
    if (TMA) {
        if (lane == 0) issue_loads(it, 0, 0);
    }
    bool failed = false;

    while (true) {
        // ---- item set-up: this lane's channel, its A row, bias, skip, start state
        const int d = it.d0 + c;
        const bool live = d < D;
        float2 A2[NQ], h[NQ];
#pragma unroll
        for (int q = 0; q < NQ; ++q) {
            float av[2] = {0.f, 0.f};
#pragma unroll
            for (int j = 0; j < 2; ++j) {
                const int n = SPT * g + 2 * q + j;
                if (live && n < N) av[j] = a.A[(size_t)d * N + n] * kLog2e;
            }
            A2[q] = make_float2(av[0], av[1]);
            h[q] = make_float2(0.f, 0.f);
        }
        const float bias = (live && a.bias) ? a.bias[d] : 0.f;
        const float skip = (live && a.Dskip) ? a.Dskip[d] : 0.f;
        if (MODE == 0) {
            const float *src = nullptr;
            bool cg = false;  // read through L2 only: another SM wrote it during this launch
            if (LBK) {
                enter_chunk<SPT, NQ>(a, it, d, live, g, lane, h);
            } else if (it.k == 0) {
                src = a.h0 ? a.h0 + ((size_t)it.b * D + d) * N : nullptr;
            } else if (chained) {
                if (lane == 0 && !wait_flag(a.flags + it.grp, it.k, kFlagLimit))
                    record_error(a.status, 4 /* SSM_ERR_TIMEOUT */);
                __syncwarp();
                (void)flag_acquire(a.flags + it.grp);  // every lane orders its reads after the hand-off
                src = a.carry + ((size_t)it.b * D + d) * N;
                cg = true;
            }
            if (src && live) {
#pragma unroll
                for (int q = 0; q < NQ; ++q) {
                    const int n = SPT * g + 2 * q;
                    float hx = 0.f, hy = 0.f;
                    if (n < N) hx = cg ? __ldcg(src + n) : src[n];
                    if (n + 1 < N) hy = cg ? __ldcg(src + n + 1) : src[n + 1];
                    h[q] = make_float2(hx, hy);
                }
            }
        }
        float dsum = 0.f;  // Σ Δ over the chunk (MODE 1)

        for (int tile = 0; tile < it.ntiles; ++tile) {
            const int t0 = it.t_begin + tile * kTT;
            unsigned char *st = stage(s);
            if (TMA) {
                const bool ok = mbar_wait_bounded(&bar[s], (phase >> s) & 1, kWaitLimit);
                phase ^= 1u << s;
                if (__any_sync(FULL, !ok)) {
                    failed = true;
                    break;
                }
                // Next tile: of this item, else the first tile of the next item.
                if (lane == 0) {
                    fence_proxy_async_smem();
                    if (tile + 1 < it.ntiles) issue_loads(it, tile + 1, s ^ 1);
                    else if (nxt < items) issue_loads(item_of(nxt), 0, s ^ 1);
                }
            } else {
                generic_loads(it, tile, s);
                __syncwarp();
            }

            // The y tile written two tiles ago must have left shared memory.
            if (TMA && MODE == 0 && lane == 0) bulk_wait_read1();
            __syncwarp();

            T *out = reinterpret_cast<T *>(smem + S::off_out + ostage * S::OUT);
            const float *Bf = reinterpret_cast<const float *>(st + S::off_B);
            const float *Cf = reinterpret_cast<const float *>(st + S::off_C);
            const T *u_t = reinterpret_cast<const T *>(st + S::off_u);
            const T *d_t = reinterpret_cast<const T *>(st + S::off_d);
            const T *z_t = reinterpret_cast<const T *>(st + S::off_z);
#pragma unroll 1
            for (int blk = 0; blk < NB8; ++blk) {
                // ---- per-token terms of the channel's 8 tokens.  With two lanes
                // per channel, lane g forms Δ, Δ·u, the gate and D·u·gate of tokens
                // 4g .. 4g+3 and the lanes swap Δ, Δ·u through shared memory.
                const int eo = blk * (CPW * 8) + c * 8;
                constexpr int OWN = 8 / NG;        // tokens whose terms this lane forms
                const int e0 = eo + OWN * g;      // its first token in the staged tile
                const int valid = it.t_end - (t0 + 8 * blk) - OWN * g;  // of its tokens, inside the chunk
                float uf[OWN], df[OWN], zf[OWN];
                if (NG == 1) {
                    IO<T>::load8(u_t + e0, uf);
                    IO<T>::load8(d_t + e0, df);
                    if (MODE == 0 && HAS_Z) IO<T>::load8(z_t + e0, zf);
                } else {
                    const float4 u4 = IO<T>::load4(u_t + e0), d4 = IO<T>::load4(d_t + e0);
                    uf[0] = u4.x; uf[1] = u4.y; uf[2 % OWN] = u4.z; uf[3 % OWN] = u4.w;
                    df[0] = d4.x; df[1] = d4.y; df[2 % OWN] = d4.z; df[3 % OWN] = d4.w;
                    if (MODE == 0 && HAS_Z) {
                        const float4 z4 = IO<T>::load4(z_t + e0);
                        zf[0] = z4.x; zf[1] = z4.y; zf[2 % OWN] = z4.z; zf[3 % OWN] = z4.w;
                    }
                }
                constexpr int OP = OWN / 2;        // own token pairs
                float2 odl[OP], odu[OP];
#pragma unroll
                for (int j = 0; j < OP; ++j) {
                    float2 x = add2(make_float2(df[2 * j], df[2 * j + 1]), make_float2(bias, bias));
                    if (a.delta_softplus) x = make_float2(IO<T>::softplus(x.x), IO<T>::softplus(x.y));
                    if (valid < OWN) {  // Δ = 0 keeps the state: Ā = 1, B̄u = 0
                        if (2 * j >= valid) x.x = 0.f;
                        if (2 * j + 1 >= valid) x.y = 0.f;
                    }
                    odl[j] = x;
                    odu[j] = mul2(x, make_float2(uf[2 * j], uf[2 * j + 1]));
                }
                // Gate and D·u·gate of the lane's own tokens (the ones it outputs).
                float2 gt[OP], dug[OP];
                if (MODE == 0) {
#pragma unroll
                    for (int m = 0; m < OP; ++m) {
                        const float2 uu = make_float2(uf[2 * m], uf[2 * m + 1]);
                        gt[m] = HAS_Z ? gate2<T>(make_float2(zf[2 * m], zf[2 * m + 1])) : make_float2(1.f, 1.f);
                        dug[m] = mul2(mul2(make_float2(skip, skip), uu), gt[m]);
                    }
                }
                float2 dl[4], du[4];  // (Δ, Δ·u) of tokens (2j, 2j+1), as pairs over tokens
                if (NG == 1) {
#pragma unroll
                    for (int j = 0; j < 4; ++j) {
                        dl[j] = odl[j];
                        du[j] = odu[j];
                    }
                } else {
                    // [c][token pair] (Δ0, Δ1, Δu0, Δu1), rows padded to 5 slots against bank conflicts
                    float4 *ex = reinterpret_cast<float4 *>(smem + S::off_ex) + c * 5;
#pragma unroll
                    for (int j = 0; j < OP; ++j)
                        ex[OP * g + j] = make_float4(odl[j].x, odl[j].y, odu[j].x, odu[j].y);
                    __syncwarp();
#pragma unroll
                    for (int j = 0; j < 4; ++j) {
                        const float4 v = ex[j];
                        dl[j] = make_float2(v.x, v.y);
                        du[j] = make_float2(v.z, v.w);
                    }
                }
                // ---- the recurrence over the block's 8 tokens.  Ā and B̄u of
                // token j+1 are formed before the state of token j is updated,
                // and the read-out C·h of token j runs after the update of token
                // j+1, so the chains interleave.  The B row a token needs is
                // loaded one iteration before it is used, the C row likewise.
                constexpr int NR = SPT / 4;  // 16-byte words of a lane's B or C row
                auto load_row = [&](const float *base, int j, float4 *r) {
                    const float *row = base + (8 * blk + j) * S::NP + SPT * g;
#pragma unroll
                    for (int q4 = 0; q4 < NR; ++q4) r[q4] = *reinterpret_cast<const float4 *>(row + 4 * q4);
                };
                float2 an[NQ], bn[NQ];
                auto decay_input = [&](int j, const float4 *br, float2 *ao, float2 *bo) {
                    const float dv = (j & 1) ? dl[j >> 1].y : dl[j >> 1].x;
                    const float uv = (j & 1) ? du[j >> 1].y : du[j >> 1].x;
                    const float2 d2 = make_float2(dv, dv), du2 = make_float2(uv, uv);
#pragma unroll
                    for (int q4 = 0; q4 < NR; ++q4) {
                        const float4 bq = br[q4];
#if SSM_SCAN_SCALAR_X
                        const float2 x0 = make_float2(dv * A2[2 * q4].x, dv * A2[2 * q4].y);
                        const float2 x1 = make_float2(dv * A2[2 * q4 + 1].x, dv * A2[2 * q4 + 1].y);
#else
                        const float2 x0 = mul2(d2, A2[2 * q4]);
                        const float2 x1 = mul2(d2, A2[2 * q4 + 1]);
#endif
                        ao[2 * q4] = make_float2(ex2(x0.x), ex2(x0.y));
                        ao[2 * q4 + 1] = make_float2(ex2(x1.x), ex2(x1.y));
                        bo[2 * q4] = mul2(make_float2(bq.x, bq.y), du2);
                        bo[2 * q4 + 1] = mul2(make_float2(bq.z, bq.w), du2);
                        if (ZOH) {  // B̄ = Δ·φ(ΔA)·B; x0, x1 hold ΔA·log2e
                            const float2 n0 = mul2(x0, make_float2(kLn2, kLn2));
                            const float2 n1 = mul2(x1, make_float2(kLn2, kLn2));
                            bo[2 * q4] = mul2(bo[2 * q4], make_float2(zoh_phi(n0.x, ao[2 * q4].x), zoh_phi(n0.y, ao[2 * q4].y)));
                            bo[2 * q4 + 1] = mul2(bo[2 * q4 + 1], make_float2(zoh_phi(n1.x, ao[2 * q4 + 1].x),
                                                                                   zoh_phi(n1.y, ao[2 * q4 + 1].y)));
                        }
                    }
                };
                float p[8];
                float2 hp[NQ];
                auto readout = [&](int j, const float2 *hs, const float4 *cr) {
                    float2 acc0 = make_float2(0.f, 0.f), acc1 = make_float2(0.f, 0.f);
#pragma unroll
                    for (int q4 = 0; q4 < NR; ++q4) {
                        const float4 cq = cr[q4];
                        if (q4 == 0) {
                            acc0 = mul2(make_float2(cq.x, cq.y), hs[0]);
                            acc1 = mul2(make_float2(cq.z, cq.w), hs[1]);
                        } else {
                            acc0 = fma2(make_float2(cq.x, cq.y), hs[2 * q4], acc0);
                            acc1 = fma2(make_float2(cq.z, cq.w), hs[2 * q4 + 1], acc1);
                        }
                    }
                    const float2 s2 = add2(acc0, acc1);
                    p[j] = s2.x + s2.y;
                };
                float4 Bnx[NR], Cnx[NR];
                {
                    float4 b0[NR];
                    load_row(Bf, 0, b0);
                    load_row(Bf, 1, Bnx);
                    decay_input(0, b0, an, bn);
                }
#pragma unroll
                for (int j = 0; j < 8; ++j) {
                    float2 ac[NQ], bc[NQ];
#pragma unroll
                    for (int q = 0; q < NQ; ++q) {
                        ac[q] = an[q];
                        bc[q] = bn[q];
                    }
                    if (j < 7) {
                        float4 bcur[NR];
#pragma unroll
                        for (int q4 = 0; q4 < NR; ++q4) bcur[q4] = Bnx[q4];
                        if (j < 6) load_row(Bf, j + 2, Bnx);
                        decay_input(j + 1, bcur, an, bn);
                    }
#pragma unroll
                    for (int q = 0; q < NQ; ++q) {
#if SSM_SCAN_SCALAR_H
                        h[q] = make_float2(fmaf(ac[q].x, h[q].x, bc[q].x), fmaf(ac[q].y, h[q].y, bc[q].y));
#else
                        h[q] = fma2(ac[q], h[q], bc[q]);
#endif
                    }
                    if (MODE == 0) {
                        if (j > 0) readout(j - 1, hp, Cnx);
                        load_row(Cf, j, Cnx);
#pragma unroll
                        for (int q = 0; q < NQ; ++q) hp[q] = h[q];
                    } else {
                        dsum += (j & 1) ? dl[j >> 1].y : dl[j >> 1].x;
                    }
                }
                if (MODE == 0) readout(7, hp, Cnx);
                if (MODE == 0) {
                    if (NG == 1) {
                        float y[8];
#pragma unroll
                        for (int m = 0; m < 4; ++m) {
                            const float2 y2 = fma2(make_float2(p[2 * m], p[2 * m + 1]), gt[m], dug[m]);
                            y[2 * m] = y2.x;
                            y[2 * m + 1] = y2.y;
                        }
                        Pack<T>::store8(out + eo, y);
                    } else {
                        // Transposed sum over the two lanes of a channel: lane g
                        // keeps tokens 4g .. 4g+3, the ones whose gate it formed.
                        float y[4];
#pragma unroll
                        for (int i = 0; i < 4; ++i) {
                            const float keep = g ? p[4 + i] : p[i], send = g ? p[i] : p[4 + i];
                            y[i] = keep + __shfl_xor_sync(FULL, send, 1);
                        }
                        const float2 y01 = fma2(make_float2(y[0], y[1]), gt[0], dug[0]);
                        const float2 y23 = fma2(make_float2(y[2], y[3]), gt[OP - 1], dug[OP - 1]);
                        Pack<T>::store4(out + eo + 4 * g, y01, y23);
                    }
                }
                __syncwarp();  // the exchange buffer is rewritten by the next block
            }

            if (MODE == 0) {
                if (TMA) {
                    fence_proxy_async_smem();
                    __syncwarp();
                    if (lane == 0) {
#pragma unroll
                        for (int j = 0; j < NB8; ++j)
                            tma_store_3d(&maps.y, out + j * (CPW * 8), t0 + 8 * j, it.d0, it.b);
                        bulk_commit();
                    }
                } else {
                    __syncwarp();
                    T *gy = static_cast<T *>(a.y);
                    for (int i = lane; i < CPW * kTT; i += 32) {
                        const int tt = i / CPW, cc = i % CPW, dch = it.d0 + cc, t = t0 + tt;
                        if (dch < D && t < it.t_end && in_range(((int64_t)it.b * D + dch) * L + t, 1, (int64_t)a.batch * D * L))
                            gy[((size_t)it.b * D + dch) * L + t] = out[(tt / 8) * (CPW * 8) + cc * 8 + (tt % 8)];
                    }
                }
                ostage ^= 1;
            }
            __syncwarp();  // this tile's B/C rows and stage are free again
            s ^= 1;
            if (LBK && MODE == 0 && tile == 0) release_leaving(a, it, lane);
        }
        if (failed) break;

        // ---- item end: hand the state on, or write the final state / aggregate
        if (MODE == 0) {
            float *dst = nullptr;
            const bool last = it.k == K - 1;
            if (last) dst = a.hL ? a.hL + ((size_t)it.b * D + d) * N : nullptr;
            else if (chained) dst = a.carry + ((size_t)it.b * D + d) * N;
            if (dst && live && in_range(((int64_t)it.b * D + d) * N, N, (int64_t)a.batch * D * N)) {
#pragma unroll
                for (int q = 0; q < NQ; ++q) {
                    const int n = SPT * g + 2 * q;
                    if (n < N) dst[n] = h[q].x;
                    if (n + 1 < N) dst[n + 1] = h[q].y;
                }
            }
            if (chained && !last) {
                // The warp barrier orders every lane's state stores before lane
                // 0's release store; a reader that acquires the flag sees them.
                __syncwarp();
                if (lane == 0) flag_release(a.flags + it.grp, it.k + 1);
            }
        } else {
            publish_pair<SPT, NQ>(a, it, d, live, g, lane, A2, dsum, h);
        }

        cur = nxt;
        if (cur >= items) break;
        nxt = grab();
        it = item_of(cur);
    }
    if (failed) record_error(a.status, 4 /* SSM_ERR_TIMEOUT */);
    if (TMA && MODE == 0 && lane == 0) bulk_wait0();
    return !failed;
}

template <typename T, int SPT, int NG, bool TMA>
__device__ __forceinline__ void scan_init_bars(bool again) {
    using S = WTile<T, SPT, NG>;
    extern __shared__ __align__(128) unsigned char smem[];
    uint64_t *bar = reinterpret_cast<uint64_t *>(smem + S::off_bar);
    if (TMA && threadIdx.x == 0) {
        if (again) {
            mbar_inval(&bar[0]);
            mbar_inval(&bar[1]);
        }
        mbar_init(&bar[0], 1);
        mbar_init(&bar[1], 1);
        fence_mbar_init();
    }
    __syncwarp();
}

// A scan whose chunks are chained or single.
template <typename T, int SPT, int NG, bool HAS_Z, bool TMA, bool ZOH>
__global__ void __launch_bounds__(32, 1)
scan_kernel(const __grid_constant__ Maps maps, const __grid_constant__ ScanArgs a) {
    scan_init_bars<T, SPT, NG, TMA>(false);
    (void)scan_pass<T, SPT, NG, HAS_Z, TMA, 0, ZOH, false>(maps, a);
}

// A scan whose chunks run at once, joined by look-back: every warp runs
// aggregate items until they run out, then main items.  Between the two
// passes the warp's stage barriers start afresh (every load it issued has
// been waited for).
template <typename T, int SPT, int NG, bool HAS_Z, bool TMA, bool ZOH>
__global__ void __launch_bounds__(32, 1)
scan_lb_kernel(const __grid_constant__ Maps maps, const __grid_constant__ ScanArgs a) {
    scan_init_bars<T, SPT, NG, TMA>(false);
    if (!scan_pass<T, SPT, NG, false, TMA, 1, ZOH, true>(maps, a)) return;
    scan_init_bars<T, SPT, NG, TMA>(true);
    (void)scan_pass<T, SPT, NG, HAS_Z, TMA, 0, ZOH, true>(maps, a);
}

// ------------------------------------------------------- warp-specialised passes
// The passes with TMA and two lanes per channel (bf16 I/O, first order), as
// producer / consumer warp pairs.  The producer takes the work items, issues each tile's
// loads and forms every token's terms — Δ = softplus(Δraw + bias), Δ·u, the
// gate and D·u·gate — into shared memory, half a tile (16 tokens) at a time;
// the consumer runs the recurrence and the read-out of the same tile from those
// terms and the staged B and C rows.  The two meet on mbarriers (every wait
// bounded): the consumer's instruction stream loses the terms and their
// exchange, and the producer's loads and MUFU work fill issue slots that the
// consumer's dependency stalls leave idle.  A CTA holds four pairs, consumers
// in warps 0-3 and producers in warps 4-7, so that the SM's four schedulers
// each run two consumers (with 2-warp CTAs the consumers of consecutive CTAs
// landed on the same two schedulers and the pass ran 23 % slower than the
// single-warp kernel instead of 8 % faster).
#ifndef SSM_SCAN_WS
#define SSM_SCAN_WS 1
#endif
// Hand-offs between the two warps of a pair: every lane arrives; waits are
// bounded (mbar_wait_bounded).
constexpr uint32_t kWsArrivals = 32;
__device__ __forceinline__ void ws_arrive(uint64_t *bar) {
    asm volatile("mbarrier.arrive.shared::cta.b64 _, [%0];" ::"r"(smem_u32(bar)) : "memory");
}
__device__ __forceinline__ bool ws_wait(uint64_t *bar, uint32_t parity) {
    return mbar_wait_bounded(bar, parity, kWaitLimit);
}

template <typename T> struct WsTile {
    using Base = WTile<T, 8, 2>;
    static constexpr int CPW = Base::CPW;
    static constexpr int BUF = Base::BUF;                // one TMA stage: u, Δ, z, B, C of a tile
    static constexpr int OUT = Base::OUT;                // one y tile
    static constexpr int off_out = 2 * BUF;              // two y tiles
    static constexpr int TP = 9;                         // float4 per channel row: 8 token pairs + 1 pad
    static constexpr int TRM = CPW * TP * 16;            // one array of a half tile's terms
    static constexpr int off_trm = off_out + 2 * OUT;    // [slot][(Δ, Δ·u) | (gate, D·u·gate)][c][TP] float4
    static constexpr int off_hdr = off_trm + 4 * TRM;    // [slot] int4 (ticket, tile, flags)
    static constexpr int off_bar = off_hdr + 2 * 16;     // 8 mbarriers
    static constexpr int PIPE = al128(off_bar + 8 * 8);  // one producer/consumer pair
    static constexpr int PAIRS = 4;                      // pairs per CTA: warps p and p + 4
    static constexpr int bytes = PAIRS * PIPE;
};

constexpr int kWsFirst = 1, kWsLast = 2, kWsEnd = 4;  // header flags

// One pass of a producer / consumer pair over its work items; false if a wait
// ran out.
// WM = 0: the main pass (y, and hL or the hand-off after each item).
// WM = 1: the aggregate pass — each chunk but the last from a zero state,
//         (Π Ā, h_end) published for the look-back (publish_pair); no
//         read-out, no y, no C.
// WM = 2: the backward's checkpoint pass — the state at every 16-token tile
//         start into a.ckpt; no read-out, no y, no C.
// LBK: the pass runs in a look-back launch (scan_ws_lb_kernel): a main pass
//      finds every chunk's start state by look-back (enter_chunk).
template <typename T, bool HAS_Z, bool ZOH, int WM, bool LBK>
__device__ __forceinline__ bool ws_pass(const Maps &maps, const ScanArgs &a) {
    constexpr bool OUTY = WM == 0, AG = WM == 1, CK = WM == 2;
    using S = WsTile<T>;
    using Wt = WTile<T, 8, 2>;
    constexpr int SPT = 8, CPW = Wt::CPW, NB8 = Wt::NB8, NQ = SPT / 2, NR = SPT / 4, TP = S::TP;
    constexpr unsigned FULL = 0xffffffffu;
    extern __shared__ __align__(128) unsigned char smem_all[];
    // Warps p (consumer) and p + 4 (producer) form pair p, with shared memory of
    // its own; the four consumers sit on the SM's four schedulers, each beside
    // its producer.
    const int warp = threadIdx.x >> 5, lane = threadIdx.x & 31;
    const int role = warp / S::PAIRS;
    unsigned char *smem = smem_all + (warp % S::PAIRS) * S::PIPE;
    uint64_t *bar = reinterpret_cast<uint64_t *>(smem + S::off_bar);
    uint64_t *tma_full = bar, *trm_full = bar + 2, *trm_empty = bar + 4, *stage_empty = bar + 6;
    int4 *hdr = reinterpret_cast<int4 *>(smem + S::off_hdr);
    const int D = a.dim, N = a.dstate, L = a.seqlen, K = a.nchunks;
    const int gpb = (D + CPW - 1) / CPW;
    const int items = a.groups * (AG ? K - 1 : K);
    const bool chained = a.chained;

    auto item_of = [&](int t) {
        Item it;
        it.k = t / a.groups;
        it.grp = t % a.groups;
        it.b = it.grp / gpb;
        it.d0 = (it.grp % gpb) * CPW;
        it.t_begin = it.k * a.chunk_len;
        it.t_end = min(L, it.t_begin + a.chunk_len);
        it.ntiles = (it.t_end - it.t_begin + kTT - 1) / kTT;
        return it;
    };
    auto stage = [&](int s) { return smem + s * S::BUF; };
    auto terms_of = [&](int slot, int which) {
        return reinterpret_cast<float4 *>(smem + S::off_trm + (2 * slot + which) * S::TRM);
    };

    if (role == 1) {
        // ================================================================ producer
        const int c = lane >> 1, hg = lane & 1;  // channel, which 8-token block of a half tile
        auto grab = [&]() {
            int t = 0;
            if (lane == 0) t = atomicAdd(a.tickets + (AG ? 1 : 0), 1);
            return __shfl_sync(FULL, t, 0);
        };
        auto issue = [&](const Item &it, int tile, int s) {  // lane 0
            const int t0 = it.t_begin + tile * kTT;
            unsigned char *st = stage(s);
            mbar_arrive_expect_tx(&tma_full[s], (HAS_Z ? 3u : 2u) * Wt::SEQ + (OUTY ? 2u : 1u) * Wt::BC);
#pragma unroll
            for (int j = 0; j < NB8; ++j) {
                tma_load_3d(st + Wt::off_u + j * Wt::BLK, &maps.u, &tma_full[s], t0 + 8 * j, it.d0, it.b);
                tma_load_3d(st + Wt::off_d + j * Wt::BLK, &maps.d, &tma_full[s], t0 + 8 * j, it.d0, it.b);
                if (HAS_Z) tma_load_3d(st + Wt::off_z + j * Wt::BLK, &maps.z, &tma_full[s], t0 + 8 * j, it.d0, it.b);
            }
            tma_load_3d(st + Wt::off_B, &maps.B, &tma_full[s], 0, t0, it.b);
            if (OUTY) tma_load_3d(st + Wt::off_C, &maps.C, &tma_full[s], 0, t0, it.b);
        };
        bool ok = true;
        // Publishes the end of the work in slot 0 after `tiles` tiles went out.
        auto publish_end = [&](uint32_t tiles) {
            if (tiles > 0) ok = ok && ws_wait(&trm_empty[0], (tiles - 1) & 1);
            if (lane == 0) hdr[0] = make_int4(0, 0, kWsEnd, 0);
            __syncwarp();
            ws_arrive(&trm_full[0]);
        };
        int cur = grab();
        if (cur >= items) {
            publish_end(0);
            return true;
        }
        Item it = item_of(cur);
        int tile = 0;
        if (lane == 0) issue(it, 0, 0);
        int nxt = grab();
        float bias = 0.f, skip = 0.f;
        auto channel_terms = [&]() {
            const int d = it.d0 + c;
            const bool live = d < D;
            bias = (live && a.bias) ? a.bias[d] : 0.f;
            skip = (live && a.Dskip) ? a.Dskip[d] : 0.f;
        };
        channel_terms();
        uint32_t i = 0;  // tiles published so far
        for (;; ++i) {
            const int s = i & 1;
            if (!ws_wait(&tma_full[s], (i >> 1) & 1)) {
                ok = false;
                break;
            }
            const int t0 = it.t_begin + tile * kTT;
            const unsigned char *st = stage(s);
            const T *u_t = reinterpret_cast<const T *>(st + Wt::off_u);
            const T *d_t = reinterpret_cast<const T *>(st + Wt::off_d);
            const T *z_t = reinterpret_cast<const T *>(st + Wt::off_z);
            const int flags = (tile == 0 ? kWsFirst : 0) | (tile + 1 == it.ntiles ? kWsLast : 0);
#pragma unroll 1
            for (int h = 0; h < 2; ++h) {
                if (i > 0 && !ws_wait(&trm_empty[h], (i - 1) & 1)) {
                    ok = false;
                    break;
                }
                const int bb = 2 * h + hg;                      // the lane's 8-token block in the tile
                const int e0 = bb * (CPW * 8) + c * 8;
                const int valid = it.t_end - (t0 + 8 * bb);    // of its tokens, inside the chunk
                float uf[8], df[8], zf[8];
                IO<T>::load8(u_t + e0, uf);
                IO<T>::load8(d_t + e0, df);
                if (HAS_Z) IO<T>::load8(z_t + e0, zf);
                float4 *dd = terms_of(h, 0) + c * TP + 4 * hg;
                float4 *gd = terms_of(h, 1) + c * TP + 4 * hg;
#pragma unroll
                for (int j = 0; j < 4; ++j) {
                    float2 x = add2(make_float2(df[2 * j], df[2 * j + 1]), make_float2(bias, bias));
                    if (a.delta_softplus) x = make_float2(IO<T>::softplus(x.x), IO<T>::softplus(x.y));
                    // Δ = 0 past the chunk's end keeps the state: Ā = 1, B̄u = 0
                    if (2 * j >= valid) x.x = 0.f;
                    if (2 * j + 1 >= valid) x.y = 0.f;
                    const float2 uu = make_float2(uf[2 * j], uf[2 * j + 1]);
                    const float2 du = mul2(x, uu);
                    dd[j] = make_float4(x.x, x.y, du.x, du.y);
                    if (OUTY) {
                        const float2 gt = HAS_Z ? gate2<T>(make_float2(zf[2 * j], zf[2 * j + 1])) : make_float2(1.f, 1.f);
                        const float2 dg = mul2(mul2(make_float2(skip, skip), uu), gt);
                        gd[j] = make_float4(gt.x, gt.y, dg.x, dg.y);
                    }
                }
                if (lane == 0) hdr[h] = make_int4(cur, tile, flags, 0);
                __syncwarp();
                ws_arrive(&trm_full[h]);
            }
            if (!ok) break;
            // The next tile: of this item, else the first tile of the next item.
            int ntile = tile + 1;
            if (ntile == it.ntiles) {
                if (nxt >= items) {
                    publish_end(i + 1);
                    break;
                }
                ntile = 0;
            }
            // Stage s ^ 1 is free once the consumer has finished tile i - 1.
            if (i > 0 && !ws_wait(&stage_empty[s ^ 1], ((i - 1) >> 1) & 1)) {
                ok = false;
                break;
            }
            if (ntile == 0) {
                cur = nxt;
                it = item_of(cur);
                nxt = grab();
                channel_terms();
            }
            if (lane == 0) {
                fence_proxy_async_smem();  // generic reads of the stage before the async-proxy writes
                issue(it, ntile, s ^ 1);
            }
            tile = ntile;
        }
        if (!ok) record_error(a.status, 4 /* SSM_ERR_TIMEOUT */);
        return ok;
    }

    // ==================================================================== consumer
    const int c = lane / 2, g = lane % 2;
    float2 A2[NQ], h[NQ];
    Item it{};
    int d = 0;
    bool live = false;
    int ostage = 0;
    float dsum = 0.f;  // Σ Δ over the item (aggregate pass)
    bool failed = false;
    for (uint32_t i = 0;; ++i) {
        const int s = i & 1;
        if (!ws_wait(&trm_full[0], i & 1)) {
            failed = true;
            break;
        }
        const int4 hd = hdr[0];
        if (hd.z & kWsEnd) break;
        const int tile = hd.y;
        if (hd.z & kWsFirst) {
            // ---- item set-up: this lane's channel, its A row and start state
            it = item_of(hd.x);
            d = it.d0 + c;
            live = d < D;
#pragma unroll
            for (int q = 0; q < NQ; ++q) {
                float av[2] = {0.f, 0.f};
#pragma unroll
                for (int j = 0; j < 2; ++j) {
                    const int n = SPT * g + 2 * q + j;
                    if (live && n < N) av[j] = a.A[(size_t)d * N + n] * kLog2e;
                }
                A2[q] = make_float2(av[0], av[1]);
                h[q] = make_float2(0.f, 0.f);
            }
            dsum = 0.f;
            const float *src = nullptr;
            bool cg = false;  // read through L2 only: another SM wrote it during this launch
            if (AG) {
                // every aggregate starts from a zero state
            } else if (LBK) {
                enter_chunk<SPT, NQ>(a, it, d, live, g, lane, h);
            } else if (it.k == 0) {
                src = a.h0 ? a.h0 + ((size_t)it.b * D + d) * N : nullptr;
            } else if (chained) {
                if (lane == 0 && !wait_flag(a.flags + it.grp, it.k, kFlagLimit))
                    record_error(a.status, 4 /* SSM_ERR_TIMEOUT */);
                __syncwarp();
                (void)flag_acquire(a.flags + it.grp);  // every lane orders its reads after the hand-off
                src = a.carry + ((size_t)it.b * D + d) * N;
                cg = true;
            }
            if (src && live) {
#pragma unroll
                for (int q = 0; q < NQ; ++q) {
                    const int n = SPT * g + 2 * q;
                    float hx = 0.f, hy = 0.f;
                    if (n < N) hx = cg ? __ldcg(src + n) : src[n];
                    if (n + 1 < N) hy = cg ? __ldcg(src + n + 1) : src[n + 1];
                    h[q] = make_float2(hx, hy);
                }
            }
        }
        if (!ws_wait(&tma_full[s], (i >> 1) & 1)) {
            failed = true;
            break;
        }
        // The y tile written two tiles ago must have left shared memory.
        if (OUTY && lane == 0) bulk_wait_read1();
        __syncwarp();
        const int t0 = it.t_begin + tile * kTT;
        const unsigned char *st = stage(s);
        T *out = reinterpret_cast<T *>(smem + S::off_out + ostage * S::OUT);
        const float *Bf = reinterpret_cast<const float *>(st + Wt::off_B);
        const float *Cf = reinterpret_cast<const float *>(st + Wt::off_C);
#pragma unroll 1
        for (int hh = 0; hh < 2; ++hh) {
            if (hh == 1 && !ws_wait(&trm_full[1], i & 1)) {
                failed = true;
                break;
            }
            if (CK) {  // the state entering this 16-token tile is its checkpoint
                const int tk = t0 + 16 * hh;
                if (tk < L && in_range(((int64_t)it.grp * a.ckpt_tiles + tk / 16) * 64, 64,
                                       (int64_t)a.groups * a.ckpt_tiles * 64)) {
                    float4 *ck = reinterpret_cast<float4 *>(a.ckpt) + ((size_t)it.grp * a.ckpt_tiles + tk / 16) * 64;
                    ck[lane] = make_float4(h[0].x, h[0].y, h[1].x, h[1].y);
                    ck[32 + lane] = make_float4(h[2].x, h[2].y, h[3].x, h[3].y);
                }
            }
#pragma unroll 2
            for (int lb = 0; lb < 2; ++lb) {
                const int blk = 2 * hh + lb;
                const float4 *dd = terms_of(hh, 0) + c * TP + 4 * lb;
                float2 dl[4], du[4];  // (Δ, Δ·u) of tokens (2j, 2j+1) of the block
#pragma unroll
                for (int j = 0; j < 4; ++j) {
                    const float4 v = dd[j];
                    dl[j] = make_float2(v.x, v.y);
                    du[j] = make_float2(v.z, v.w);
                }
                // ---- the recurrence over the block's 8 tokens, scheduled as in
                // scan_kernel: Ā and B̄u one token ahead, the read-out one behind.
                auto load_row = [&](const float *base, int j, float4 *r) {
                    const float *row = base + (8 * blk + j) * Wt::NP + SPT * g;
#pragma unroll
                    for (int q4 = 0; q4 < NR; ++q4) r[q4] = *reinterpret_cast<const float4 *>(row + 4 * q4);
                };
                float2 an[NQ], bn[NQ];
                auto decay_input = [&](int j, const float4 *br, float2 *ao, float2 *bo) {
                    const float dv = (j & 1) ? dl[j >> 1].y : dl[j >> 1].x;
                    const float uv = (j & 1) ? du[j >> 1].y : du[j >> 1].x;
                    const float2 d2 = make_float2(dv, dv), du2 = make_float2(uv, uv);
#pragma unroll
                    for (int q4 = 0; q4 < NR; ++q4) {
                        const float4 bq = br[q4];
                        const float2 x0 = mul2(d2, A2[2 * q4]);
                        const float2 x1 = mul2(d2, A2[2 * q4 + 1]);
                        ao[2 * q4] = make_float2(ex2(x0.x), ex2(x0.y));
                        ao[2 * q4 + 1] = make_float2(ex2(x1.x), ex2(x1.y));
                        bo[2 * q4] = mul2(make_float2(bq.x, bq.y), du2);
                        bo[2 * q4 + 1] = mul2(make_float2(bq.z, bq.w), du2);
                        if (ZOH) {  // B̄ = Δ·φ(ΔA)·B; x0, x1 hold ΔA·log2e
                            const float2 n0 = mul2(x0, make_float2(kLn2, kLn2));
                            const float2 n1 = mul2(x1, make_float2(kLn2, kLn2));
                            bo[2 * q4] = mul2(bo[2 * q4], make_float2(zoh_phi(n0.x, ao[2 * q4].x), zoh_phi(n0.y, ao[2 * q4].y)));
                            bo[2 * q4 + 1] = mul2(bo[2 * q4 + 1], make_float2(zoh_phi(n1.x, ao[2 * q4 + 1].x),
                                                                                   zoh_phi(n1.y, ao[2 * q4 + 1].y)));
                        }
                    }
                };
                float p[8];
                float2 hp[NQ];
                auto readout = [&](int j, const float2 *hs, const float4 *cr) {
                    float2 acc = mul2(make_float2(cr[0].x, cr[0].y), hs[0]);
                    acc = fma2(make_float2(cr[0].z, cr[0].w), hs[1], acc);
#pragma unroll
                    for (int q4 = 1; q4 < NR; ++q4) {
                        acc = fma2(make_float2(cr[q4].x, cr[q4].y), hs[2 * q4], acc);
                        acc = fma2(make_float2(cr[q4].z, cr[q4].w), hs[2 * q4 + 1], acc);
                    }
                    p[j] = acc.x + acc.y;
                };
                float4 Bnx[NR], Cnx[NR];
                {
                    float4 b0[NR];
                    load_row(Bf, 0, b0);
                    load_row(Bf, 1, Bnx);
                    decay_input(0, b0, an, bn);
                }
#pragma unroll
                for (int j = 0; j < 8; ++j) {
                    float2 ac[NQ], bc[NQ];
#pragma unroll
                    for (int q = 0; q < NQ; ++q) {
                        ac[q] = an[q];
                        bc[q] = bn[q];
                    }
                    if (j < 7) {
                        float4 bcur[NR];
#pragma unroll
                        for (int q4 = 0; q4 < NR; ++q4) bcur[q4] = Bnx[q4];
                        if (j < 6) load_row(Bf, j + 2, Bnx);
                        decay_input(j + 1, bcur, an, bn);
                    }
#pragma unroll
                    for (int q = 0; q < NQ; ++q) h[q] = fma2(ac[q], h[q], bc[q]);
                    if (AG) dsum += (j & 1) ? dl[j >> 1].y : dl[j >> 1].x;
                    if (OUTY) {
                        if (j > 0) readout(j - 1, hp, Cnx);
                        load_row(Cf, j, Cnx);
#pragma unroll
                        for (int q = 0; q < NQ; ++q) hp[q] = h[q];
                    }
                }
                if (!OUTY) continue;
                readout(7, hp, Cnx);
                // Transposed sum over the two lanes of a channel: lane g keeps
                // tokens 4g .. 4g+3, whose gate terms sit in pairs 2g, 2g+1.
                float y[4];
#pragma unroll
                for (int k2 = 0; k2 < 4; ++k2) {
                    const float keep = g ? p[4 + k2] : p[k2], send = g ? p[k2] : p[4 + k2];
                    y[k2] = keep + __shfl_xor_sync(FULL, send, 1);
                }
                const float4 *gd = terms_of(hh, 1) + c * TP + 4 * lb + 2 * g;
                const float4 g0 = gd[0], g1 = gd[1];
                const float2 y01 = fma2(make_float2(y[0], y[1]), make_float2(g0.x, g0.y), make_float2(g0.z, g0.w));
                const float2 y23 = fma2(make_float2(y[2], y[3]), make_float2(g1.x, g1.y), make_float2(g1.z, g1.w));
                Pack<T>::store4(out + blk * (CPW * 8) + c * 8 + 4 * g, y01, y23);
            }
            __syncwarp();
            ws_arrive(&trm_empty[hh]);  // this half's terms are read
        }
        if (failed) break;
        if (OUTY) {
            fence_proxy_async_smem();
            __syncwarp();
            if (lane == 0) {
#pragma unroll
                for (int j = 0; j < NB8; ++j) tma_store_3d(&maps.y, out + j * (CPW * 8), t0 + 8 * j, it.d0, it.b);
                bulk_commit();
            }
            ostage ^= 1;
        }
        __syncwarp();
        ws_arrive(&stage_empty[s]);  // this tile's B, C rows are read
        if (LBK && OUTY && (hd.z & kWsFirst)) release_leaving(a, it, lane);
        // ---- item end (aggregate pass): publish the chunk's (Π Ā, h_end from zero)
        if (AG && (hd.z & kWsLast)) publish_pair<SPT, NQ>(a, it, d, live, g, lane, A2, dsum, h);
        if (!AG && (hd.z & kWsLast)) {
            // ---- item end: hand the state on, or write the final state
            float *dst = nullptr;
            const bool last = it.k == K - 1;
            if (last) dst = (!CK && a.hL) ? a.hL + ((size_t)it.b * D + d) * N : nullptr;
            else if (chained) dst = a.carry + ((size_t)it.b * D + d) * N;
            if (dst && live && in_range(((int64_t)it.b * D + d) * N, N, (int64_t)a.batch * D * N)) {
#pragma unroll
                for (int q = 0; q < NQ; ++q) {
                    const int n = SPT * g + 2 * q;
                    if (n < N) dst[n] = h[q].x;
                    if (n + 1 < N) dst[n + 1] = h[q].y;
                }
            }
            if (chained && !last) {
                // The warp barrier orders every lane's state stores before lane
                // 0's release store; a reader that acquires the flag sees them.
                __syncwarp();
                if (lane == 0) flag_release(a.flags + it.grp, it.k + 1);
            }
        }
    }
    if (failed) record_error(a.status, 4 /* SSM_ERR_TIMEOUT */);
    if (OUTY && lane == 0) bulk_wait0();
    return !failed;
}

// Each pair's eight barriers, set up by its consumer's lane 0 (again: after a
// pass, with nothing pending on them).
template <typename T>
__device__ __forceinline__ void ws_init_bars(bool again) {
    using S = WsTile<T>;
    extern __shared__ __align__(128) unsigned char smem_all[];
    const int warp = threadIdx.x >> 5;
    uint64_t *bar = reinterpret_cast<uint64_t *>(smem_all + (warp % S::PAIRS) * S::PIPE + S::off_bar);
    if (warp / S::PAIRS == 0 && (threadIdx.x & 31) == 0) {
#pragma unroll
        for (int i = 0; i < 8; ++i) {
            if (again) mbar_inval(&bar[i]);
            mbar_init(&bar[i], i < 2 ? 1 : kWsArrivals);
        }
        fence_mbar_init();
    }
}

template <typename T, bool HAS_Z, bool ZOH, int WM>
__global__ void __launch_bounds__(256, 2)
scan_ws_kernel(const __grid_constant__ Maps maps, const __grid_constant__ ScanArgs a) {
    ws_init_bars<T>(false);
    __syncthreads();
    (void)ws_pass<T, HAS_Z, ZOH, WM, false>(maps, a);
}

// The look-back launch of the warp-specialised scan: every pair runs
// aggregate items until they run out, then main items.  Between the passes
// the pair's two warps meet on a named barrier (one per pair; barrier 0 is
// the block's), and unless a wait of either ran out, the consumer sets the
// pair's barriers up afresh before they meet again.  The warps tell each
// other how their pass ended in the second header slot, which the consumer
// never reads during a pass.
template <typename T, bool HAS_Z, bool ZOH>
__global__ void __launch_bounds__(256, 2)
scan_ws_lb_kernel(const __grid_constant__ Maps maps, const __grid_constant__ ScanArgs a) {
    using S = WsTile<T>;
    extern __shared__ __align__(128) unsigned char smem_all[];
    ws_init_bars<T>(false);
    __syncthreads();
    const bool ok = ws_pass<T, false, ZOH, 1, true>(maps, a);
    const int warp = threadIdx.x >> 5, pair = warp % S::PAIRS, role = warp / S::PAIRS;
    volatile int *ended = reinterpret_cast<volatile int *>(smem_all + pair * S::PIPE + S::off_hdr + 16);
    // immediate barrier ids, so that the block reserves five barriers, not all sixteen
    static_assert(S::PAIRS == 4, "one named barrier per pair");
    auto pair_sync = [&]() {
        switch (pair) {
            case 0: asm volatile("bar.sync 1, 64;" ::: "memory"); break;
            case 1: asm volatile("bar.sync 2, 64;" ::: "memory"); break;
            case 2: asm volatile("bar.sync 3, 64;" ::: "memory"); break;
            default: asm volatile("bar.sync 4, 64;" ::: "memory"); break;
        }
    };
    if ((threadIdx.x & 31) == 0) ended[role] = ok ? 1 : 0;
    pair_sync();
    const bool both = ended[0] && ended[1];  // read before the next pass rewrites the slot
    if (!both) return;
    ws_init_bars<T>(true);
    pair_sync();
    (void)ws_pass<T, HAS_Z, ZOH, 0, true>(maps, a);
}

// B and C, [b][N][L] in the I/O type, widened once per launch to fp32
// token-major rows [b][L][np] (zero for n >= N), the layout every warp's TMA
// loads take per tile.  One block per (32 tokens, sequence), staged through
// shared memory so reads and writes are both coalesced.
template <typename T>
__global__ void __launch_bounds__(256) widen_bc_kernel(const ScanArgs a) {
    __shared__ float tile[2][16][33];
    const int b = blockIdx.y, t0 = blockIdx.x * 32, N = a.dstate, L = a.seqlen, np = a.np;
    const T *B = static_cast<const T *>(a.B) + (size_t)b * N * L;
    const T *C = static_cast<const T *>(a.C) + (size_t)b * N * L;
    for (int i = threadIdx.x; i < 2 * 16 * 32; i += blockDim.x) {
        const int m = i / (16 * 32), n = (i / 32) % 16, tt = i % 32, t = t0 + tt;
        float v = 0.f;
        if (n < N && t < L) v = IO<T>::to_f((m ? C : B)[(size_t)n * L + t]);
        tile[m][n][tt] = v;
    }
    __syncthreads();
    for (int i = threadIdx.x; i < 2 * 32 * np; i += blockDim.x) {
        const int m = i / (32 * np), tt = (i / np) % 32, n = i % np, t = t0 + tt;
        if (t < L && in_range(((int64_t)b * L + t) * np + n, 1, (int64_t)a.batch * L * np))
            (m ? a.Ct : a.Bt)[((size_t)b * L + t) * np + n] = tile[m][n][tt];
    }
}

// ------------------------------------------------------------------ host side

TensorMapEncodeFn tensor_map_encoder() {
    static TensorMapEncodeFn fn = nullptr;
    static std::once_flag once;
    std::call_once(once, [] {
        void *p = nullptr;
        cudaDriverEntryPointQueryResult q;
        if (cudaGetDriverEntryPointByVersion("cuTensorMapEncodeTiled", &p, 12000, cudaEnableDefault, &q) ==
                cudaSuccess &&
            q == cudaDriverEntryPointSuccess)
            fn = reinterpret_cast<TensorMapEncodeFn>(p);
    });
    return fn;
}

namespace {

using EncodeFn = TensorMapEncodeFn;
EncodeFn encode_fn() { return tensor_map_encoder(); }

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

// Lanes per channel and states per lane for a state size N.
struct Split {
    int spt, ng;
};
Split split_for(int64_t dstate) {
    if (dstate <= 4) return {4, 1};
    if (dstate <= 8) return {8, 1};
    return SSM_SCAN_N16_LANES == 1 ? Split{16, 1} : Split{8, 2};
}

// LB: the look-back kernel, else the plain one.
template <typename T, int SPT, int NG, bool HAS_Z, bool TMA, bool LB, bool ZOH>
cudaError_t launch_one(const Maps &maps, const ScanArgs &a, int items, cudaStream_t st) {
    using S = WTile<T, SPT, NG>;
    auto kern = LB ? scan_lb_kernel<T, SPT, NG, HAS_Z, TMA, ZOH> : scan_kernel<T, SPT, NG, HAS_Z, TMA, ZOH>;
    static PerDevice resident;  // resident warps per SM for this instantiation
    int per_sm = 0;
    cudaError_t e = resident.get(
        [&](int *v) {
            cudaError_t r = cudaFuncSetAttribute(kern, cudaFuncAttributeMaxDynamicSharedMemorySize, S::bytes);
            if (r != cudaSuccess) return r;
            int n = 0;
            r = cudaOccupancyMaxActiveBlocksPerMultiprocessor(&n, kern, 32, S::bytes);
            *v = std::max(1, std::min(n, kWarpsPerSM));
            return r;
        },
        &per_sm);
    if (e != cudaSuccess) return e;
    const int grid = std::max(1, std::min(items, sm_count() * per_sm));
    kern<<<grid, 32, S::bytes, st>>>(maps, a);
    return cudaGetLastError();
}

// WM < 0: the look-back kernel; else scan_ws_kernel's pass WM.
template <typename T, bool HAS_Z, bool ZOH, int WM = 0>
cudaError_t launch_ws(const Maps &maps, const ScanArgs &a, int items, cudaStream_t st) {
    using S = WsTile<T>;
    auto kern = WM < 0 ? scan_ws_lb_kernel<T, HAS_Z, ZOH> : scan_ws_kernel<T, HAS_Z, ZOH, (WM < 0 ? 0 : WM)>;
    static PerDevice resident;  // resident CTAs (four consumer warps each) per SM
    int per_sm = 0;
    cudaError_t e = resident.get(
        [&](int *v) {
            cudaError_t r = cudaFuncSetAttribute(kern, cudaFuncAttributeMaxDynamicSharedMemorySize, S::bytes);
            if (r != cudaSuccess) return r;
            int n = 0;
            r = cudaOccupancyMaxActiveBlocksPerMultiprocessor(&n, kern, 32 * 2 * S::PAIRS, S::bytes);
            *v = std::max(1, std::min(n, kWarpsPerSM / S::PAIRS));
            return r;
        },
        &per_sm);
    if (e != cudaSuccess) return e;
    const int pairs = std::max(1, std::min(items, sm_count() * per_sm * S::PAIRS));
    kern<<<(pairs + S::PAIRS - 1) / S::PAIRS, 32 * 2 * S::PAIRS, S::bytes, st>>>(maps, a);
    return cudaGetLastError();
}

template <typename T, int SPT, int NG, bool HAS_Z, bool TMA, bool ZOH>
cudaError_t launch_all(const Maps &maps, const ScanArgs &a, cudaStream_t st) {
    cudaError_t e;
    widen_bc_kernel<T><<<dim3((a.seqlen + 31) / 32, a.batch), 256, 0, st>>>(a);
    e = cudaGetLastError();
    if (e != cudaSuccess) return e;
    // bf16 I/O, first order: the warp-specialised form keeps eight consumer
    // warps per SM within 128 registers and 26 KB of shared memory per CTA.
    constexpr bool ws = SSM_SCAN_WS && TMA && SPT == 8 && NG == 2 && sizeof(T) == 2 && !ZOH;
    // Chunks that run at once (K > 1, not chained) carry their start states by
    // look-back inside the one launch, which holds every aggregate item of
    // chunks 0 .. K-2 and then every main item.
    const bool lb = a.nchunks > 1 && !a.chained;
    const int items = a.groups * a.nchunks;
    if constexpr (ws) return lb ? launch_ws<T, HAS_Z, ZOH, -1>(maps, a, items, st) : launch_ws<T, HAS_Z, ZOH, 0>(maps, a, items, st);
    return lb ? launch_one<T, SPT, NG, HAS_Z, TMA, true, ZOH>(maps, a, items, st)
              : launch_one<T, SPT, NG, HAS_Z, TMA, false, ZOH>(maps, a, items, st);
}

template <typename T, int SPT, int NG, bool ZOH>
cudaError_t dispatch_z_tma_d(const Maps &maps, const ScanArgs &a, bool tma, cudaStream_t st) {
    const bool z = a.z != nullptr;
    if (tma)
        return z ? launch_all<T, SPT, NG, true, true, ZOH>(maps, a, st)
                 : launch_all<T, SPT, NG, false, true, ZOH>(maps, a, st);
    return z ? launch_all<T, SPT, NG, true, false, ZOH>(maps, a, st)
             : launch_all<T, SPT, NG, false, false, ZOH>(maps, a, st);
}
template <typename T, int SPT, int NG>
cudaError_t dispatch_z_tma(const Maps &maps, const ScanArgs &a, bool tma, cudaStream_t st) {
    return a.zoh ? dispatch_z_tma_d<T, SPT, NG, true>(maps, a, tma, st)
                 : dispatch_z_tma_d<T, SPT, NG, false>(maps, a, tma, st);
}

template <typename T>
cudaError_t dispatch_split(const Maps &maps, const ScanArgs &a, Split sp, bool tma, cudaStream_t st) {
    if (sp.spt == 4) return dispatch_z_tma<T, 4, 1>(maps, a, tma, st);
    if (sp.spt == 8 && sp.ng == 1) return dispatch_z_tma<T, 8, 1>(maps, a, tma, st);
#if SSM_SCAN_N16_LANES == 1
    return dispatch_z_tma<T, 16, 1>(maps, a, tma, st);
#else
    return dispatch_z_tma<T, 8, 2>(maps, a, tma, st);
#endif
}

}  // namespace

// Look-back terms of the chunk-length model below, µs.
constexpr double kLookBackPerChunk = 1.1, kLookBackFixed = 8.0;

int scan_groups(int64_t dstate) { return dstate <= 4 ? 1 : (dstate <= 8 ? 2 : 4); }

ScanPlan scan_plan(int64_t batch, int64_t dim, int64_t dstate, int64_t seqlen, int64_t requested) {
    ScanPlan p;
    const Split sp = split_for(dstate);
    p.np = sp.spt * sp.ng;
    p.cpw = 32 / sp.ng;
    p.groups = batch * ((dim + p.cpw - 1) / p.cpw);
    const int64_t resident = (int64_t)kSMs * kWarpsPerSM;
    const int64_t Lr = ((seqlen + 63) / 64) * 64;
    // Chained when the groups alone fill the resident warps (a look-back split
    // would add aggregate items for parallelism the GPU does not need).
    p.chained = p.groups * 4 >= resident * 3;
    if (p.chained) {
        p.chunk_len = requested > 0 ? std::min<int64_t>(requested, Lr) : std::min<int64_t>(kDefaultChunk, Lr);
    } else if (requested > 0) {
        p.chunk_len = std::min<int64_t>(requested, Lr);
    } else {
        // Look-back: pick the chunk length with the least modelled time, in µs,
        //   throughput:   all token-items of both kinds (an aggregate item
        //                 costs ≈0.7 of a main one) spread over the resident
        //                 warps, ≈0.1 µs per token per warp when they are all busy;
        //   critical path: one chunk walked by one warp as both kinds of item,
        //                 ≈0.07 µs per token when few warps share an SM;
        //   look-back:    per chunk and in all (kLookBackPerChunk, kLookBackFixed).
        // The constants are fits to B300 timings of the 2 × 1536 × 16 × 2048 and
        // 1 × 5120 × 16 × 131072 layers over chunk lengths 64 .. 8192.  A single
        // chunk (no aggregate items) is one of the candidates.
        double best = 1e300;
        p.chunk_len = Lr;
        for (int64_t len = Lr; len >= 64; len -= 64) {
            const int64_t K = (seqlen + len - 1) / len;
            if (K > 64) break;
            const double items = (double)p.groups * ((double)K + 0.7 * (double)(K - 1)) * (double)len;
            const double t = items * 0.1 / (double)resident + 1.7 * (double)len * 0.07 +
                             (K > 1 ? kLookBackPerChunk * (double)K + kLookBackFixed : 0.0);
            if (t < best * 0.999) {
                best = t;
                p.chunk_len = len;
            }
        }
    }
    p.nchunks = (seqlen + p.chunk_len - 1) / p.chunk_len;
    if (p.nchunks == 1) p.chained = false;
    return p;
}

bool scan_ckpt_supported(const ScanPlan &plan, int64_t dstate, int64_t seqlen, bool bf16, int zoh) {
    const Split sp = split_for(dstate);
    return SSM_SCAN_WS && bf16 && zoh == 0 && sp.spt == 8 && sp.ng == 2 && plan.chained && (seqlen * 2) % 16 == 0;
}

cudaError_t scan_ckpt_launch(const ScanArgs &a, cudaStream_t st) {
    using T = __nv_bfloat16;
    const int cpw = 16;
    Maps maps;
    memset(&maps, 0, sizeof(maps));
    const CUtensorMapDataType dt = CU_TENSOR_MAP_DATA_TYPE_BFLOAT16;
    const bool ok = make_map(&maps.u, dt, 2, a.u, a.seqlen, a.dim, a.batch, 8, cpw) &&
                    make_map(&maps.d, dt, 2, a.delta, a.seqlen, a.dim, a.batch, 8, cpw) &&
                    make_map(&maps.B, CU_TENSOR_MAP_DATA_TYPE_FLOAT32, 4, a.Bt, a.np, a.seqlen, a.batch, a.np, kTT);
    if (!ok || !a.ckpt || !a.chained) return cudaErrorInvalidValue;
    widen_bc_kernel<T><<<dim3((a.seqlen + 31) / 32, a.batch), 256, 0, st>>>(a);
    const cudaError_t e = cudaGetLastError();
    if (e != cudaSuccess) return e;
    return launch_ws<T, false, false, 2>(maps, a, a.groups * a.nchunks, st);
}

cudaError_t scan_launch(const ScanArgs &a, bool bf16, cudaStream_t st) {
    const Split sp = split_for(a.dstate);
    const int cpw = 32 / sp.ng;
    const size_t es = bf16 ? 2 : 4;
    // TMA needs a row pitch that is a multiple of 16 bytes.
    const bool tma = ((size_t)a.seqlen * es) % 16 == 0;
    Maps maps;
    memset(&maps, 0, sizeof(maps));
    if (tma) {
        const CUtensorMapDataType dt = bf16 ? CU_TENSOR_MAP_DATA_TYPE_BFLOAT16 : CU_TENSOR_MAP_DATA_TYPE_FLOAT32;
        bool ok = make_map(&maps.u, dt, es, a.u, a.seqlen, a.dim, a.batch, 8, cpw) &&
                  make_map(&maps.d, dt, es, a.delta, a.seqlen, a.dim, a.batch, 8, cpw) &&
                  make_map(&maps.B, CU_TENSOR_MAP_DATA_TYPE_FLOAT32, 4, a.Bt, a.np, a.seqlen, a.batch, a.np, kTT) &&
                  make_map(&maps.C, CU_TENSOR_MAP_DATA_TYPE_FLOAT32, 4, a.Ct, a.np, a.seqlen, a.batch, a.np, kTT) &&
                  make_map(&maps.y, dt, es, a.y, a.seqlen, a.dim, a.batch, 8, cpw);
        if (ok && a.z) ok = make_map(&maps.z, dt, es, a.z, a.seqlen, a.dim, a.batch, 8, cpw);
        if (!ok) return cudaErrorInvalidValue;
    }
    return bf16 ? dispatch_split<__nv_bfloat16>(maps, a, sp, tma, st) : dispatch_split<float>(maps, a, sp, tma, st);
}

SSM_DEBUG_WORD_READER(debug_word_fwd)

}  // namespace ssm
