// api.cu — the C ABI of libssmscan (declared in include/ssm_scan.h):
// argument validation, workspace layout, launches on the caller's stream and
// status reporting.  No entry point allocates memory.
#include <stdint.h>
#include <string.h>

#include "../../include/ssm_scan.h"
#include "ssm_internal.h"

namespace {

constexpr size_t kHeader = 256;  // status word + padding

inline size_t align256(size_t x) { return (x + 255) & ~size_t(255); }
inline bool aligned16(const void *p) { return (reinterpret_cast<uintptr_t>(p) & 15) == 0; }
inline bool aligned4(const void *p) { return (reinterpret_cast<uintptr_t>(p) & 3) == 0; }

struct Layout {
    ssm::ScanPlan plan;
    size_t flags_off, agg_off, carry_off, bt_off, ct_off, zero_bytes, total;
};

bool scan_sizes_ok(const ssm_scan_params *p) {
    if (!p) return false;
    if (p->batch < 1 || p->dim < 1 || p->seqlen < 1 || p->dstate < 1) return false;
    if (p->batch > 65535 || p->dim > (1 << 30) || p->seqlen > INT32_MAX) return false;
    if (p->chunk_len < 0 || (p->chunk_len > 0 && p->chunk_len % 64 != 0)) return false;
    return true;
}

// Workspace: a 256-byte header (status word, two work counters), then
//   chained:  one int flag per channel group, and one b × D × N fp32 state;
//   look-back: one int flag per (channel group, chunk), per-chunk aggregates
//             [b][D][K-1][N] (float2) and carried states [b][D][K][N] (fp32);
// then, always, B and C widened to fp32 token-major rows [b][L][np].
// The header and the flags are cleared before every launch.
Layout scan_layout(const ssm_scan_params *p) {
    Layout l;
    l.plan = ssm::scan_plan(p->batch, p->dim, p->dstate, p->seqlen, p->chunk_len);
    const size_t bdn = (size_t)p->batch * p->dim * p->dstate;
    l.flags_off = l.agg_off = l.carry_off = kHeader;
    l.zero_bytes = kHeader;
    l.total = kHeader;
    if (l.plan.chained) {
        const size_t flag_bytes = align256((size_t)l.plan.groups * sizeof(int));
        l.carry_off = kHeader + flag_bytes;
        l.zero_bytes = kHeader + flag_bytes;
        l.total = l.carry_off + align256(bdn * sizeof(float));
    } else if (l.plan.nchunks > 1) {
        const size_t flag_bytes = align256((size_t)l.plan.groups * (size_t)l.plan.nchunks * sizeof(int));
        const size_t agg_bytes = align256(bdn * (size_t)(l.plan.nchunks - 1) * sizeof(float2));
        l.agg_off = kHeader + flag_bytes;
        l.zero_bytes = l.agg_off;
        l.carry_off = l.agg_off + agg_bytes;
        l.total = l.carry_off + align256(bdn * (size_t)l.plan.nchunks * sizeof(float));
    }
    const size_t bt_bytes = align256((size_t)p->batch * p->seqlen * l.plan.np * sizeof(float));
    l.bt_off = l.total;
    l.ct_off = l.bt_off + bt_bytes;
    l.total = l.ct_off + bt_bytes;
    return l;
}

bool overlaps(const void *a, size_t na, const void *b, size_t nb) {
    if (!a || !b) return false;
    const uintptr_t x = reinterpret_cast<uintptr_t>(a), y = reinterpret_cast<uintptr_t>(b);
    return x < y + nb && y < x + na;
}

bool bwd_sizes_ok(const ssm_scan_bwd_params *p) {
    if (!p) return false;
    if (p->batch < 1 || p->dim < 1 || p->seqlen < 1 || p->dstate < 1) return false;
    if (p->batch > 65535 || p->dim > (1 << 30) || p->seqlen > INT32_MAX / 2) return false;
    if (p->chunk_len < 0 || (p->chunk_len > 0 && p->chunk_len % ssm::kBwdTile != 0)) return false;
    return true;
}

struct BwdLayout {
    int64_t groups, ntiles, chunk_len, nchunks;
    size_t flags_fwd, flags_rev, carry_fwd, carry_rev, ckpt, zero_bytes, total;
    // the checkpoint pass on the forward scan kernel (when scan_ckpt_supported)
    bool scan_ckpt;
    ssm::ScanPlan plan;
    size_t scan_flags, scan_carry, scan_bt, scan_ct;
    size_t own_total;  // the workspace the backward's own checkpoint pass needs
};

// Backward workspace: the 256-byte header (status word, two work counters of
// the backward passes, two of the forward kernel's checkpoint launch), one int
// flag per channel group for each pass (and for the checkpoint launch), the two
// b × D × N fp32 hand-off states, the state at every tile start,
// [group][tile][256] fp32, and for the checkpoint launch its own hand-off
// state and B, C widened to fp32.  The header and the flags are cleared before
// every call.
BwdLayout bwd_layout(const ssm_scan_bwd_params *p) {
    BwdLayout l;
    const int cpw = ssm::bwd_cpw(p->dstate);
    l.groups = p->batch * ((p->dim + cpw - 1) / cpw);
    l.ntiles = (p->seqlen + ssm::kBwdTile - 1) / ssm::kBwdTile;
    l.chunk_len = p->chunk_len > 0 ? p->chunk_len : ssm::kBwdChunk;
    l.nchunks = (p->seqlen + l.chunk_len - 1) / l.chunk_len;
    l.plan = ssm::scan_plan(p->batch, p->dim, p->dstate, p->seqlen, 0);
    l.scan_ckpt = ssm::scan_ckpt_supported(l.plan, p->dstate, p->seqlen, p->io_dtype == SSM_BF16, p->zoh) &&
                  l.plan.groups == l.groups;
    const size_t flag_bytes = align256((size_t)l.groups * sizeof(int));
    const size_t bdn = align256((size_t)p->batch * p->dim * p->dstate * sizeof(float));
    l.flags_fwd = kHeader;
    l.flags_rev = l.flags_fwd + flag_bytes;
    l.zero_bytes = l.flags_rev + flag_bytes;
    l.carry_fwd = l.zero_bytes;
    l.carry_rev = l.carry_fwd + bdn;
    l.ckpt = l.carry_rev + bdn;
    l.total = l.ckpt + (size_t)l.groups * l.ntiles * 256 * sizeof(float);
    l.own_total = l.total;
    l.scan_flags = l.scan_carry = l.scan_bt = l.scan_ct = l.total;
    if (l.scan_ckpt) {  // after the backward's own regions, cleared separately
        const size_t bt = align256((size_t)p->batch * p->seqlen * l.plan.np * sizeof(float));
        l.scan_flags = l.total;
        l.scan_carry = l.scan_flags + flag_bytes;
        l.scan_bt = l.scan_carry + bdn;
        l.scan_ct = l.scan_bt + bt;
        l.total = l.scan_ct + bt;
    }
    return l;
}

}  // namespace

extern "C" {

size_t ssm_scan_bwd_workspace_size(const ssm_scan_bwd_params *p) {
    if (!bwd_sizes_ok(p)) return 0;
    return bwd_layout(p).total;
}

ssm_status ssm_scan_bwd(const ssm_scan_bwd_params *p, ssm_stream_t stream) {
    if (!bwd_sizes_ok(p)) return SSM_ERR_INVALID_ARG;
    if (p->io_dtype != SSM_F32 && p->io_dtype != SSM_BF16) return SSM_ERR_INVALID_ARG;
    if (p->dstate > SSM_MAX_DSTATE) return SSM_ERR_UNSUPPORTED;
    if (p->zoh != 0 && p->zoh != 1) return SSM_ERR_INVALID_ARG;
    if (p->delta_softplus != 0 && p->delta_softplus != 1) return SSM_ERR_INVALID_ARG;
    if (!p->u || !p->delta || !p->B || !p->C || !p->A || !p->dy || !p->du || !p->ddelta || !p->dB || !p->dC ||
        !p->dA || !p->workspace)
        return SSM_ERR_INVALID_ARG;
    const size_t es = p->io_dtype == SSM_BF16 ? 2 : 4;
    const void *aio[] = {p->u, p->delta, p->z, p->B, p->C, p->dy, p->du, p->ddelta, p->dz};
    for (const void *q : aio)
        if (q && (reinterpret_cast<uintptr_t>(q) % es) != 0) return SSM_ERR_INVALID_ARG;
    const void *a4[] = {p->A, p->Dskip, p->delta_bias, p->h0, p->dhL, p->dB, p->dC, p->dA, p->dDskip,
                        p->ddelta_bias, p->dh0};
    for (const void *q : a4)
        if (q && !aligned4(q)) return SSM_ERR_INVALID_ARG;
    if (!aligned16(p->workspace)) return SSM_ERR_INVALID_ARG;
    const size_t seq = (size_t)p->batch * p->dim * p->seqlen * es;
    const size_t bc = (size_t)p->batch * p->dstate * p->seqlen * es;
    const size_t bcf = (size_t)p->batch * p->dstate * p->seqlen * 4;
    const void *ins[] = {p->u, p->delta, p->z, p->dy};
    const void *outs[] = {p->du, p->ddelta, p->dz};
    for (const void *o : outs) {
        for (const void *i : ins)
            if (overlaps(o, seq, i, seq)) return SSM_ERR_INVALID_ARG;
        if (overlaps(o, seq, p->B, bc) || overlaps(o, seq, p->C, bc)) return SSM_ERR_INVALID_ARG;
    }
    if (overlaps(p->du, seq, p->ddelta, seq) || overlaps(p->du, seq, p->dz, seq) ||
        overlaps(p->ddelta, seq, p->dz, seq) || overlaps(p->dB, bcf, p->dC, bcf) || overlaps(p->dB, bcf, p->B, bc) ||
        overlaps(p->dC, bcf, p->C, bc))
        return SSM_ERR_INVALID_ARG;
    const BwdLayout l = bwd_layout(p);
    // A workspace without room for the forward kernel's checkpoint launch still
    // runs, with the backward's own checkpoint pass.
    if (p->workspace_bytes < l.own_total) return SSM_ERR_INVALID_ARG;
    const bool scan_ckpt = l.scan_ckpt && p->workspace_bytes >= l.total;
    if (l.groups * l.nchunks > INT32_MAX / 2 || l.groups * l.ntiles > INT32_MAX / 2) return SSM_ERR_UNSUPPORTED;

    cudaStream_t st = reinterpret_cast<cudaStream_t>(stream);
    unsigned char *ws = static_cast<unsigned char *>(p->workspace);
    if (cudaMemsetAsync(ws, 0, l.zero_bytes, st) != cudaSuccess) return SSM_ERR_CUDA;
    const size_t dn = (size_t)p->dim * p->dstate * sizeof(float);
    if (cudaMemsetAsync(p->dB, 0, bcf, st) != cudaSuccess || cudaMemsetAsync(p->dC, 0, bcf, st) != cudaSuccess ||
        cudaMemsetAsync(p->dA, 0, dn, st) != cudaSuccess)
        return SSM_ERR_CUDA;
    if (p->dDskip && cudaMemsetAsync(p->dDskip, 0, p->dim * sizeof(float), st) != cudaSuccess) return SSM_ERR_CUDA;
    if (p->ddelta_bias && cudaMemsetAsync(p->ddelta_bias, 0, p->dim * sizeof(float), st) != cudaSuccess)
        return SSM_ERR_CUDA;

    ssm::BwdArgs a;
    a.batch = (int)p->batch;
    a.dim = (int)p->dim;
    a.dstate = (int)p->dstate;
    a.seqlen = (int)p->seqlen;
    a.u = p->u;
    a.delta = p->delta;
    a.z = p->z;
    a.B = p->B;
    a.C = p->C;
    a.dy = p->dy;
    a.A = p->A;
    a.Dskip = p->Dskip;
    a.bias = p->delta_bias;
    a.h0 = p->h0;
    a.dhL = p->dhL;
    a.delta_softplus = p->delta_softplus;
    a.zoh = p->zoh;
    a.du = p->du;
    a.ddelta = p->ddelta;
    a.dz = p->z ? p->dz : nullptr;
    a.dB = p->dB;
    a.dC = p->dC;
    a.dA = p->dA;
    a.dDskip = p->dDskip;
    a.dbias = p->ddelta_bias;
    a.dh0 = p->dh0;
    a.status = reinterpret_cast<int *>(ws);
    a.tickets = reinterpret_cast<int *>(ws) + 1;
    a.flags_fwd = reinterpret_cast<int *>(ws + l.flags_fwd);
    a.flags_rev = reinterpret_cast<int *>(ws + l.flags_rev);
    a.carry_fwd = reinterpret_cast<float *>(ws + l.carry_fwd);
    a.carry_rev = reinterpret_cast<float *>(ws + l.carry_rev);
    a.ckpt = reinterpret_cast<float *>(ws + l.ckpt);
    a.chunk_len = (int)l.chunk_len;
    a.nchunks = (int)l.nchunks;
    a.groups = (int)l.groups;
    a.ntiles = (int)l.ntiles;
    a.ckpt_ready = 0;
    if (scan_ckpt && aligned16(p->u) && aligned16(p->delta)) {
        // The checkpoint pass as the forward scan's warp-specialised kernel.
        if (cudaMemsetAsync(ws + l.scan_flags, 0, (size_t)l.groups * sizeof(int), st) != cudaSuccess)
            return SSM_ERR_CUDA;
        ssm::ScanArgs f;
        memset(&f, 0, sizeof(f));
        f.batch = a.batch;
        f.dim = a.dim;
        f.dstate = a.dstate;
        f.seqlen = a.seqlen;
        f.u = p->u;
        f.delta = p->delta;
        f.B = p->B;
        f.C = p->C;
        f.A = p->A;
        f.bias = p->delta_bias;
        f.delta_softplus = p->delta_softplus;
        f.h0 = p->h0;
        f.status = a.status;
        f.tickets = reinterpret_cast<int *>(ws) + 4;
        f.flags = reinterpret_cast<int *>(ws + l.scan_flags);
        f.carry = reinterpret_cast<float *>(ws + l.scan_carry);
        f.chunk_len = (int)l.plan.chunk_len;
        f.nchunks = (int)l.plan.nchunks;
        f.groups = (int)l.plan.groups;
        f.chained = 1;
        f.Bt = reinterpret_cast<float *>(ws + l.scan_bt);
        f.Ct = reinterpret_cast<float *>(ws + l.scan_ct);
        f.np = l.plan.np;
        f.ckpt = a.ckpt;
        f.ckpt_tiles = a.ntiles;
        if (ssm::scan_ckpt_launch(f, st) != cudaSuccess) return SSM_ERR_CUDA;
        a.ckpt_ready = 1;
    }
    return ssm::bwd_launch(a, p->io_dtype == SSM_BF16, st) == cudaSuccess ? SSM_OK : SSM_ERR_CUDA;
}

size_t ssm_scan_workspace_size(const ssm_scan_params *p) {
    if (!scan_sizes_ok(p)) return 0;
    return scan_layout(p).total;
}

ssm_status ssm_scan_plan(const ssm_scan_params *p, int64_t out[4]) {
    if (!scan_sizes_ok(p) || !out) return SSM_ERR_INVALID_ARG;
    const ssm::ScanPlan plan = scan_layout(p).plan;
    out[0] = plan.chunk_len;
    out[1] = plan.nchunks;
    out[2] = plan.chained ? 1 : 0;
    out[3] = plan.groups;
    return SSM_OK;
}

ssm_status ssm_scan_fwd(const ssm_scan_params *p, ssm_stream_t stream) {
    if (!scan_sizes_ok(p)) return SSM_ERR_INVALID_ARG;
    if (p->io_dtype != SSM_F32 && p->io_dtype != SSM_BF16) return SSM_ERR_INVALID_ARG;
    if (p->dstate > SSM_MAX_DSTATE) return SSM_ERR_UNSUPPORTED;
    if (p->zoh != 0 && p->zoh != 1) return SSM_ERR_INVALID_ARG;
    if (p->delta_softplus != 0 && p->delta_softplus != 1) return SSM_ERR_INVALID_ARG;
    if (!p->u || !p->delta || !p->B || !p->C || !p->A || !p->y || !p->workspace) return SSM_ERR_INVALID_ARG;
    const void *a16[] = {p->u, p->delta, p->z, p->B, p->C, p->y, p->h0, p->hL, p->workspace};
    for (const void *q : a16)
        if (q && !aligned16(q)) return SSM_ERR_INVALID_ARG;
    const void *a4[] = {p->A, p->Dskip, p->delta_bias};
    for (const void *q : a4)
        if (q && !aligned4(q)) return SSM_ERR_INVALID_ARG;
    const size_t es = p->io_dtype == SSM_BF16 ? 2 : 4;
    const size_t seq = (size_t)p->batch * p->dim * p->seqlen * es;
    const size_t bc = (size_t)p->batch * p->dstate * p->seqlen * es;
    if (overlaps(p->y, seq, p->u, seq) || overlaps(p->y, seq, p->delta, seq) || overlaps(p->y, seq, p->z, seq) ||
        overlaps(p->y, seq, p->B, bc) || overlaps(p->y, seq, p->C, bc))
        return SSM_ERR_INVALID_ARG;
    const Layout l = scan_layout(p);
    if (p->workspace_bytes < l.total) return SSM_ERR_INVALID_ARG;
    if (l.plan.groups * l.plan.nchunks > INT32_MAX / 2) return SSM_ERR_UNSUPPORTED;

    cudaStream_t st = reinterpret_cast<cudaStream_t>(stream);
    unsigned char *ws = static_cast<unsigned char *>(p->workspace);
    if (cudaMemsetAsync(ws, 0, l.zero_bytes, st) != cudaSuccess) return SSM_ERR_CUDA;

    ssm::ScanArgs a;
    a.batch = (int)p->batch;
    a.dim = (int)p->dim;
    a.dstate = (int)p->dstate;
    a.seqlen = (int)p->seqlen;
    a.u = p->u;
    a.delta = p->delta;
    a.z = p->z;
    a.B = p->B;
    a.C = p->C;
    a.A = p->A;
    a.Dskip = p->Dskip;
    a.bias = p->delta_bias;
    a.delta_softplus = p->delta_softplus;
    a.zoh = p->zoh;
    a.h0 = p->h0;
    a.y = p->y;
    a.hL = p->hL;
    a.status = reinterpret_cast<int *>(ws);
    a.tickets = reinterpret_cast<int *>(ws) + 1;
    a.flags = reinterpret_cast<int *>(ws + l.flags_off);
    a.agg = reinterpret_cast<float2 *>(ws + l.agg_off);
    a.carry = reinterpret_cast<float *>(ws + l.carry_off);
    a.chunk_len = (int)l.plan.chunk_len;
    a.nchunks = (int)l.plan.nchunks;
    a.groups = (int)l.plan.groups;
    a.chained = l.plan.chained ? 1 : 0;
    a.Bt = reinterpret_cast<float *>(ws + l.bt_off);
    a.Ct = reinterpret_cast<float *>(ws + l.ct_off);
    a.np = l.plan.np;
    a.ckpt = nullptr;
    a.ckpt_tiles = 0;
    return ssm::scan_launch(a, p->io_dtype == SSM_BF16, st) == cudaSuccess ? SSM_OK : SSM_ERR_CUDA;
}

ssm_status ssm_state_update(const ssm_step_params *p, ssm_stream_t stream) {
    if (!p) return SSM_ERR_INVALID_ARG;
    if (p->batch < 1 || p->dim < 1 || p->dstate < 1) return SSM_ERR_INVALID_ARG;
    if (p->batch * p->dim > (int64_t(1) << 31) / 4) return SSM_ERR_UNSUPPORTED;
    if (p->io_dtype != SSM_F32 && p->io_dtype != SSM_BF16) return SSM_ERR_INVALID_ARG;
    if (p->dstate > SSM_MAX_DSTATE) return SSM_ERR_UNSUPPORTED;
    if (p->zoh != 0 && p->zoh != 1) return SSM_ERR_INVALID_ARG;
    if (p->delta_softplus != 0 && p->delta_softplus != 1) return SSM_ERR_INVALID_ARG;
    if (!p->state || !p->u || !p->delta || !p->B || !p->C || !p->A || !p->y) return SSM_ERR_INVALID_ARG;
    // The decode kernel reads every input with scalar loads, so element
    // alignment is enough; the state is accessed 16 bytes at a time only when
    // its base is 16-byte aligned and N is a multiple of 4.
    const size_t es = p->io_dtype == SSM_BF16 ? 2 : 4;
    const void *aio[] = {p->u, p->delta, p->z, p->B, p->C, p->y};
    for (const void *q : aio)
        if (q && (reinterpret_cast<uintptr_t>(q) % es) != 0) return SSM_ERR_INVALID_ARG;
    const void *a4[] = {p->state, p->A, p->Dskip, p->delta_bias};
    for (const void *q : a4)
        if (q && !aligned4(q)) return SSM_ERR_INVALID_ARG;
    const size_t nch = (size_t)p->batch * p->dim;
    if (overlaps(p->y, nch * es, p->state, nch * p->dstate * 4) || overlaps(p->y, nch * es, p->u, nch * es) ||
        overlaps(p->y, nch * es, p->delta, nch * es) || overlaps(p->y, nch * es, p->z, nch * es))
        return SSM_ERR_INVALID_ARG;

    ssm::StepArgs a;
    a.batch = (int)p->batch;
    a.dim = (int)p->dim;
    a.dstate = (int)p->dstate;
    a.state = p->state;
    a.u = p->u;
    a.delta = p->delta;
    a.z = p->z;
    a.B = p->B;
    a.C = p->C;
    a.A = p->A;
    a.Dskip = p->Dskip;
    a.bias = p->delta_bias;
    a.delta_softplus = p->delta_softplus;
    a.zoh = p->zoh;
    a.y = p->y;
    return ssm::step_launch(a, p->io_dtype == SSM_BF16, reinterpret_cast<cudaStream_t>(stream)) == cudaSuccess
               ? SSM_OK
               : SSM_ERR_CUDA;
}

namespace {
// SSD workspace: a 256-byte header (the work counter), a flag per chain, then
// one fp32 P × N state per chain.
struct SsdLayout {
    size_t flags, carry, total;
};
SsdLayout ssd_layout(const ssm_ssd_params *p) {
    const size_t chains = (size_t)p->batch * p->nheads;
    SsdLayout l;
    l.flags = 256;
    l.carry = align256(l.flags + chains * sizeof(int));
    l.total = l.carry + chains * (size_t)p->headdim * p->dstate * sizeof(float);
    return l;
}
bool ssd_sizes_ok(const ssm_ssd_params *p) {
    return p->batch >= 1 && p->seqlen >= 1 && p->nheads >= 1 && p->headdim >= 1 && p->dstate >= 1 &&
           p->batch * p->nheads <= INT32_MAX / 2 && p->seqlen <= INT32_MAX / 2 && p->headdim <= 4096 &&
           p->dstate <= 4096;
}
}  // namespace

size_t ssm_ssd_workspace_size(const ssm_ssd_params *p) {
    if (!p || !ssd_sizes_ok(p)) return 0;
    return ssd_layout(p).total;
}

ssm_status ssm_ssd_fwd(const ssm_ssd_params *p, ssm_stream_t stream) {
    if (!p) return SSM_ERR_INVALID_ARG;
    if (p->batch < 1 || p->seqlen < 1 || p->nheads < 1 || p->headdim < 1 || p->dstate < 1) return SSM_ERR_INVALID_ARG;
    if (p->io_dtype != SSM_F32 && p->io_dtype != SSM_BF16) return SSM_ERR_INVALID_ARG;
    if (p->dt_softplus != 0 && p->dt_softplus != 1) return SSM_ERR_INVALID_ARG;
    if (!p->x || !p->dt || !p->A || !p->B || !p->C || !p->y) return SSM_ERR_INVALID_ARG;
    if (p->io_dtype != SSM_BF16 || !ssm::ssd_supported(p->headdim, p->dstate)) return SSM_ERR_UNSUPPORTED;
    if (p->batch * p->nheads > INT32_MAX / 2 || p->seqlen > INT32_MAX / 2) return SSM_ERR_UNSUPPORTED;
    const void *a16[] = {p->x, p->B, p->C, p->y};
    for (const void *q : a16)
        if (!aligned16(q)) return SSM_ERR_INVALID_ARG;
    if (reinterpret_cast<uintptr_t>(p->dt) % 2 != 0) return SSM_ERR_INVALID_ARG;
    const void *a4[] = {p->A, p->Dskip, p->dt_bias, p->h0, p->hL, p->status};
    for (const void *q : a4)
        if (q && !aligned4(q)) return SSM_ERR_INVALID_ARG;
    const size_t seq = (size_t)p->batch * p->seqlen * p->nheads * p->headdim * 2;
    const size_t bc = (size_t)p->batch * p->seqlen * p->dstate * 2;
    if (overlaps(p->y, seq, p->x, seq) || overlaps(p->y, seq, p->B, bc) || overlaps(p->y, seq, p->C, bc) ||
        overlaps(p->y, seq, p->dt, (size_t)p->batch * p->seqlen * p->nheads * 2))
        return SSM_ERR_INVALID_ARG;
    ssm::SsdArgs a;
    a.batch = (int)p->batch;
    a.seqlen = (int)p->seqlen;
    a.nheads = (int)p->nheads;
    a.x = p->x;
    a.dt = p->dt;
    a.B = p->B;
    a.C = p->C;
    a.A = p->A;
    a.Dskip = p->Dskip;
    a.dt_bias = p->dt_bias;
    a.dt_softplus = p->dt_softplus;
    a.h0 = p->h0;
    a.y = p->y;
    a.hL = p->hL;
    a.status = p->status;
    const ssm::SsdPlan plan = ssm::ssd_plan(p->batch, p->seqlen, p->nheads, p->workspace != nullptr);
    a.seg_chunks = plan.seg_chunks;
    a.ticket = nullptr;
    a.flags = nullptr;
    a.carry = nullptr;
    const cudaStream_t st = reinterpret_cast<cudaStream_t>(stream);
    if (p->workspace) {
        const SsdLayout l = ssd_layout(p);
        if (p->workspace_bytes < l.total || (reinterpret_cast<uintptr_t>(p->workspace) & 255) != 0)
            return SSM_ERR_INVALID_ARG;
        unsigned char *ws = static_cast<unsigned char *>(p->workspace);
        const size_t hdr = l.carry;   // counter and flags
        if (overlaps(ws, l.total, p->y, seq) || overlaps(ws, l.total, p->x, seq)) return SSM_ERR_INVALID_ARG;
        if (cudaMemsetAsync(ws, 0, hdr, st) != cudaSuccess) return SSM_ERR_CUDA;
        a.ticket = reinterpret_cast<int *>(ws);
        a.flags = reinterpret_cast<int *>(ws + l.flags);
        a.carry = reinterpret_cast<float *>(ws + l.carry);
    }
    return ssm::ssd_launch(a, plan.nseg, st) == cudaSuccess ? SSM_OK : SSM_ERR_CUDA;
}

ssm_status ssm_conv1d_fwd(const ssm_conv_params *p, ssm_stream_t stream) {
    if (!p) return SSM_ERR_INVALID_ARG;
    if (p->batch < 1 || p->dim < 1 || p->seqlen < 1) return SSM_ERR_INVALID_ARG;
    if (p->width < 1) return SSM_ERR_INVALID_ARG;
    if (p->width > SSM_MAX_CONV_WIDTH) return SSM_ERR_UNSUPPORTED;
    if (p->io_dtype != SSM_F32 && p->io_dtype != SSM_BF16) return SSM_ERR_INVALID_ARG;
    if (p->silu != 0 && p->silu != 1) return SSM_ERR_INVALID_ARG;
    if (!p->x || !p->weight || !p->u) return SSM_ERR_INVALID_ARG;
    if (p->batch > (int64_t(1) << 40) / p->dim || p->batch * p->dim > (int64_t(1) << 40) / p->seqlen)
        return SSM_ERR_UNSUPPORTED;
    const size_t es = p->io_dtype == SSM_BF16 ? 2 : 4;
    const void *aio[] = {p->x, p->u, p->state_in, p->state_out};
    for (const void *q : aio)
        if (q && (reinterpret_cast<uintptr_t>(q) % es) != 0) return SSM_ERR_INVALID_ARG;
    if (!aligned4(p->weight) || (p->bias && !aligned4(p->bias))) return SSM_ERR_INVALID_ARG;
    const size_t seq = (size_t)p->batch * p->dim * p->seqlen * es;
    const size_t st = (size_t)p->batch * p->dim * (p->width - 1) * es;
    if (overlaps(p->u, seq, p->x, seq)) return SSM_ERR_INVALID_ARG;
    if (st > 0 && (overlaps(p->state_out, st, p->state_in, st) || overlaps(p->state_out, st, p->x, seq) ||
                   overlaps(p->state_out, st, p->u, seq)))
        return SSM_ERR_INVALID_ARG;
    ssm::ConvArgs a;
    a.batch = p->batch;
    a.dim = p->dim;
    a.seqlen = p->seqlen;
    a.width = (int)p->width;
    a.x = p->x;
    a.w = p->weight;
    a.bias = p->bias;
    a.state_in = p->width > 1 ? p->state_in : nullptr;
    a.u = p->u;
    a.state_out = p->width > 1 ? p->state_out : nullptr;
    a.silu = p->silu;
    return ssm::conv_launch(a, p->io_dtype == SSM_BF16, reinterpret_cast<cudaStream_t>(stream)) == cudaSuccess
               ? SSM_OK
               : SSM_ERR_CUDA;
}

ssm_status ssm_conv1d_step(const ssm_conv_step_params *p, ssm_stream_t stream) {
    if (!p) return SSM_ERR_INVALID_ARG;
    if (p->batch < 1 || p->dim < 1 || p->width < 1) return SSM_ERR_INVALID_ARG;
    if (p->width > SSM_MAX_CONV_WIDTH) return SSM_ERR_UNSUPPORTED;
    if (p->io_dtype != SSM_F32 && p->io_dtype != SSM_BF16) return SSM_ERR_INVALID_ARG;
    if (p->silu != 0 && p->silu != 1) return SSM_ERR_INVALID_ARG;
    if (!p->x || !p->weight || !p->u || (p->width > 1 && !p->state)) return SSM_ERR_INVALID_ARG;
    if (p->batch > (int64_t(1) << 40) / p->dim) return SSM_ERR_UNSUPPORTED;
    const size_t es = p->io_dtype == SSM_BF16 ? 2 : 4;
    const void *aio[] = {p->x, p->u, p->state};
    for (const void *q : aio)
        if (q && (reinterpret_cast<uintptr_t>(q) % es) != 0) return SSM_ERR_INVALID_ARG;
    if (!aligned4(p->weight) || (p->bias && !aligned4(p->bias))) return SSM_ERR_INVALID_ARG;
    const size_t nch = (size_t)p->batch * p->dim;
    const size_t st = nch * (p->width - 1) * es;
    if (overlaps(p->u, nch * es, p->x, nch * es) || (st > 0 && overlaps(p->u, nch * es, p->state, st)))
        return SSM_ERR_INVALID_ARG;
    ssm::ConvStepArgs a;
    a.batch = p->batch;
    a.dim = p->dim;
    a.width = (int)p->width;
    a.state = p->width > 1 ? p->state : nullptr;
    a.x = p->x;
    a.w = p->weight;
    a.bias = p->bias;
    a.u = p->u;
    a.silu = p->silu;
    return ssm::conv_step_launch(a, p->io_dtype == SSM_BF16, reinterpret_cast<cudaStream_t>(stream)) ==
                   cudaSuccess
               ? SSM_OK
               : SSM_ERR_CUDA;
}

ssm_status ssm_workspace_status(const void *workspace, ssm_stream_t stream) {
    if (!workspace) return SSM_ERR_INVALID_ARG;
    cudaStream_t st = reinterpret_cast<cudaStream_t>(stream);
    if (cudaStreamSynchronize(st) != cudaSuccess) return SSM_ERR_CUDA;
    int code = 0;
    if (cudaMemcpy(&code, workspace, sizeof(int), cudaMemcpyDeviceToHost) != cudaSuccess) return SSM_ERR_CUDA;
    return code == 0 ? SSM_OK : (code == SSM_ERR_TIMEOUT ? SSM_ERR_TIMEOUT : SSM_ERR_CUDA);
}

const char *ssm_status_string(ssm_status s) {
    switch (s) {
        case SSM_OK: return "ok";
        case SSM_ERR_INVALID_ARG: return "invalid argument";
        case SSM_ERR_UNSUPPORTED: return "unsupported by this build";
        case SSM_ERR_CUDA: return "CUDA error";
        case SSM_ERR_TIMEOUT: return "device-side wait timed out";
        case SSM_ERR_BOUNDS: return "debug build: a store outside its buffer was skipped";
    }
    return "unknown status";
}

ssm_status ssm_debug_status(int reset) {
#ifdef SSM_DEBUG
    if (cudaDeviceSynchronize() != cudaSuccess) return SSM_ERR_CUDA;
    const int words[] = {ssm::debug_word_conv(reset != 0), ssm::debug_word_step(reset != 0),
                         ssm::debug_word_bwd(reset != 0), ssm::debug_word_fwd(reset != 0),
                         ssm::debug_word_ssd(reset != 0)};
    ssm_status st = SSM_OK;
    for (int w : words) {
        if (w < 0) return SSM_ERR_CUDA;
        if (w != 0 && st == SSM_OK) st = SSM_ERR_BOUNDS;
    }
    return st;
#else
    (void)reset;
    return SSM_ERR_UNSUPPORTED;
#endif
}

ssm_status ssm_bench_mufu_ex2(float *sink, int blocks, int iters, ssm_stream_t stream) {
    if (!sink || blocks < 1 || iters < 1 || !aligned4(sink)) return SSM_ERR_INVALID_ARG;
    return ssm::mufu_ex2_launch(sink, blocks, iters, reinterpret_cast<cudaStream_t>(stream)) == cudaSuccess
               ? SSM_OK
               : SSM_ERR_CUDA;
}

ssm_status ssm_selftest_flag_wait(void *workspace, size_t workspace_bytes, int polls, ssm_stream_t stream) {
    if (!workspace || workspace_bytes < kHeader || !aligned16(workspace) || polls < 1 || polls > (1 << 24))
        return SSM_ERR_INVALID_ARG;
    cudaStream_t st = reinterpret_cast<cudaStream_t>(stream);
    if (cudaMemsetAsync(workspace, 0, kHeader, st) != cudaSuccess) return SSM_ERR_CUDA;
    int *hdr = static_cast<int *>(workspace);
    // the status word at offset 0; the never-set flag past the work counters
    return ssm::flag_wait_selftest_launch(hdr, hdr + 16, polls, st) == cudaSuccess ? SSM_OK : SSM_ERR_CUDA;
}

const char *ssm_version(void) { return "libssmscan sm_103a"; }

}  // extern "C"
