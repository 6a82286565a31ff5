"""ssm_scan_fwd_noalloc, the scan entry point for callers that cannot allocate
device memory (its chunk scratch is a fixed array inside the library).

It runs the same kernels as ssm_scan_fwd on the same inputs, so its output must
equal ssm_scan_fwd's bit for bit, call after call.  The shared scratch keeps
the previous call's contents — chained plans keep their hand-off flags and
states there, look-back plans their chunk flags, pairs and carried states —
so each case runs several calls in a row on different inputs: two chained
layers, then a look-back one, then a chained one again.  One of them is also checked against
the oracle.  This file is collected last so that a run stopping at its first
failure has already run every other test.
"""

import numpy as np
import pytest
import torch

from mamba_selective_scan_02_b300 import api, capi
from ssm_testutil import assert_close, oracle_scan_sampled, sample_channels

pytestmark = pytest.mark.gpu

# A layer whose default plan is chained (enough channel groups to fill the GPU)
# and one whose plan is look-back (few groups, the sequence cut into chunks).
CHAINED = dict(b=4, D=5000, N=16, L=512)
LOOK_BACK = dict(b=2, D=96, N=16, L=1000)


def _inputs(seed, b, D, N, L, dtype=torch.bfloat16):
    g = torch.Generator().manual_seed(seed)
    rn = lambda *s, std=1.0: (torch.randn(*s, generator=g) * std).to(dtype).cuda()
    bias = torch.log(torch.expm1(torch.empty(D).uniform_(1e-3, 1e-1, generator=g))).float()
    return dict(u=rn(b, D, L), delta=rn(b, D, L, std=0.5), z=rn(b, D, L), B=rn(b, N, L), C=rn(b, N, L),
                A=-torch.arange(1, N + 1, dtype=torch.float32).repeat(D, 1).cuda(),
                Dskip=torch.randn(D, generator=g).cuda(), bias=bias.cuda(),
                h0=(torch.randn(b, D, N, generator=g) * 0.5).cuda())


def _params(inp, y, hL, chunk_len, workspace=None):
    return api.scan_params(inp["u"], inp["delta"], inp["A"], inp["B"], inp["C"], inp["Dskip"], inp["z"],
                           inp["bias"], inp["h0"], y=y, hL=hL, chunk_len=chunk_len, workspace=workspace)


def _plan(inp, chunk_len):
    y = torch.empty_like(inp["u"])
    return capi.ssm_scan_plan(_params(inp, y, None, chunk_len))


def _with_workspace(inp, chunk_len):
    y, hL = api.scan_fwd(inp["u"], inp["delta"], inp["A"], inp["B"], inp["C"], inp["Dskip"], inp["z"],
                         inp["bias"], inp["h0"], chunk_len=chunk_len)
    torch.cuda.synchronize()
    return y, hL


def _no_alloc(inp, chunk_len):
    y = torch.empty_like(inp["u"])
    hL = torch.empty_like(inp["h0"])
    p = _params(inp, y, hL, chunk_len)
    assert capi.ssm_scan_workspace_size(p) <= capi.SSM_NOALLOC_SCRATCH_BYTES
    st = torch.cuda.current_stream().cuda_stream
    capi.check(capi.ssm_scan_fwd_noalloc(p, st), "ssm_scan_fwd_noalloc")
    torch.cuda.synchronize()
    return y, hL


def _check_equal(inp, chunk_len, what):
    y_ref, h_ref = _with_workspace(inp, chunk_len)
    y, hL = _no_alloc(inp, chunk_len)
    assert torch.equal(y, y_ref), f"{what}: y differs from ssm_scan_fwd"
    assert torch.equal(hL, h_ref), f"{what}: hL differs from ssm_scan_fwd"
    return y, hL


@pytest.mark.parametrize("chunk_len", [0, 64])
def test_no_alloc_equals_workspace_entry_point_call_after_call(chunk_len):
    calls = [(CHAINED, 21), (CHAINED, 22), (LOOK_BACK, 23), (CHAINED, 24)]
    kinds = []
    for n, (shape, seed) in enumerate(calls):
        inp = _inputs(seed, **shape)
        kinds.append(_plan(inp, chunk_len)["chained"])
        _check_equal(inp, chunk_len, f"call {n + 1} ({shape}, seed {seed})")
    # The sequence really alternates between the two kinds of plan.
    assert kinds[0] and kinds[1] and kinds[3], kinds
    assert not kinds[2], kinds


def test_no_alloc_chained_against_the_oracle():
    inp = _inputs(25, **CHAINED)
    assert _plan(inp, 64)["chained"]
    y, hL = _no_alloc(inp, 64)
    picks = sample_channels(CHAINED["b"], CHAINED["D"], 12, seed=5)
    want_y, want_h = oracle_scan_sampled(inp, picks)
    got_y = np.stack([y[bi, di].double().cpu().numpy() for bi, di in picks])
    got_h = np.stack([hL[bi, di].double().cpu().numpy() for bi, di in picks])
    assert_close(got_y, want_y, torch.bfloat16, "no-alloc chained y")
    assert_close(got_h, want_h, torch.bfloat16, "no-alloc chained hL")


def test_no_alloc_rejects_sizes_beyond_its_scratch():
    inp = _inputs(13, b=1, D=8, N=16, L=64)
    y = torch.empty_like(inp["u"])
    p = _params(inp, y, None, 0)
    p.batch, p.dim, p.seqlen, p.chunk_len = 64, 8192, 1 << 20, 64   # scratch need far above the maximum
    assert capi.ssm_scan_workspace_size(p) > capi.SSM_NOALLOC_SCRATCH_BYTES
    st = torch.cuda.current_stream().cuda_stream
    assert capi.ssm_scan_fwd_noalloc(p, st) == capi.SSM_ERR_UNSUPPORTED
