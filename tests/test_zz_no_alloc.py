"""ssm_scan_fwd_noalloc, the scan entry point for callers that cannot allocate
device memory (its chunk scratch is a fixed array inside the library).

It must give what ssm_scan_fwd gives with a caller-allocated workspace, call
after call: the shared scratch keeps the previous call's contents, so two calls
in a row on different inputs are checked.  This file is collected last so that a
run stopping at its first failure has already run every other test.
"""

import pytest
import torch

from mamba_selective_scan_02_b300 import api, capi
from ssm_testutil import assert_close

pytestmark = pytest.mark.gpu


def _inputs(seed, b=2, D=96, N=16, L=1000, dtype=torch.bfloat16):
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


def _with_workspace(inp, chunk_len):
    y, hL = api.scan_fwd(inp["u"], inp["delta"], inp["A"], inp["B"], inp["C"], inp["Dskip"], inp["z"],
                         inp["bias"], inp["h0"], chunk_len=chunk_len)
    torch.cuda.synchronize()
    return y, hL


def _no_alloc(inp, chunk_len):
    y = torch.empty_like(inp["u"])
    hL = torch.empty_like(inp["h0"])
    p = _params(inp, y, hL, chunk_len)
    st = torch.cuda.current_stream().cuda_stream
    capi.check(capi.ssm_scan_fwd_noalloc(p, st), "ssm_scan_fwd_noalloc")
    torch.cuda.synchronize()
    return y, hL


@pytest.mark.parametrize("chunk_len", [128, 0])
def test_no_alloc_matches_workspace_entry_point_twice(chunk_len):
    for call, seed in enumerate((11, 12)):   # two calls in a row, different inputs
        inp = _inputs(seed)
        y_ref, h_ref = _with_workspace(inp, chunk_len)
        y, hL = _no_alloc(inp, chunk_len)
        assert_close(y.double().cpu().numpy(), y_ref.double().cpu().numpy(), torch.bfloat16,
                     f"no-alloc y, call {call + 1}")
        assert_close(hL.cpu().numpy(), h_ref.cpu().numpy(), torch.bfloat16, f"no-alloc hL, call {call + 1}")


def test_no_alloc_rejects_sizes_beyond_its_scratch():
    inp = _inputs(13, b=1, D=8, N=16, L=64)
    y = torch.empty_like(inp["u"])
    p = _params(inp, y, None, 0)
    p.batch, p.dim, p.seqlen, p.chunk_len = 64, 8192, 1 << 20, 64   # scratch need far above the maximum
    assert capi.ssm_scan_workspace_size(p) > capi.SSM_NOALLOC_SCRATCH_BYTES
    st = torch.cuda.current_stream().cuda_stream
    assert capi.ssm_scan_fwd_noalloc(p, st) == capi.SSM_ERR_UNSUPPORTED
