"""Guard bands on every output the kernels write.

compute-sanitizer is closed on this machine, so these stand in for its bounds
checks: each output is the front of a larger buffer whose tail holds a fixed
bit pattern, and after the call the tail must be bit for bit what it was.  The
outputs themselves must equal those of the same call into ordinary tensors
(bit for bit where the kernel is deterministic; the backward's fp32 atomic sums
are compared to a tight tolerance instead).  Shapes pick each kernel variant
the dispatch chooses between: the decode step's general, 16-state and streamed
kernels, the convolution's per-row and streamed kernels, its decode step for
D a multiple of 8 and otherwise.  The SSD kernel's y and hL have the same
check in test_ssd_parity.py; the forward scan's in test_scan_parity.py.
"""

import numpy as np
import pytest
import torch

from mamba_selective_scan_02_b300 import api

pytestmark = pytest.mark.gpu

PAD = 4096   # elements of guard band after each output


def poisoned(shape, dtype):
    """(tensor at the front of a larger buffer, its guard band, the band's original bits)."""
    n = int(np.prod(shape))
    buf = torch.empty(n + PAD, dtype=dtype, device="cuda")
    bits = buf.view(torch.int16 if dtype == torch.bfloat16 else torch.int32)
    bits.fill_(0x5A3C)
    return buf[:n].view(shape), buf[n:], buf[n:].clone()


def band_intact(band, ref, what):
    assert torch.equal(band, ref), f"{what}: the guard band past the output was written"


def _rn(g, *shape, std=1.0, dtype=torch.float32):
    return (torch.randn(*shape, generator=g) * std).to(dtype).cuda()


# ---------------------------------------------------------------- decode step

@pytest.mark.parametrize("b,D,N,dtype", [
    (3, 37, 5, torch.float32),       # general kernel, ragged state rows
    (2, 96, 16, torch.bfloat16),     # 16-state kernel (D not a multiple of 128)
    (2, 256, 16, torch.bfloat16),    # streamed 128-channel tiles
])
def test_state_update_guard_bands(b, D, N, dtype):
    g = torch.Generator().manual_seed(b * 1000 + D)
    u, dl, z = _rn(g, b, D, dtype=dtype), _rn(g, b, D, std=0.5, dtype=dtype), _rn(g, b, D, dtype=dtype)
    B, C = _rn(g, b, N, dtype=dtype), _rn(g, b, N, dtype=dtype)
    A = -torch.rand(D, N, generator=g).add_(0.5).cuda()
    Dskip, bias = _rn(g, D), _rn(g, D, std=0.1)
    s0 = _rn(g, b, D, N)
    state, sband, sref = poisoned((b, D, N), torch.float32)
    state.copy_(s0)
    y, yband, yref = poisoned((b, D), dtype)
    api.state_update(state, u, dl, A, B, C, Dskip, z, bias, y=y)
    want_state = s0.clone()
    want_y = api.state_update(want_state, u, dl, A, B, C, Dskip, z, bias)
    torch.cuda.synchronize()
    band_intact(sband, sref, "state")
    band_intact(yband, yref, "y")
    assert torch.equal(state, want_state)
    assert torch.equal(y, want_y)


# ---------------------------------------------------------------- convolution

@pytest.mark.parametrize("b,D,L,W,dtype", [
    (2, 24, 203, 4, torch.bfloat16),  # L not a multiple of 8: per-row kernel
    (2, 40, 512, 4, torch.bfloat16),  # streamed kernel
    (3, 17, 96, 2, torch.float32),    # width 2, fp32
])
def test_conv1d_guard_bands(b, D, L, W, dtype):
    g = torch.Generator().manual_seed(L + W)
    x = _rn(g, b, D, L, dtype=dtype)
    w, bias = _rn(g, D, W, std=0.5), _rn(g, D, std=0.1)
    s_in = _rn(g, b, D, W - 1, dtype=dtype)
    u, uband, uref = poisoned((b, D, L), dtype)
    so, sband, sref = poisoned((b, D, W - 1), dtype)
    api.conv1d(x, w, bias, s_in, u=u, state_out=so)
    want_u, want_so = api.conv1d(x, w, bias, s_in)
    torch.cuda.synchronize()
    band_intact(uband, uref, "u")
    band_intact(sband, sref, "state_out")
    assert torch.equal(u, want_u)
    assert torch.equal(so, want_so)


@pytest.mark.parametrize("b,D,W,dtype", [
    (5, 64, 4, torch.bfloat16),       # D a multiple of 8: eight channels per thread
    (3, 21, 4, torch.float32),        # one channel per thread
    (2, 40, 3, torch.bfloat16),
])
def test_conv1d_step_guard_bands(b, D, W, dtype):
    g = torch.Generator().manual_seed(D + W)
    x = _rn(g, b, D, dtype=dtype)
    w, bias = _rn(g, D, W, std=0.5), _rn(g, D, std=0.1)
    s0 = _rn(g, b, D, W - 1, dtype=dtype)
    st, sband, sref = poisoned((b, D, W - 1), dtype)
    st.copy_(s0)
    u, uband, uref = poisoned((b, D), dtype)
    api.conv1d_step(st, x, w, bias, u=u)
    want_st = s0.clone()
    want_u = api.conv1d_step(want_st, x, w, bias)
    torch.cuda.synchronize()
    band_intact(sband, sref, "state")
    band_intact(uband, uref, "u")
    assert torch.equal(st, want_st)
    assert torch.equal(u, want_u)


# ---------------------------------------------------------------- backward

@pytest.mark.parametrize("b,D,N,L,dtype", [
    (2, 48, 16, 300, torch.bfloat16),   # ragged tail, several 128-token chunks
    (1, 33, 7, 150, torch.float32),     # fp32, odd state size
])
def test_scan_bwd_guard_bands_on_all_nine_outputs(b, D, N, L, dtype):
    g = torch.Generator().manual_seed(D * N + L)
    u, dl, z = _rn(g, b, D, L, dtype=dtype), _rn(g, b, D, L, std=0.5, dtype=dtype), _rn(g, b, D, L, dtype=dtype)
    B, C, dy = _rn(g, b, N, L, dtype=dtype), _rn(g, b, N, L, dtype=dtype), _rn(g, b, D, L, dtype=dtype)
    A = -torch.rand(D, N, generator=g).add_(0.5).cuda()
    Dskip = _rn(g, D)
    bias = torch.log(torch.expm1(torch.empty(D).uniform_(1e-3, 1e-1, generator=g))).float().cuda()
    h0, dhL = _rn(g, b, D, N, std=0.5), _rn(g, b, D, N, std=0.5)
    f32 = torch.float32
    outs = dict(du=poisoned((b, D, L), dtype), ddelta=poisoned((b, D, L), dtype), dz=poisoned((b, D, L), dtype),
                dB=poisoned((b, N, L), f32), dC=poisoned((b, N, L), f32), dA=poisoned((D, N), f32),
                dD=poisoned((D,), f32), ddelta_bias=poisoned((D,), f32), dh0=poisoned((b, D, N), f32))
    ws = torch.empty(api.bwd_workspace_bytes(b, D, N, L, 0, dtype), dtype=torch.uint8, device="cuda")
    t = {k: v[0] for k, v in outs.items()}
    p = api.bwd_params(u, dl, A, B, C, dy, Dskip, z, bias, h0, dhL, du=t["du"], ddelta=t["ddelta"], dB=t["dB"],
                       dC=t["dC"], dA=t["dA"], dz=t["dz"], dD=t["dD"], ddelta_bias=t["ddelta_bias"], dh0=t["dh0"],
                       workspace=ws)
    from mamba_selective_scan_02_b300 import capi
    capi.check(capi.ssm_scan_bwd(p, torch.cuda.current_stream().cuda_stream), "ssm_scan_bwd")
    want = api.scan_bwd(u, dl, A, B, C, dy, Dskip, z, bias, h0, dhL)
    torch.cuda.synchronize()
    assert api.workspace_status(ws) == capi.SSM_OK
    for k, (out, band, ref) in outs.items():
        band_intact(band, ref, k)
        got, exp = out.double(), want[k].double()
        scale = 1.0 + exp.abs() + exp.pow(2).mean().sqrt()
        assert torch.all((got - exp).abs() <= 1e-5 * scale), f"{k}: differs from the same call into plain tensors"
