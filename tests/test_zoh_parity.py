"""Exact zero-order hold on the GPU: B̄ = (e^{ΔA} − 1)/A · B instead of the
first-order Δ·B ("Mamba and selective state spaces, from first principles" —
"Discretisation: zero-order hold").  The CUDA scan and decode step against the
fp64 oracle's ZOH mode, and the two closed forms the same section states: the
N = 1 gated RNN and the reset to the current input when Δ is large."""

import numpy as np
import pytest
import torch
from scipy.special import expit

from mamba_selective_scan_02_b300 import api
from ssm_testutil import assert_close, gpu_scan, oracle_scan, to_device
from oracle import oracle as orc

pytestmark = pytest.mark.gpu


def _case(b, D, N, L, dtype, seed, h0=True):
    g = torch.Generator().manual_seed(seed)
    rn = lambda *s, std=1.0: (torch.randn(*s, generator=g) * std).to(dtype)
    return dict(u=rn(b, D, L), delta=rn(b, D, L, std=0.5), z=rn(b, D, L), B=rn(b, N, L), C=rn(b, N, L),
                A=-torch.arange(1, N + 1, dtype=torch.float32).repeat(D, 1) * (0.5 + torch.rand(D, 1, generator=g)),
                Dskip=torch.randn(D, generator=g),
                bias=torch.log(torch.expm1(torch.empty(D).uniform_(1e-3, 1e-1, generator=g))).float(),
                h0=torch.randn(b, D, N, generator=g) * 0.5 if h0 else None)


@pytest.mark.parametrize("b,D,N,L,dtype,chunk", [
    (1, 40, 16, 200, torch.float32, 0),
    (2, 64, 16, 512, torch.bfloat16, 128),      # look-back chunks
    (1, 33, 5, 203, torch.float32, 0),          # plain loads, small N
    (4, 3600, 16, 512, torch.bfloat16, 64),     # chained chunks, partial last group
])
def test_scan_zoh_matches_oracle(b, D, N, L, dtype, chunk):
    inp = _case(b, D, N, L, dtype, seed=D + N + L)
    y_ref, h_ref = orc.scan(inp["u"], inp["delta"], inp["A"], inp["B"], inp["C"], Dskip=inp["Dskip"],
                            z=inp["z"], bias=inp["bias"], h0=inp["h0"], zoh=True, threads=8)
    y, hL = gpu_scan(to_device(inp), zoh=True, chunk_len=chunk)
    assert_close(y.double().cpu().numpy(), y_ref, dtype, "zoh y")
    assert_close(hL.double().cpu().numpy(), h_ref, dtype, "zoh hL")


def test_gated_rnn_closed_form_on_gpu():
    """N = 1, A = −1, B = C = 1, D = 0, Δ = softplus(z_t), no output gate:
    h_t = (1 − σ(z_t)) h_{t−1} + σ(z_t) x_t (the gated RNN of the same section)."""
    L = 300
    g = torch.Generator().manual_seed(7)
    zt = torch.randn(1, 1, L, generator=g) * 2
    x = torch.randn(1, 1, L, generator=g)
    dev = dict(u=x.cuda(), delta=zt.cuda(), A=torch.full((1, 1), -1.0).cuda(),
               B=torch.ones(1, 1, L).cuda(), C=torch.ones(1, 1, L).cuda())
    y, hL = api.scan_fwd(dev["u"], dev["delta"], dev["A"], dev["B"], dev["C"], zoh=True)
    torch.cuda.synchronize()
    s = expit(zt.double().numpy()[0, 0])
    h, want = 0.0, []
    for t in range(L):
        h = (1 - s[t]) * h + s[t] * x.double().numpy()[0, 0, t]
        want.append(h)
    assert_close(y.double().cpu().numpy()[0, 0], np.array(want), torch.float32, "gated RNN")


def test_large_step_resets_to_input_on_gpu():
    """Δ → ∞ with A = −1, B = 1 under exact ZOH: h_t = u_t whatever came before."""
    L, D = 64, 8
    g = torch.Generator().manual_seed(8)
    u = torch.randn(1, D, L, generator=g)
    y, hL = api.scan_fwd(u.cuda(), torch.full((1, D, L), 200.0).cuda(), torch.full((D, 1), -1.0).cuda(),
                         torch.ones(1, 1, L).cuda(), torch.ones(1, 1, L).cuda(),
                         h0=torch.full((1, D, 1), 5.0).cuda(), delta_softplus=False, zoh=True)
    torch.cuda.synchronize()
    assert_close(y.double().cpu().numpy(), u.double().numpy(), torch.float32, "reset to input")


@pytest.mark.parametrize("D,dtype", [(256, torch.bfloat16), (130, torch.float32)])
def test_decode_zoh_matches_oracle(D, dtype):
    b, N, T = 3, 16, 12
    inp = _case(b, D, N, T, dtype, seed=D)
    y_ref, h_ref = orc.scan(inp["u"], inp["delta"], inp["A"], inp["B"], inp["C"], Dskip=inp["Dskip"],
                            z=inp["z"], bias=inp["bias"], h0=inp["h0"], zoh=True)
    dev = to_device(inp)
    state = dev["h0"].clone()
    ys = []
    for t in range(T):
        sl = lambda x: x[..., t].contiguous()
        ys.append(api.state_update(state, sl(dev["u"]), sl(dev["delta"]), dev["A"], sl(dev["B"]),
                                   sl(dev["C"]), dev["Dskip"], sl(dev["z"]), dev["bias"], zoh=True))
    torch.cuda.synchronize()
    assert_close(torch.stack(ys, -1).double().cpu().numpy(), y_ref, dtype, "decode zoh y")
    assert_close(state.cpu().numpy(), h_ref, dtype, "decode zoh state")
