"""Seeded sweep of random small shapes for every kernel family against the
fp64 oracle: odd channel counts, ragged lengths, every state size up to 16,
optional inputs on and off, both I/O types and both discretisations.  The
draws are fixed by the seeds below, so a failure reproduces."""

import numpy as np
import pytest
import torch

from mamba_selective_scan_02_b300 import api
from mamba_selective_scan_02_b300.inputs import make_conv_inputs, make_ssd_inputs
from oracle import oracle as orc

import ssm_testutil as tu

DT = {0: torch.float32, 1: torch.bfloat16}


def scan_case(seed):
    rng = np.random.default_rng(seed)
    b = int(rng.integers(1, 4))
    D = int(rng.integers(1, 70))
    N = int(rng.integers(1, 17))
    L = int(rng.integers(1, 400))
    dtype = DT[int(rng.integers(0, 2))]
    opts = dict(z=bool(rng.integers(0, 2)), h0=bool(rng.integers(0, 2)), zoh=bool(rng.integers(0, 2)),
                softplus=bool(rng.integers(0, 2)), skip=bool(rng.integers(0, 2)),
                chunk=int(rng.choice([0, 64, 128])))
    return b, D, N, L, dtype, opts


@pytest.mark.gpu
@pytest.mark.parametrize("seed", range(24))
def test_scan_random_shape(seed):
    b, D, N, L, dtype, o = scan_case(seed)
    g = torch.Generator(device="cuda").manual_seed(1000 + seed)
    rn = lambda *s, std=1.0: (torch.randn(*s, generator=g, device="cuda") * std).to(dtype)
    u, z = rn(b, D, L), rn(b, D, L) if o["z"] else None
    delta = rn(b, D, L, std=0.5)
    if not o["softplus"]:
        delta = (delta.float().abs() * 0.1 + 0.01).to(dtype)
    B, C = rn(b, N, L), rn(b, N, L)
    A = -(torch.rand(D, N, generator=g, device="cuda") * 3 + 0.1)
    Dsk = torch.randn(D, generator=g, device="cuda") if o["skip"] else None
    bias = torch.randn(D, generator=g, device="cuda") * 0.5
    if not o["softplus"]:
        bias = bias.abs() * 0.1          # Δ = Δraw + bias must stay positive without softplus
    h0 = torch.randn(b, D, N, generator=g, device="cuda") * 0.3 if o["h0"] else None
    y, hL = api.scan_fwd(u, delta, A, B, C, Dsk, z, bias, h0, delta_softplus=o["softplus"], zoh=o["zoh"],
                         chunk_len=o["chunk"])
    torch.cuda.synchronize()
    c = lambda t: None if t is None else t.cpu()
    wy, wh = orc.scan(c(u), c(delta), c(A), c(B), c(C), Dskip=c(Dsk), z=c(z), bias=c(bias), h0=c(h0),
                      delta_softplus=o["softplus"], zoh=o["zoh"])
    tu.assert_close(y.float().cpu().numpy(), wy, dtype, f"y seed {seed}")
    tu.assert_close(hL.cpu().numpy(), wh, dtype, f"hL seed {seed}")


@pytest.mark.gpu
@pytest.mark.parametrize("seed", range(12))
def test_backward_random_shape(seed):
    b, D, N, L, dtype, o = scan_case(500 + seed)
    L = min(L, 200)
    g = torch.Generator(device="cuda").manual_seed(2000 + seed)
    rn = lambda *s, std=1.0: (torch.randn(*s, generator=g, device="cuda") * std).to(dtype)
    u, delta, z, dy = rn(b, D, L), rn(b, D, L, std=0.5), rn(b, D, L) if o["z"] else None, rn(b, D, L)
    B, C = rn(b, N, L), rn(b, N, L)
    A = -(torch.rand(D, N, generator=g, device="cuda") * 2 + 0.2)
    Dsk = torch.randn(D, generator=g, device="cuda")
    bias = torch.randn(D, generator=g, device="cuda") * 0.5
    h0 = torch.randn(b, D, N, generator=g, device="cuda") * 0.3 if o["h0"] else None
    dhL = torch.randn(b, D, N, generator=g, device="cuda") * 0.3
    out = api.scan_bwd(u, delta, A, B, C, dy, Dsk, z, bias, h0, dhL, zoh=o["zoh"], chunk_len=o["chunk"] // 16 * 16)
    torch.cuda.synchronize()
    c = lambda t: None if t is None else t.cpu()
    want = orc.scan_bwd(c(u), c(delta), c(A), c(B), c(C), c(dy), Dskip=c(Dsk), z=c(z), bias=c(bias), h0=c(h0),
                        dhL=c(dhL), zoh=o["zoh"])
    tol = tu.TOL[dtype]
    for name, key in (("du", "du"), ("ddelta", "ddelta"), ("dz", "dz"), ("dh0", "dh0"), ("dB", "dB"),
                      ("dC", "dC"), ("dA", "dA"), ("dD", "dDskip"), ("ddelta_bias", "dbias")):
        if out[name] is None or want[key] is None:
            continue
        got = out[name].double().cpu().numpy()
        w = np.asarray(want[key])
        scale = 1.0 + np.abs(w) + np.sqrt(np.mean(w ** 2, axis=-1, keepdims=True))
        assert np.all(np.abs(got - w) <= tol * scale), f"{name} seed {seed}"


@pytest.mark.gpu
@pytest.mark.parametrize("seed", range(12))
def test_conv_random_shape(seed):
    rng = np.random.default_rng(3000 + seed)
    b, D, L, W = int(rng.integers(1, 4)), int(rng.integers(1, 70)), int(rng.integers(1, 700)), int(rng.integers(1, 5))
    io = "bf16" if rng.integers(0, 2) else "f32"
    inp = make_conv_inputs(b, D, L, W, io, seed=seed, device="cuda", with_state=bool(rng.integers(0, 2)))
    u, st = api.conv1d(inp["x"], inp["weight"], inp["bias"], inp["state"])
    torch.cuda.synchronize()
    wu, wst = orc.conv1d(inp["x"].cpu(), inp["weight"].cpu(), inp["bias"].cpu(),
                         None if inp["state"] is None else inp["state"].cpu())
    tol = 4e-3 if io == "bf16" else 1e-5
    assert np.all(np.abs(u.double().cpu().numpy() - wu) <= tol * (1 + np.abs(wu))), f"conv seed {seed}"
    assert torch.equal(st.cpu(), torch.from_numpy(wst).to(st.dtype)), f"conv state seed {seed}"


@pytest.mark.gpu
@pytest.mark.parametrize("seed", range(8))
def test_ssd_random_shape(seed):
    rng = np.random.default_rng(4000 + seed)
    b, L, H = int(rng.integers(1, 3)), int(rng.integers(1, 300)), int(rng.integers(1, 6))
    inp = make_ssd_inputs(b, L, H, seed=seed, device="cuda", with_h0=bool(rng.integers(0, 2)))
    y, hL = api.ssd_fwd(inp["x"], inp["dt"], inp["A"], inp["B"], inp["C"], inp["D"], inp["dt_bias"], inp["h0"])
    torch.cuda.synchronize()
    c = {k: (v.cpu() if torch.is_tensor(v) else v) for k, v in inp.items()}
    wy, wh = orc.ssd(c["x"], c["dt"], c["A"], c["B"], c["C"], Dskip=c["D"], dt_bias=c["dt_bias"], h0=c["h0"])
    assert np.all(np.abs(y.double().cpu().numpy() - wy) <= 2e-2 * (1 + np.abs(wy))), f"ssd y seed {seed}"
    sc = 1 + np.abs(wh) + np.sqrt(np.mean(wh ** 2))
    assert np.all(np.abs(hL.double().cpu().numpy() - wh) <= 2e-2 * sc), f"ssd hL seed {seed}"
