"""The Mamba-2 (SSD) kernel against the fp64 oracle's recurrence.

The kernel multiplies bf16 operands on the tensor cores with fp32
accumulation: x, B, C enter as the bf16 inputs themselves, while the decay-
masked C·Bᵀ block, the x scaled by the state weights and the carried state
enter as a bf16 value plus a bf16 remainder (about 2^-17 relative each)
before sums of 128 terms.  The contract's bf16 tolerance, |err| <=
2e-2·(1 + |y|), covers it; the final state (fp32, built from such products) is
held to the same bound relative to its scale.
"""

import numpy as np
import pytest
import torch

from mamba_selective_scan_02_b300 import api
from mamba_selective_scan_02_b300.inputs import make_ssd_inputs
from oracle import oracle as orc

TOL = 2e-2


def check(name, got, want, scale=None):
    got = got.double().cpu().numpy()
    want = np.asarray(want, np.float64)
    assert got.shape == want.shape, (name, got.shape, want.shape)
    assert np.all(np.isfinite(got)), f"{name}: non-finite values from the GPU"
    sc = 1.0 + np.abs(want) if scale is None else scale
    err = np.abs(got - want)
    bad = err > TOL * sc
    if bad.any():
        i = np.unravel_index(np.argmax(err / sc), err.shape)
        raise AssertionError(f"{name}: {bad.sum()} of {err.size} outside tolerance; worst at {i}: "
                             f"got {got[i]!r} want {want[i]!r} (ratio {(err / sc).max() / TOL:.2f})")
    return float((err / sc).max() / TOL)


def run(inp, softplus=True):
    y, hL = api.ssd_fwd(inp["x"], inp["dt"], inp["A"], inp["B"], inp["C"], inp["D"], inp["dt_bias"], inp["h0"],
                        dt_softplus=softplus)
    torch.cuda.synchronize()
    c = {k: (v.cpu() if torch.is_tensor(v) else v) for k, v in inp.items()}
    wy, wh = orc.ssd(c["x"], c["dt"], c["A"], c["B"], c["C"], Dskip=c["D"], dt_bias=c["dt_bias"], h0=c["h0"],
                     dt_softplus=softplus)
    return y, hL, wy, wh


@pytest.mark.gpu
@pytest.mark.parametrize("shape", [(2, 300, 3),    # ragged: two full 128-token chunks and a partial one
                                   (1, 128, 2),    # exactly one chunk
                                   (1, 1, 1),      # a single token
                                   (3, 130, 5),    # one chunk and two tokens
                                   (1, 520, 2)])   # four chunks and a short tail
@pytest.mark.parametrize("h0", [False, True])
def test_ssd_every_element(shape, h0):
    b, L, H = shape
    inp = make_ssd_inputs(b, L, H, seed=L + H, device="cuda", with_h0=h0)
    y, hL, wy, wh = run(inp)
    check("y", y, wy)
    check("hL", hL, wh, scale=1.0 + np.abs(wh) + np.sqrt(np.mean(wh ** 2)))


@pytest.mark.gpu
def test_ssd_plain_options():
    # no skip, no Δ bias, no softplus (Δ = dt itself, kept positive)
    inp = make_ssd_inputs(2, 150, 2, seed=3, device="cuda")
    inp["dt"] = (inp["dt"].float().abs() * 0.05 + 0.01).to(torch.bfloat16)
    inp["D"] = None
    inp["dt_bias"] = None
    y, hL, wy, wh = run(inp, softplus=False)
    check("y", y, wy)
    check("hL", hL, wh, scale=1.0 + np.abs(wh) + np.sqrt(np.mean(wh ** 2)))


@pytest.mark.gpu
def test_ssd_mamba2_layer_sampled():
    # the Mamba-2 2.7B layer shape the benchmark times: sampled (sequence, head) pairs
    b, L, H = 4, 2048, 80
    inp = make_ssd_inputs(b, L, H, seed=7, device="cuda")
    y, hL = api.ssd_fwd(inp["x"], inp["dt"], inp["A"], inp["B"], inp["C"], inp["D"], inp["dt_bias"])
    torch.cuda.synchronize()
    rng = np.random.default_rng(0)
    pairs = {(0, 0), (b - 1, H - 1)} | {(int(rng.integers(b)), int(rng.integers(H))) for _ in range(6)}
    for bi, h in sorted(pairs):
        wy, wh = orc.ssd(inp["x"][bi:bi + 1, :, h:h + 1].cpu(), inp["dt"][bi:bi + 1, :, h:h + 1].cpu(),
                         inp["A"][h:h + 1].cpu(), inp["B"][bi:bi + 1].cpu(), inp["C"][bi:bi + 1].cpu(),
                         Dskip=inp["D"][h:h + 1].cpu(), dt_bias=inp["dt_bias"][h:h + 1].cpu())
        check(f"y[{bi}, :, {h}]", y[bi:bi + 1, :, h:h + 1], wy)
        check(f"hL[{bi}, {h}]", hL[bi:bi + 1, h:h + 1], wh, scale=1.0 + np.abs(wh) + np.sqrt(np.mean(wh ** 2)))


def _poisoned(shape, dtype, pad=4096):
    """A tensor of `shape` at the front of a larger buffer whose tail holds a
    fixed bit pattern, so that a write past the end shows."""
    n = int(np.prod(shape))
    buf = torch.empty(n + pad, dtype=dtype, device="cuda")
    buf.view(torch.int16 if dtype == torch.bfloat16 else torch.int32).fill_(0x7B3D)
    return buf[:n].view(shape), buf[n:], buf[n:].clone()


@pytest.mark.gpu
@pytest.mark.parametrize("L", [1, 127, 129, 300])
def test_ssd_writes_nothing_past_y_and_hL(L):
    b, H, P, N = 2, 3, 64, 128
    inp = make_ssd_inputs(b, L, H, seed=11 + L, device="cuda", with_h0=True)
    y, ytail, yref = _poisoned((b, L, H, P), torch.bfloat16)
    hL, htail, href = _poisoned((b, H, P, N), torch.float32)
    status = torch.zeros(1, dtype=torch.int32, device="cuda")
    api.ssd_fwd(inp["x"], inp["dt"], inp["A"], inp["B"], inp["C"], inp["D"], inp["dt_bias"], inp["h0"],
                y=y, hL=hL, status=status)
    torch.cuda.synchronize()
    assert int(status.item()) == 0
    assert torch.equal(ytail, yref), "y: bytes past the end were written"
    assert torch.equal(htail, href), "hL: bytes past the end were written"
    c = {k: (v.cpu() if torch.is_tensor(v) else v) for k, v in inp.items()}
    wy, wh = orc.ssd(c["x"], c["dt"], c["A"], c["B"], c["C"], Dskip=c["D"], dt_bias=c["dt_bias"], h0=c["h0"])
    check("y", y, wy)
    check("hL", hL, wh, scale=1.0 + np.abs(wh) + np.sqrt(np.mean(wh ** 2)))


@pytest.mark.gpu
@pytest.mark.parametrize("b,L,H", [(2, 300, 3), (1, 1000, 2), (3, 520, 4), (1, 128, 1)])
@pytest.mark.parametrize("h0", [False, True])
def test_ssd_segments_equal_whole_chains(b, L, H, h0):
    # the segment hand-off passes the fp32 state exactly: split and unsplit
    # launches must agree bit for bit
    inp = make_ssd_inputs(b, L, H, seed=b * L + H, device="cuda", with_h0=h0)
    args = (inp["x"], inp["dt"], inp["A"], inp["B"], inp["C"], inp["D"], inp["dt_bias"], inp["h0"])
    status = torch.zeros(1, dtype=torch.int32, device="cuda")
    y1, h1 = api.ssd_fwd(*args, split=True, status=status)
    y2, h2 = api.ssd_fwd(*args, split=False)
    torch.cuda.synchronize()
    assert int(status.item()) == 0
    assert torch.equal(y1, y2)
    assert torch.equal(h1, h2)


@pytest.mark.gpu
def test_ssd_workspace_reused_across_calls():
    # the call clears the counter and flags itself: one workspace serves calls
    # of different sizes in a row
    ws = torch.empty(api.ssd_workspace_bytes(2, 1000, 4), dtype=torch.uint8, device="cuda")
    for seed, (b, L, H) in enumerate([(2, 1000, 4), (1, 700, 3), (2, 1000, 4)]):
        inp = make_ssd_inputs(b, L, H, seed=seed, device="cuda")
        args = (inp["x"], inp["dt"], inp["A"], inp["B"], inp["C"], inp["D"], inp["dt_bias"], None)
        y1, h1 = api.ssd_fwd(*args, workspace=ws)
        y2, h2 = api.ssd_fwd(*args, split=False)
        torch.cuda.synchronize()
        assert torch.equal(y1, y2) and torch.equal(h1, h2), (b, L, H)
