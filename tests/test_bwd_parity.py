"""The backward scan kernels against the fp64 oracle's gradient.

Per-element outputs (du, dΔraw, dz, dh0) use the method's tolerances:
fp32 I/O |err| <= 1e-4·(1 + |x|), bf16 I/O |err| <= 2e-2·(1 + |x|).  The
reductions (dB, dC over channels; dA, dD, dbias over batch and time) are fp32
sums of many terms accumulated with atomics in no fixed order; each term
carries the same relative error as a per-element output, so they are held to
the same tolerance relative to (1 + |x| + the row's RMS), the scale at which
cancellation between terms happens.
"""

import numpy as np
import pytest
import torch

from mamba_selective_scan_02_b300 import api
from mamba_selective_scan_02_b300.inputs import make_inputs
from oracle import oracle as orc

import ssm_testutil as tu

DT = {"f32": torch.float32, "bf16": torch.bfloat16}
ELEMENTWISE = ("du", "ddelta", "dz", "dh0")
REDUCED = ("dB", "dC", "dA", "dD", "ddelta_bias")
ORACLE_KEY = {"du": "du", "ddelta": "ddelta", "dz": "dz", "dh0": "dh0", "dB": "dB", "dC": "dC",
              "dA": "dA", "dD": "dDskip", "ddelta_bias": "dbias"}


def check(name, got, want, dtype):
    got = got.double().cpu().numpy() if torch.is_tensor(got) else np.asarray(got, np.float64)
    want = np.asarray(want, np.float64)
    assert got.shape == want.shape, (name, got.shape, want.shape)
    assert np.all(np.isfinite(got)), f"{name}: non-finite values from the GPU"
    tol = tu.TOL[dtype]
    scale = 1.0 + np.abs(want)
    if name in REDUCED:
        scale = scale + np.sqrt(np.mean(want ** 2, axis=-1, keepdims=True))
    err = np.abs(got - want)
    bad = err > tol * scale
    if bad.any():
        i = np.unravel_index(np.argmax(err / scale), err.shape)
        raise AssertionError(f"{name}: {bad.sum()} of {err.size} outside tolerance; worst at {i}: "
                             f"got {got[i]!r} want {want[i]!r}")


def draw(io, b, D, N, L, seed, gate=True, h0=True):
    w = make_inputs("small_layer_L2048" if io == "bf16" else "tiny_fp32", device="cuda", batch=b, dim=D,
                    seqlen=L, seed=seed)
    g = torch.Generator(device="cuda").manual_seed(seed + 1000)
    dt = DT[io]
    A = -torch.rand((D, N), generator=g, device="cuda") * 1.5 - 0.25
    B = torch.randn((b, N, L), generator=g, device="cuda").to(dt)
    C = torch.randn((b, N, L), generator=g, device="cuda").to(dt)
    dy = torch.randn((b, D, L), generator=g, device="cuda").to(dt)
    dhL = torch.randn((b, D, N), generator=g, device="cuda") * 0.5
    hz = torch.randn((b, D, N), generator=g, device="cuda") * 0.3 if h0 else None
    return dict(u=w["u"], delta=w["delta"], z=w["z"] if gate else None, B=B, C=C, A=A, D=w["Dskip"],
                bias=w["bias"], h0=hz, dy=dy, dhL=dhL)


def run_both(inp, zoh, chunk_len=0, threads=8):
    out = api.scan_bwd(inp["u"], inp["delta"], inp["A"], inp["B"], inp["C"], inp["dy"], inp["D"], inp["z"],
                       inp["bias"], inp["h0"], inp["dhL"], zoh=zoh, chunk_len=chunk_len)
    torch.cuda.synchronize()
    assert api.workspace_status(out["workspace"]) == 0
    cpu = {k: (v.cpu() if torch.is_tensor(v) else v) for k, v in inp.items()}
    want = orc.scan_bwd(cpu["u"], cpu["delta"], cpu["A"], cpu["B"], cpu["C"], cpu["dy"], Dskip=cpu["D"],
                        z=cpu["z"], bias=cpu["bias"], h0=cpu["h0"], dhL=cpu["dhL"], zoh=zoh, threads=threads)
    return out, want


@pytest.mark.gpu
@pytest.mark.parametrize("io", ["f32", "bf16"])
@pytest.mark.parametrize("N", [16, 5])
@pytest.mark.parametrize("zoh", [False, True])
@pytest.mark.parametrize("gate", [True, False])
@pytest.mark.parametrize("shape,chunk", [((2, 40, 300), 64),     # ragged D and L: scalar loads, partial tile
                                         ((2, 48, 256), 64),     # aligned: vector loads, four chained chunks
                                         ((1, 17, 33), 0),       # one chunk, three partial tiles
                                         ((2, 16, 16), 0),       # exactly one tile
                                         ((1, 20, 1), 0)])       # a single token
def test_bwd_every_element(io, N, zoh, gate, shape, chunk):
    b, D, L = shape
    inp = draw(io, b, D, N, L, seed=L + N + 7 * zoh, gate=gate)
    out, want = run_both(inp, zoh, chunk)
    dtype = DT[io]
    for name in ELEMENTWISE + REDUCED:
        if out[name] is None or want[ORACLE_KEY[name]] is None:
            continue
        check(f"{name} {shape} N={N} zoh={zoh} gate={gate}", out[name], want[ORACLE_KEY[name]], dtype)


@pytest.mark.gpu
def test_bwd_without_optional_inputs():
    # no h0, no dhL, no skip, no bias, no softplus: the plainest form
    b, D, N, L = 2, 32, 16, 128
    inp = draw("f32", b, D, N, L, seed=5, h0=False)
    inp["dhL"] = None
    inp["D"] = None
    inp["bias"] = None
    inp["delta"] = inp["delta"].abs() + 0.05
    out = api.scan_bwd(inp["u"], inp["delta"], inp["A"], inp["B"], inp["C"], inp["dy"], None, inp["z"], None,
                       None, None, delta_softplus=False)
    torch.cuda.synchronize()
    cpu = {k: (v.cpu() if torch.is_tensor(v) else v) for k, v in inp.items()}
    want = orc.scan_bwd(cpu["u"], cpu["delta"], cpu["A"], cpu["B"], cpu["C"], cpu["dy"], z=cpu["z"],
                        delta_softplus=False)
    for name in ("du", "ddelta", "dz", "dB", "dC", "dA"):
        check(name, out[name], want[ORACLE_KEY[name]], torch.float32)
    assert out["dD"] is None and out["ddelta_bias"] is None and out["dh0"] is None


def sampled_check(b, D, N, L, seed, nchan=12, own_checkpoints=False):
    """Per-channel gradients on sampled channels, the per-channel sums over the
    batch for those channels, and dB, dC of the first sequence over all D
    channels, against the oracle.  own_checkpoints: a workspace with no room
    for the forward kernel's checkpoint launch (the backward's own pass runs)."""
    inp = draw("bf16", b, D, N, L, seed=seed)
    ws = None
    if own_checkpoints:
        small = api.bwd_workspace_bytes(b, D, N, L, dtype=torch.float32)
        assert small < api.bwd_workspace_bytes(b, D, N, L, dtype=torch.bfloat16)
        ws = torch.empty(small, dtype=torch.uint8, device="cuda")
    out = api.scan_bwd(inp["u"], inp["delta"], inp["A"], inp["B"], inp["C"], inp["dy"], inp["D"], inp["z"],
                       inp["bias"], inp["h0"], inp["dhL"], workspace=ws)
    torch.cuda.synchronize()
    assert api.workspace_status(out["workspace"]) == 0
    dtype = torch.bfloat16
    chans = sorted({d for _, d in tu.sample_channels(b, D, nchan, seed=seed + 2)})
    for d in chans:
        sl = lambda t: None if t is None else t[:, d:d + 1].cpu()
        want = orc.scan_bwd(sl(inp["u"]), sl(inp["delta"]), inp["A"][d:d + 1].cpu(), inp["B"].cpu(),
                            inp["C"].cpu(), sl(inp["dy"]), Dskip=inp["D"][d:d + 1].cpu(), z=sl(inp["z"]),
                            bias=inp["bias"][d:d + 1].cpu(), h0=sl(inp["h0"]), dhL=sl(inp["dhL"]))
        for name in ELEMENTWISE:
            check(f"{name}[:, {d}]", out[name][:, d:d + 1], want[ORACLE_KEY[name]], dtype)
        check(f"dA[{d}]", out["dA"][d:d + 1], want["dA"], dtype)
        check(f"dD[{d}]", out["dD"][d:d + 1], want["dDskip"], dtype)
        check(f"ddelta_bias[{d}]", out["ddelta_bias"][d:d + 1], want["dbias"], dtype)
    b0 = lambda t: None if t is None else t[0:1].cpu()
    want = orc.scan_bwd(b0(inp["u"]), b0(inp["delta"]), inp["A"].cpu(), b0(inp["B"]), b0(inp["C"]),
                        b0(inp["dy"]), Dskip=inp["D"].cpu(), z=b0(inp["z"]), bias=inp["bias"].cpu(),
                        h0=b0(inp["h0"]), dhL=b0(inp["dhL"]), threads=16)
    check("dB[0]", out["dB"][0:1], want["dB"], dtype)
    check("dC[0]", out["dC"][0:1], want["dC"], dtype)


@pytest.mark.gpu
def test_bwd_mamba28b_layer_sampled():
    # The layer shape the forward is measured on, in the launch configuration
    # the benchmark times: the state checkpoints come from the forward scan's
    # warp-specialised kernel (a chained plan of 384-token chunks), the reverse
    # pass walks 128-token chunks.
    sampled_check(4, 5120, 16, 2048, seed=2)


@pytest.mark.gpu
def test_bwd_forward_checkpoints_ragged():
    # Enough channel groups (896) for the forward kernel's checkpoint launch, on
    # a sequence of two chained chunks whose last 32-token tile holds 8 tokens.
    sampled_check(2, 7168, 16, 456, seed=5, nchan=8)
    # the same shape with the backward's own checkpoint pass
    sampled_check(2, 7168, 16, 456, seed=5, nchan=8, own_checkpoints=True)
