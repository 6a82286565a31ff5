"""The causal depthwise convolution + SiLU kernels against the fp64 oracle.

Tolerances follow from the arithmetic: the kernels accumulate the W taps in
fp32 with fused multiply-adds and form SiLU with MUFU approximations
(ex2 + rcp for fp32 I/O, tanh for bf16 I/O), then round once to the I/O type.

  fp32 I/O: |err| <= 1e-5 · (1 + |u|)   (a few fp32 ulps of accumulation and
                                          the approximations' ~2^-21 relative error)
  bf16 I/O: |err| <= 4e-3 · (1 + |u|)   (half a bf16 ulp, 2^-9 relative, plus
                                          tanh.approx's error on σ)

The carried states are copies of inputs and must match bit for bit.
"""

import numpy as np
import pytest
import torch

from mamba_selective_scan_02_b300 import api
from mamba_selective_scan_02_b300.inputs import make_conv_inputs, make_inputs
from oracle import oracle as orc

import ssm_testutil as tu

CONV_TOL = {torch.float32: 1e-5, torch.bfloat16: 4e-3}
DT = {"f32": torch.float32, "bf16": torch.bfloat16}


def check(got, want, dtype, what):
    got = got.double().cpu().numpy() if torch.is_tensor(got) else np.asarray(got, np.float64)
    want = np.asarray(want, np.float64)
    assert got.shape == want.shape, (what, got.shape, want.shape)
    assert np.all(np.isfinite(got)), f"{what}: non-finite values from the GPU"
    err = np.abs(got - want)
    bound = CONV_TOL[dtype] * (1.0 + np.abs(want))
    bad = err > bound
    if bad.any():
        i = np.unravel_index(np.argmax(err / bound), err.shape)
        raise AssertionError(f"{what}: {bad.sum()} of {err.size} outside tolerance; worst at {i}: "
                             f"got {got[i]!r} want {want[i]!r}")


def exact(got, want, dtype, what):
    want_t = torch.from_numpy(np.ascontiguousarray(want)).to(dtype)
    assert torch.equal(got.cpu(), want_t), f"{what}: not bit-exact"


@pytest.mark.gpu
@pytest.mark.parametrize("io", ["f32", "bf16"])
@pytest.mark.parametrize("width", [1, 2, 3, 4])
@pytest.mark.parametrize("shape", [(2, 64, 1536),    # vector path, three 512-token segments
                                   (2, 37, 1000),    # ragged: scalar path, partial granules
                                   (3, 16, 8),       # one granule
                                   (1, 5, 2),        # shorter than the carried state
                                   (1, 3, 1)])
def test_conv_every_element(io, width, shape):
    b, D, L = shape
    dtype = DT[io]
    inp = make_conv_inputs(b, D, L, width, io, seed=width * 100 + L, device="cuda")
    for with_state in (True, False):
        st_in = inp["state"] if with_state else None
        for silu in (True, False):
            u, st = api.conv1d(inp["x"], inp["weight"], inp["bias"], st_in, silu=silu)
            torch.cuda.synchronize()
            wu, wst = orc.conv1d(inp["x"].cpu(), inp["weight"].cpu(), inp["bias"].cpu(),
                                 None if st_in is None else st_in.cpu(), silu=silu)
            check(u, wu, dtype, f"u {shape} W={width} state={with_state} silu={silu}")
            exact(st, wst, dtype, f"state {shape} W={width}")


@pytest.mark.gpu
def test_conv_no_bias_no_state_outputs():
    inp = make_conv_inputs(2, 48, 512, 4, "bf16", seed=7, device="cuda")
    u, st = api.conv1d(inp["x"], inp["weight"], None, None, return_state=False)
    torch.cuda.synchronize()
    assert st is None
    wu, _ = orc.conv1d(inp["x"].cpu(), inp["weight"].cpu())
    check(u, wu, torch.bfloat16, "u without bias")


@pytest.mark.gpu
def test_conv_split_sequence_carries_state():
    # the state written by one call, fed to the next, gives the whole sequence
    inp = make_conv_inputs(2, 40, 1024, 4, "f32", seed=9, device="cuda")
    x = inp["x"]
    u, st = api.conv1d(x, inp["weight"], inp["bias"], inp["state"])
    ua, sa = api.conv1d(x[..., :520].contiguous(), inp["weight"], inp["bias"], inp["state"])
    ub, sb = api.conv1d(x[..., 520:].contiguous(), inp["weight"], inp["bias"], sa)
    torch.cuda.synchronize()
    wu, wst = orc.conv1d(x.cpu(), inp["weight"].cpu(), inp["bias"].cpu(), inp["state"].cpu())
    check(torch.cat([ua, ub], -1), wu, torch.float32, "split sequence")
    exact(sb, wst, torch.float32, "state after split")


@pytest.mark.gpu
def test_conv_mamba28b_layer_sampled():
    # the layer shape the scan is measured on, in the launch configuration the
    # benchmark times: every final state, and sampled rows of u
    b, D, L = 4, 5120, 2048
    inp = make_conv_inputs(b, D, L, 4, "bf16", seed=11, device="cuda")
    u, st = api.conv1d(inp["x"], inp["weight"], inp["bias"], inp["state"])
    torch.cuda.synchronize()
    chans = tu.sample_channels(b, D, 48, seed=3)
    for bi, d in chans:
        wu, wst = orc.conv1d(inp["x"][bi:bi + 1, d:d + 1].cpu(), inp["weight"][d:d + 1].cpu(),
                             inp["bias"][d:d + 1].cpu(), inp["state"][bi:bi + 1, d:d + 1].cpu())
        check(u[bi:bi + 1, d:d + 1], wu, torch.bfloat16, f"u row ({bi},{d})")
        exact(st[bi:bi + 1, d:d + 1], wst, torch.bfloat16, f"state ({bi},{d})")
    # every final state is the last three inputs of its row (oracle on the
    # last three tokens from the carried inputs before them)
    x3 = inp["x"][..., -3:].cpu()
    _, wst = orc.conv1d(x3, inp["weight"].cpu(), inp["bias"].cpu(), inp["x"][..., -6:-3].cpu())
    exact(st, wst, torch.bfloat16, "every final state")


@pytest.mark.gpu
@pytest.mark.parametrize("io", ["f32", "bf16"])
@pytest.mark.parametrize("width", [1, 2, 4])
def test_conv_step_tokens(io, width):
    b, D, T = 3, 300, 6
    dtype = DT[io]
    inp = make_conv_inputs(b, D, T, width, io, seed=5 + width, device="cuda", decode=True)
    state = inp["state"].clone() if width > 1 else None
    wstate = inp["state"].cpu().double().numpy().copy()
    for t in range(T):
        u = api.conv1d_step(state, inp["x"][t], inp["weight"], inp["bias"])
        torch.cuda.synchronize()
        wu, wstate = orc.conv1d_step(wstate, inp["x"][t].cpu(), inp["weight"].cpu(), inp["bias"].cpu())
        check(u, wu, dtype, f"decode token {t} W={width}")
        if width > 1:
            exact(state, wstate, dtype, f"decode state after token {t} W={width}")


@pytest.mark.gpu
def test_conv_then_scan_block_branch():
    # the SSM branch of the block: x -> conv + SiLU -> u -> selective scan
    w = make_inputs("small_layer_L2048", device="cuda", batch=2, dim=96, seqlen=300, seed=21)
    cin = make_conv_inputs(2, 96, 300, 4, "bf16", seed=22, device="cuda")
    u, _ = api.conv1d(cin["x"], cin["weight"], cin["bias"], cin["state"])
    y, hL = api.scan_fwd(u, w["delta"], w["A"], w["B"], w["C"], w["Dskip"], w["z"], w["bias"])
    torch.cuda.synchronize()
    wu, _ = orc.conv1d(cin["x"].cpu(), cin["weight"].cpu(), cin["bias"].cpu(), cin["state"].cpu())
    wy, wh = orc.scan(wu, w["delta"].cpu(), w["A"].cpu(), w["B"].cpu(), w["C"].cpu(),
                      Dskip=w["Dskip"].cpu(), z=w["z"].cpu(), bias=w["bias"].cpu())
    tu.assert_close(y.float().cpu().numpy(), wy, torch.bfloat16, "conv -> scan y")
    tu.assert_close(hL.cpu().numpy(), wh, torch.bfloat16, "conv -> scan state")
