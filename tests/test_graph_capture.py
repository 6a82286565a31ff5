"""The entry points are capturable in a CUDA graph (a serving loop replays one
captured decode step per token, or one captured layer scan): every call only
enqueues work on the given stream — memsets, launches with by-value
arguments — so a replay equals the eager call bit for bit."""

import pytest
import torch

from mamba_selective_scan_02_b300 import api, capi
from mamba_selective_scan_02_b300.inputs import make_conv_inputs, make_inputs, make_ssd_inputs


@pytest.mark.gpu
def test_scan_decode_conv_ssd_replay_in_a_graph():
    dev = torch.device("cuda")
    w = make_inputs("small_layer_L2048", device=dev, batch=2, dim=256, seqlen=1024, seed=31)
    ws = torch.empty(api.workspace_bytes(w["u"], w["delta"], w["A"], w["B"], w["C"]), dtype=torch.uint8, device=dev)
    y = torch.empty_like(w["u"])
    hL = torch.empty((2, 256, 16), dtype=torch.float32, device=dev)
    ps = api.scan_params(w["u"], w["delta"], w["A"], w["B"], w["C"], w["Dskip"], w["z"], w["bias"], None,
                         y=y, hL=hL, workspace=ws)
    state = torch.randn((2, 256, 16), device=dev) * 0.1
    state_ref = state.clone()
    yt = torch.empty((2, 256), dtype=w["u"].dtype, device=dev)
    # the decode token's inputs (kept referenced: the parameter struct holds raw pointers)
    tok = {k: w[k][:, :, 0].contiguous() for k in ("u", "delta", "B", "C", "z")}
    pt = api.step_params(state, tok["u"], tok["delta"], w["A"], tok["B"], tok["C"], w["Dskip"], tok["z"],
                         w["bias"], y=yt)
    ci = make_conv_inputs(2, 256, 1, 4, "bf16", seed=32, device=dev, decode=True)
    cstate = ci["state"].clone()
    cu = torch.empty((2, 256), dtype=torch.bfloat16, device=dev)
    si = make_ssd_inputs(1, 256, 4, seed=33, device=dev)
    sy = torch.empty_like(si["x"])
    shl = torch.empty((1, 4, 64, 128), dtype=torch.float32, device=dev)
    # with a workspace: each chain runs as segments handing the state on (a
    # memset of the work counter and flags, then the launch)
    sws = torch.empty(api.ssd_workspace_bytes(1, 256, 4), dtype=torch.uint8, device=dev)
    pssd = api.ssd_params(si["x"], si["dt"], si["A"], si["B"], si["C"], si["D"], si["dt_bias"], None, y=sy, hL=shl,
                          workspace=sws)

    side = torch.cuda.Stream(dev)
    # eager reference results (and the first call of each entry point, which
    # caches kernel attributes) on the capture stream
    with torch.cuda.stream(side):
        assert capi.ssm_scan_fwd(ps, side.cuda_stream) == capi.SSM_OK
        assert capi.ssm_state_update(pt, side.cuda_stream) == capi.SSM_OK
        api.conv1d_step(cstate, ci["x"][0], ci["weight"], ci["bias"], u=cu, stream=side.cuda_stream)
        assert capi.ssm_ssd_fwd(pssd, side.cuda_stream) == capi.SSM_OK
    torch.cuda.synchronize()
    want = [y.clone(), hL.clone(), yt.clone(), state.clone(), cu.clone(), cstate.clone(), sy.clone(), shl.clone()]

    # capture the same calls from the original states, replay, compare
    state.copy_(state_ref)
    cstate.copy_(ci["state"])
    torch.cuda.synchronize()
    g = torch.cuda.CUDAGraph()
    with torch.cuda.graph(g, stream=side):
        assert capi.ssm_scan_fwd(ps, side.cuda_stream) == capi.SSM_OK
        assert capi.ssm_state_update(pt, side.cuda_stream) == capi.SSM_OK
        api.conv1d_step(cstate, ci["x"][0], ci["weight"], ci["bias"], u=cu, stream=side.cuda_stream)
        assert capi.ssm_ssd_fwd(pssd, side.cuda_stream) == capi.SSM_OK
    for t in (y, hL, yt, cu, sy, shl):
        t.zero_()
    torch.cuda.synchronize()
    g.replay()
    torch.cuda.synchronize()
    got = [y, hL, yt, state, cu, cstate, sy, shl]
    for a_, b_ in zip(got, want):
        assert torch.equal(a_, b_)
    assert api.workspace_status(ws) == capi.SSM_OK
