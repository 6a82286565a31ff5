"""Decode step: CUDA state update against the fp64 oracle, and against the scan."""

import pytest
import torch

from mamba_selective_scan_02_b300 import api
from mamba_selective_scan_02_b300.inputs import WORKLOADS, make_inputs
from oracle import oracle as orc
from ssm_testutil import assert_close, gpu_scan, oracle_scan

pytestmark = pytest.mark.gpu


def test_decode_workload_64_tokens_sampled_sequences():
    """256 sequences × 5120 channels × N=16, 64 consecutive tokens; the oracle
    follows a sample of whole sequences (all their channels) token by token."""
    w = WORKLOADS["decode_b256_64tok"]
    inp = make_inputs(w, device="cuda")
    state = inp["h0"].clone()
    rows = [0, 1, 77, 128, 255]
    st_ref = inp["h0"][rows].double().cpu().numpy()
    A = inp["A"].cpu()
    for t in range(w.seqlen):
        y = api.state_update(state, inp["u"][t], inp["delta"][t], inp["A"], inp["B"][t], inp["C"][t],
                             inp["Dskip"], inp["z"][t], inp["bias"])
        y_ref, st_ref = orc.step(st_ref, inp["u"][t][rows].cpu(), inp["delta"][t][rows].cpu(), A,
                                 inp["B"][t][rows].cpu(), inp["C"][t][rows].cpu(),
                                 Dskip=inp["Dskip"].cpu(), z=inp["z"][t][rows].cpu(),
                                 bias=inp["bias"].cpu())
        if t % 8 == 0 or t == w.seqlen - 1:
            assert_close(y[rows].double().cpu().numpy(), y_ref, torch.bfloat16, f"token {t} y")
    torch.cuda.synchronize()
    assert_close(state[rows].cpu().numpy(), st_ref, torch.bfloat16, "carried state after 64 tokens")
    assert torch.isfinite(state).all()


@pytest.mark.parametrize("b,D,N,dtype,z", [
    (3, 40, 16, torch.bfloat16, True),
    (2, 33, 5, torch.float32, True),
    (1, 7, 1, torch.float32, False),
    (4, 64, 8, torch.bfloat16, False),
    (2, 130, 12, torch.float32, True),
])
def test_decode_equals_scan(b, D, N, dtype, z):
    T = 24
    g = torch.Generator().manual_seed(b + D + N)
    rn = lambda *s, std=1.0: (torch.randn(*s, generator=g) * std).to(dtype)
    inp = dict(u=rn(b, D, T), delta=rn(b, D, T, std=0.5), z=rn(b, D, T) if z else None,
               B=rn(b, N, T), C=rn(b, N, T),
               A=-torch.arange(1, N + 1, dtype=torch.float32).repeat(D, 1),
               Dskip=torch.randn(D, generator=g), bias=torch.randn(D, generator=g) * 0.3 - 2,
               h0=torch.randn(b, D, N, generator=g) * 0.1)
    y_ref, h_ref = oracle_scan(inp)
    dev = {k: (v.cuda() if torch.is_tensor(v) else v) for k, v in inp.items()}
    state = dev["h0"].clone()
    ys = []
    for t in range(T):
        sl = lambda x: None if x is None else x[..., t].contiguous()
        ys.append(api.state_update(state, sl(dev["u"]), sl(dev["delta"]), dev["A"], sl(dev["B"]),
                                   sl(dev["C"]), dev["Dskip"], sl(dev["z"]), dev["bias"]))
    y_dec = torch.stack(ys, -1)
    torch.cuda.synchronize()
    assert_close(y_dec.double().cpu().numpy(), y_ref, dtype, "decode steps vs oracle scan")
    assert_close(state.cpu().numpy(), h_ref, dtype, "decode state vs oracle")
    y_scan, h_scan = gpu_scan(dev)
    assert_close(y_dec.double().cpu().numpy(), y_scan.double().cpu().numpy(), dtype, "decode vs GPU scan")
    assert_close(state.cpu().numpy(), h_scan.cpu().numpy(), dtype, "decode state vs GPU scan")
