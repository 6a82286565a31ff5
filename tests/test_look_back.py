"""The forward scan's look-back carry (few channel groups, the sequence cut into
chunks that run at once in one launch).

Chunk k's pair (P_k, S_k) = (Π Ā over the chunk, the state it reaches from
zero) maps the state entering the chunk to the state leaving it,
h -> P_k·h + S_k (the affine composition of "Mamba and selective state spaces,
from first principles", "The hardware-aware scan").  Each chunk finds the
state it starts from by walking back to the nearest predecessor whose leaving
state is out and carrying that state forward through the pairs in between.
The kernel promises that whichever predecessor the walk stops at, the state it
publishes is bit for bit h0 carried chunk by chunk, one fused multiply-add per
state and chunk, so that the output does not depend on timing.

These tests read the workspace after a call (its layout: a 256-byte header,
one int flag per (channel group, chunk), the pairs [b][D][K-1][N] as float2,
the carried states [b][D][K][N] as fp32, each region rounded up to 256 bytes)
and check that promise against the pairs the same launch published; then
that repeated calls agree bit for bit, and that every kernel variant the
dispatch picks matches the oracle.
"""

import numpy as np
import pytest
import torch

from mamba_selective_scan_02_b300 import api, capi
from ssm_testutil import assert_close
from oracle import oracle as orc

pytestmark = pytest.mark.gpu


def _al(n):
    return -(-n // 256) * 256


def _inputs(b, D, N, L, dtype, seed, zoh_safe=False, gate=True, init=True):
    g = torch.Generator().manual_seed(seed)

    def rn(*s, std=1.0):
        return (torch.randn(*s, generator=g) * std).to(dtype)
    A = -torch.rand(D, N, generator=g).add_(0.5)
    if zoh_safe:
        A = A - 0.1
    return dict(u=rn(b, D, L), delta=rn(b, D, L, std=0.5), z=rn(b, D, L) if gate else None, B=rn(b, N, L),
                C=rn(b, N, L), A=A, Dskip=torch.randn(D, generator=g),
                bias=torch.log(torch.expm1(torch.empty(D).uniform_(1e-3, 1e-1, generator=g))).float(),
                h0=torch.randn(b, D, N, generator=g) * 0.5 if init else None)


def _run(inp, chunk_len, zoh=False):
    d = {k: (v.cuda().contiguous() if v is not None else None) for k, v in inp.items()}
    b, D, L = d["u"].shape
    N = d["B"].shape[1]
    y = torch.empty_like(d["u"])
    hL = torch.empty(b, D, N, dtype=torch.float32, device="cuda")
    ws = torch.empty(api.workspace_bytes(d["u"], d["delta"], d["A"], d["B"], d["C"], chunk_len, zoh),
                     dtype=torch.uint8, device="cuda")
    ws.fill_(0xA5)   # stale bytes: the call must clear what it relies on
    p = api.scan_params(d["u"], d["delta"], d["A"], d["B"], d["C"], d["Dskip"], d["z"], d["bias"], d["h0"],
                        y=y, hL=hL, zoh=zoh, chunk_len=chunk_len, workspace=ws)
    plan = capi.ssm_scan_plan(p)
    capi.check(capi.ssm_scan_fwd(p, torch.cuda.current_stream().cuda_stream), "ssm_scan_fwd")
    assert api.workspace_status(ws) == capi.SSM_OK
    return y, hL, ws.cpu().numpy(), plan


# (b, D, N, L, dtype, chunk_len, zoh[, gate, h0]): each a look-back plan of a
# different kernel or edge
CASES = [
    (1, 20, 16, 641, torch.bfloat16, 64, False, False, False),  # plain loads, last chunk one token, no z, no h0
    (1, 20, 16, 648, torch.bfloat16, 64, False, False, False),  # warp-specialised, last chunk one 8-token tile
    (2, 8, 5, 129, torch.float32, 64, False, True, False),      # fp32, last chunk one token, h0 = 0
    (1, 32, 16, 700, torch.bfloat16, 64, False),     # warp-specialised, 11 chunks, ragged last chunk
    (2, 48, 16, 4096, torch.bfloat16, 64, False),    # warp-specialised, 64 chunks (the most the plan cuts)
    (2, 24, 5, 173, torch.float32, 64, False),       # fp32, 8 states per lane
    (1, 40, 16, 520, torch.float32, 128, False),     # fp32, two lanes per channel
    (1, 36, 4, 300, torch.bfloat16, 64, False),      # bf16, 4 states
    (1, 33, 16, 330, torch.bfloat16, 64, False),     # row pitch not 16-B aligned: plain loads
    (2, 32, 16, 512, torch.bfloat16, 128, True),     # exact zero-order hold
]


@pytest.mark.parametrize("case", CASES)
def test_carried_states_are_the_sequential_chain(case):
    b, D, N, L, dtype, chunk, zoh = case[:7]
    gate, init = case[7:9] if len(case) > 7 else (True, True)
    inp = _inputs(b, D, N, L, dtype, seed=b * 7 + D + N + L, zoh_safe=zoh, gate=gate, init=init)
    y, hL, ws, plan = _run(inp, chunk, zoh)
    K, G = plan["nchunks"], plan["groups"]
    assert not plan["chained"] and K == -(-L // chunk) and K > 1
    off = 256
    flags = ws[off:off + G * K * 4].view(np.int32).reshape(G, K)
    off += _al(G * K * 4)
    agg = ws[off:off + b * D * (K - 1) * N * 8].view(np.float32).reshape(b, D, K - 1, N, 2)
    off += _al(b * D * (K - 1) * N * 8)
    carry = ws[off:off + b * D * K * N * 4].view(np.float32).reshape(b, D, K, N)
    # every chunk but the last published its pair and then its leaving state
    assert (flags[:, :K - 1] == 2).all() and (flags[:, K - 1] == 0).all()
    # the chain from h0: h_{k+1} = fma(P_k, h_k, S_k) in fp32.  The product of two
    # floats is exact in fp64 and the sum is rounded once there, then to fp32: the
    # same value as the fp32 fma unless the fp64 sum lands on an fp32 rounding
    # midpoint, which these few thousand steps do not.
    h = (inp["h0"] if inp["h0"] is not None else torch.zeros(b, D, N)).numpy().astype(np.float32)
    for k in range(K - 1):
        P, S = agg[:, :, k, :, 0], agg[:, :, k, :, 1]
        assert np.isfinite(P).all() and np.isfinite(S).all() and (P >= 0).all() and (P <= 1).all()
        h = (P.astype(np.float64) * h.astype(np.float64) + S.astype(np.float64)).astype(np.float32)
        assert np.array_equal(carry[:, :, k + 1].view(np.int32), h.view(np.int32)), \
            f"chunk {k}: the published leaving state is not the sequential chain"
    # and the outputs are the method's
    y_ref, h_ref = orc.scan(inp["u"], inp["delta"], inp["A"], inp["B"], inp["C"], Dskip=inp["Dskip"], z=inp["z"],
                            bias=inp["bias"], h0=inp["h0"], zoh=zoh, threads=8)
    assert_close(y.double().cpu().numpy(), y_ref, dtype, "look-back y")
    assert_close(hL.double().cpu().numpy(), h_ref, dtype, "look-back hL")


def test_repeated_calls_agree_bit_for_bit():
    """64 chunks of 2 groups: the walks stop at different predecessors from one
    call to the next, and the outputs may not change."""
    inp = _inputs(1, 32, 16, 4096, torch.bfloat16, seed=77)
    y0, h0, _, plan = _run(inp, 64)
    assert plan["nchunks"] == 64 and not plan["chained"]
    for _ in range(6):
        y1, h1, _, _ = _run(inp, 64)
        assert torch.equal(y0, y1) and torch.equal(h0, h1)


def test_look_back_beside_other_work():
    """The look-back launch while another stream keeps SMs busy: a wait never
    reaches its bound, and the result is unchanged."""
    inp = _inputs(2, 48, 16, 2048, torch.bfloat16, seed=5)
    y0, h0, _, _ = _run(inp, 64)
    side = torch.cuda.Stream()
    a = torch.randn(4096, 4096, device="cuda")
    with torch.cuda.stream(side):
        for _ in range(4):
            a = a @ a.T
            a = a / a.norm()
    y1, h1, _, _ = _run(inp, 64)
    torch.cuda.synchronize()
    assert torch.equal(y0, y1) and torch.equal(h0, h1)
