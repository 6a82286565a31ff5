"""Small calls of every entry point, shared by the debug-build test.

``run_cases()`` returns every output as a CPU tensor, keyed by case.  Run as a
script with SSM_SCAN_LIBRARY=debug, it does the same against the debug build
of the library (index checks on every store), reads the build's debug status
before and after, and saves both to the path given as its argument; the test
then compares those outputs with the release library's.
"""

from __future__ import annotations

import os
import sys

import torch

HERE = os.path.dirname(os.path.abspath(__file__))
ROOT = os.path.dirname(HERE)
if ROOT not in sys.path:
    sys.path.insert(0, ROOT)

from mamba_selective_scan_02_b300 import api  # noqa: E402
from mamba_selective_scan_02_b300.inputs import make_ssd_inputs  # noqa: E402


def _rn(g, *shape, std=1.0, dtype=torch.float32):
    return (torch.randn(*shape, generator=g) * std).to(dtype).cuda()


def _scan_inputs(g, b, D, N, L, dtype):
    return dict(u=_rn(g, b, D, L, dtype=dtype), delta=_rn(g, b, D, L, std=0.5, dtype=dtype),
                z=_rn(g, b, D, L, dtype=dtype), B=_rn(g, b, N, L, dtype=dtype), C=_rn(g, b, N, L, dtype=dtype),
                A=-torch.rand(D, N, generator=g).add_(0.5).cuda(), Dskip=_rn(g, D),
                bias=torch.log(torch.expm1(torch.empty(D).uniform_(1e-3, 1e-1, generator=g))).float().cuda(),
                h0=_rn(g, b, D, N, std=0.5))


# (name, batch, dim, dstate, seqlen, dtype, chunk_len): the fp32 kernel, the
# warp-specialised bf16 kernel with a chained plan and with a look-back plan
SCANS = [("scan_f32", 2, 24, 5, 173, torch.float32, 0),
         ("scan_bf16_chained", 2, 1200, 16, 300, torch.bfloat16, 64),
         ("scan_bf16_look_back", 1, 32, 16, 700, torch.bfloat16, 64)]
STEPS = [("step_general", 3, 37, 5, torch.float32), ("step_16", 2, 96, 16, torch.bfloat16),
         ("step_stream", 2, 256, 16, torch.bfloat16)]
CONVS = [("conv_rows", 2, 24, 203, 4, torch.bfloat16), ("conv_stream", 2, 40, 512, 4, torch.bfloat16)]
CONV_STEPS = [("conv_step8", 5, 64, 4, torch.bfloat16), ("conv_step1", 3, 21, 4, torch.float32)]
BWDS = [("bwd_bf16", 2, 48, 16, 300, torch.bfloat16), ("bwd_f32", 1, 33, 7, 150, torch.float32)]
SSDS = [("ssd_ragged", 2, 300, 3)]


def run_cases() -> dict:
    out = {}
    for name, b, D, N, L, dt, ck in SCANS:
        g = torch.Generator().manual_seed(sum(map(ord, name)))
        s = _scan_inputs(g, b, D, N, L, dt)
        y, hL = api.scan_fwd(s["u"], s["delta"], s["A"], s["B"], s["C"], s["Dskip"], s["z"], s["bias"], s["h0"],
                             chunk_len=ck)
        out[name] = {"y": y, "hL": hL}
    for name, b, D, N, dt in STEPS:
        g = torch.Generator().manual_seed(len(name) + D)
        s = _scan_inputs(g, b, D, N, 1, dt)
        st = _rn(g, b, D, N)
        y = api.state_update(st, s["u"][..., 0].contiguous(), s["delta"][..., 0].contiguous(), s["A"],
                             s["B"][..., 0].contiguous(), s["C"][..., 0].contiguous(), s["Dskip"],
                             s["z"][..., 0].contiguous(), s["bias"])
        out[name] = {"y": y, "state": st}
    for name, b, D, L, W, dt in CONVS:
        g = torch.Generator().manual_seed(L + W)
        x, w, bias, s_in = _rn(g, b, D, L, dtype=dt), _rn(g, D, W), _rn(g, D, std=0.1), _rn(g, b, D, W - 1, dtype=dt)
        u, so = api.conv1d(x, w, bias, s_in)
        out[name] = {"u": u, "state_out": so}
    for name, b, D, W, dt in CONV_STEPS:
        g = torch.Generator().manual_seed(D + W)
        x, w, bias, st = _rn(g, b, D, dtype=dt), _rn(g, D, W), _rn(g, D, std=0.1), _rn(g, b, D, W - 1, dtype=dt)
        u = api.conv1d_step(st, x, w, bias)
        out[name] = {"u": u, "state": st}
    for name, b, D, N, L, dt in BWDS:
        g = torch.Generator().manual_seed(D * N + L)
        s = _scan_inputs(g, b, D, N, L, dt)
        dy, dhL = _rn(g, b, D, L, dtype=dt), _rn(g, b, D, N, std=0.5)
        r = api.scan_bwd(s["u"], s["delta"], s["A"], s["B"], s["C"], dy, s["Dskip"], s["z"], s["bias"], s["h0"], dhL)
        out[name] = {k: v for k, v in r.items() if k != "workspace" and v is not None}
    for name, b, L, H in SSDS:
        si = make_ssd_inputs(b, L, H, seed=L + H, device="cuda", with_h0=True)
        y, hL = api.ssd_fwd(si["x"], si["dt"], si["A"], si["B"], si["C"], si["D"], si["dt_bias"], si["h0"])
        out[name] = {"y": y, "hL": hL}
    torch.cuda.synchronize()
    return {case: {k: v.cpu() for k, v in d.items()} for case, d in out.items()}


def main(path: str) -> None:
    from mamba_selective_scan_02_b300 import capi
    assert capi.debug_selected(), "run with SSM_SCAN_LIBRARY=debug"
    before = capi.ssm_debug_status(reset=True)
    outs = run_cases()
    after = capi.ssm_debug_status(reset=False)
    torch.save({"library": capi.library_path(), "before": before, "after": after, "outputs": outs}, path)


if __name__ == "__main__":
    main(sys.argv[1])
