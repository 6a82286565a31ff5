"""Shared helpers for the GPU parity tests: run the CUDA path, run the oracle on
the same seeded inputs, compare with the tolerances of the method's contract:

  fp32 I/O:             |err| <= 1e-4 · (1 + |y|)
  bf16 I/O, fp32 state: |err| <= 2e-2 · (1 + |y|)
"""

from __future__ import annotations

import numpy as np
import torch

from oracle import oracle as orc

TOL = {torch.float32: 1e-4, torch.bfloat16: 2e-2}


def tol_for(dtype):
    return TOL[dtype]


def assert_close(got, want, dtype, what=""):
    got = np.asarray(got, dtype=np.float64)
    want = np.asarray(want, dtype=np.float64)
    assert got.shape == want.shape, (what, got.shape, want.shape)
    assert np.all(np.isfinite(got)), f"{what}: non-finite values from the GPU"
    err = np.abs(got - want)
    bound = TOL[dtype] * (1.0 + np.abs(want))
    bad = err > bound
    if bad.any():
        i = np.unravel_index(np.argmax(err / bound), err.shape)
        raise AssertionError(f"{what}: {bad.sum()} of {err.size} outside tolerance; worst at {i}: "
                             f"got {got[i]!r} want {want[i]!r} (bound {bound[i]:.3e})")
    return float((err / bound).max()) if err.size else 0.0


def to_device(inp: dict, device="cuda") -> dict:
    out = dict(inp)
    for k in ("u", "delta", "z", "B", "C", "A", "Dskip", "bias", "h0"):
        if out.get(k) is not None:
            out[k] = out[k].to(device).contiguous()
    return out


def to_host(inp: dict) -> dict:
    return {k: (v.cpu() if torch.is_tensor(v) else v) for k, v in inp.items()}


def gpu_scan(inp: dict, **kw):
    from mamba_selective_scan_02_b300 import api
    y, hL = api.scan_fwd(inp["u"], inp["delta"], inp["A"], inp["B"], inp["C"], inp.get("Dskip"),
                         inp.get("z"), inp.get("bias"), inp.get("h0"), **kw)
    torch.cuda.synchronize()
    return y, hL


def oracle_scan(inp: dict, delta_softplus=True, threads=8):
    return orc.scan(inp["u"], inp["delta"], inp["A"], inp["B"], inp["C"], Dskip=inp.get("Dskip"),
                    z=inp.get("z"), bias=inp.get("bias"), h0=inp.get("h0"),
                    delta_softplus=delta_softplus, threads=threads)


def oracle_scan_sampled(inp: dict, channels, delta_softplus=True):
    """Oracle on a few (b, d) rows of a (possibly multi-GB, device-resident) input."""
    def rows(t, bi, di):
        return None if t is None else t[bi:bi + 1, di:di + 1].cpu()
    ys, hs = [], []
    for bi, di in channels:
        y, h = orc.scan(rows(inp["u"], bi, di), rows(inp["delta"], bi, di), inp["A"][di:di + 1].cpu(),
                        inp["B"][bi:bi + 1].cpu(), inp["C"][bi:bi + 1].cpu(),
                        Dskip=None if inp.get("Dskip") is None else inp["Dskip"][di:di + 1].cpu(),
                        z=rows(inp.get("z"), bi, di),
                        bias=None if inp.get("bias") is None else inp["bias"][di:di + 1].cpu(),
                        h0=rows(inp.get("h0"), bi, di), delta_softplus=delta_softplus)
        ys.append(y[0, 0])
        hs.append(h[0, 0])
    return np.stack(ys), np.stack(hs)


def sample_channels(batch, dim, n, seed=0):
    rng = np.random.default_rng(seed)
    picks = {(0, 0), (batch - 1, dim - 1)}
    while len(picks) < min(n, batch * dim):
        picks.add((int(rng.integers(batch)), int(rng.integers(dim))))
    return sorted(picks)
