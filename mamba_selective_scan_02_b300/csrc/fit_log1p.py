"""Fits the polynomial behind ``log1p_unit`` in ssm_device.cuh.

log1p(w) on w in [0, 1] is written as w * q(w) with q a degree-7 polynomial.
q is fitted to log1p(w)/w on 4,000 Chebyshev nodes by least squares, then
reweighted (Lawson's iteration) towards the minimax fit in relative error.
The script prints the coefficients, rounded to fp32, and the worst relative
error of fp32 Horner evaluation on a fine grid.  Run:

    python mamba_selective_scan_02_b300/csrc/fit_log1p.py
"""

import numpy as np


def fit(deg: int = 7, nodes: int = 4000, rounds: int = 200) -> np.ndarray:
    k = np.arange(nodes)
    x = 0.5 - 0.5 * np.cos(np.pi * (k + 0.5) / nodes)
    f = np.log1p(x) / x
    w = np.ones(nodes)
    V = np.vander(x, deg + 1, increasing=True)
    for _ in range(rounds):
        c, *_ = np.linalg.lstsq(V * np.sqrt(w)[:, None], f * np.sqrt(w), rcond=None)
        e = np.abs(V @ c - f) / f
        w *= e / e.max() + 1e-12
        w /= w.sum()
    return c.astype(np.float32)


def horner_fp32(c: np.ndarray, w: np.ndarray) -> np.ndarray:
    w = w.astype(np.float32)
    p = np.full_like(w, c[-1])
    for cc in c[-2::-1]:
        p = (p * w + cc).astype(np.float32)
    return (p * w).astype(np.float64)


if __name__ == "__main__":
    c = fit()
    grid = np.linspace(1e-6, 1.0, 200001)
    rel = np.abs(horner_fp32(c, grid) - np.log1p(grid)) / np.log1p(grid)
    print("coefficients (w^0 .. w^7):", ", ".join(f"{float(v)!r}f" for v in c))
    print(f"max relative error, fp32 Horner: {rel.max():.3e}")
