"""ctypes wrapper around the fp64 C oracle (test infrastructure only).

Every array crosses as a C-contiguous float64 numpy array; ``None`` stands for
the NULL pointers the C side accepts (no gate, zero skip, zero bias, zero
initial state).  The arithmetic lives entirely in ``ssm_oracle.c``.
"""

from __future__ import annotations

import ctypes
import os
import subprocess
from concurrent.futures import ThreadPoolExecutor

import numpy as np

_HERE = os.path.dirname(os.path.abspath(__file__))
_SRC = os.path.join(_HERE, "ssm_oracle.c")
_LIB = os.path.join(_HERE, "libssm_oracle.so")
_lib = None

_D = ctypes.POINTER(ctypes.c_double)
_I64 = ctypes.c_int64


def source_path() -> str:
    return _SRC


def build(src: str = _SRC, out: str = _LIB, force: bool = False) -> str:
    """Compile the oracle with gcc (IEEE fp64, no fast-math).  Returns the .so path."""
    if force or not os.path.exists(out) or os.path.getmtime(out) < os.path.getmtime(src):
        tmp = out + ".tmp%d" % os.getpid()
        subprocess.run(["gcc", "-O2", "-std=c99", "-fPIC", "-shared", "-o", tmp, src, "-lm"],
                       check=True)
        os.replace(tmp, out)
    return out


def load(path: str | None = None):
    """Load (building first if needed) and return the ctypes library."""
    global _lib
    if path is not None:
        return _bind(ctypes.CDLL(path))
    if _lib is None:
        _lib = _bind(ctypes.CDLL(build()))
    return _lib


def _bind(lib):
    lib.oracle_scan.restype = ctypes.c_int
    lib.oracle_scan.argtypes = [_I64, _I64, _I64, _I64,
                                _D, _D, _D, _D, _D, _D, _D, _D,
                                ctypes.c_int, ctypes.c_int, _D, _D, _D, _I64, _I64]
    lib.oracle_conv1d.restype = ctypes.c_int
    lib.oracle_conv1d.argtypes = [_I64, _I64, _I64, _I64, _D, _D, _D, ctypes.c_int, _D, _D, _D]
    lib.oracle_conv1d_step.restype = ctypes.c_int
    lib.oracle_conv1d_step.argtypes = [_I64, _I64, _I64, _D, _D, _D, _D, ctypes.c_int, _D]
    lib.oracle_scan_bwd.restype = ctypes.c_int
    lib.oracle_scan_bwd.argtypes = [_I64, _I64, _I64, _I64,
                                    _D, _D, _D, _D, _D, _D, _D, _D,
                                    ctypes.c_int, ctypes.c_int, _D, _D, _D,
                                    _D, _D, _D, _D, _D, _D, _D, _D, _D, _I64, _I64]
    lib.oracle_ssd.restype = ctypes.c_int
    lib.oracle_ssd.argtypes = [_I64, _I64, _I64, _I64, _I64, _D, _D, _D, _D, _D, _D, _D,
                               ctypes.c_int, _D, _D, _D]
    lib.oracle_step.restype = ctypes.c_int
    lib.oracle_step.argtypes = [_I64, _I64, _I64,
                                _D, _D, _D, _D, _D, _D, _D, _D, _D,
                                ctypes.c_int, ctypes.c_int, _D]
    return lib


def _f64(a):
    if a is None:
        return None
    if hasattr(a, "detach"):  # torch tensor
        a = a.detach().to("cpu").double().numpy()
    return np.ascontiguousarray(a, dtype=np.float64)


def _p(a):
    return None if a is None else a.ctypes.data_as(_D)


def scan(u, delta, A, B, C, Dskip=None, z=None, bias=None, h0=None,
         delta_softplus=True, zoh=False, threads: int = 1, lib=None):
    """Forward scan.  u, delta, z: (b, D, L); B, C: (b, N, L); A: (D, N);
    Dskip, bias: (D,); h0: (b, D, N).  Returns (y (b, D, L), hL (b, D, N)) in fp64.

    ``threads`` > 1 splits the independent (b, d) channels over host threads; each
    thread runs the unchanged sequential oracle on its own channel range."""
    lib = lib or load()
    u, delta, z, B, C, A, Dskip, bias, h0 = map(_f64, (u, delta, z, B, C, A, Dskip, bias, h0))
    b, dim, L = u.shape
    N = A.shape[1]
    assert delta.shape == u.shape and B.shape == (b, N, L) and C.shape == (b, N, L)
    assert z is None or z.shape == u.shape
    y = np.empty((b, dim, L), np.float64)
    hL = np.empty((b, dim, N), np.float64)
    nch = b * dim

    def run(c0, c1):
        rc = lib.oracle_scan(b, dim, N, L, _p(u), _p(delta), _p(z), _p(B), _p(C), _p(A),
                             _p(Dskip), _p(bias), int(bool(delta_softplus)), int(bool(zoh)),
                             _p(h0), _p(y), _p(hL), c0, c1)
        if rc != 0:
            raise RuntimeError("oracle_scan failed")

    if threads <= 1 or nch < 2:
        run(0, nch)
    else:
        bounds = np.linspace(0, nch, min(threads, nch) + 1).astype(np.int64)
        with ThreadPoolExecutor(len(bounds) - 1) as ex:
            list(ex.map(lambda i: run(int(bounds[i]), int(bounds[i + 1])), range(len(bounds) - 1)))
    return y, hL


def scan_channels(channels, u, delta, A, B, C, Dskip=None, z=None, bias=None, h0=None,
                  delta_softplus=True, zoh=False, lib=None):
    """Oracle on a sample of (b, d) channels of a large problem.

    ``channels`` is a list of (b, d).  Only those rows are widened to fp64, so the
    inputs may be multi-GB torch/numpy arrays.  Returns lists of y rows (L,) and
    final states (N,)."""
    ys, hs = [], []
    for (bi, di) in channels:
        row = lambda t: None if t is None else t[bi:bi + 1, di:di + 1]
        yc, hc = scan(row(u), row(delta), A[di:di + 1], B[bi:bi + 1], C[bi:bi + 1],
                      Dskip=None if Dskip is None else Dskip[di:di + 1],
                      z=row(z), bias=None if bias is None else bias[di:di + 1],
                      h0=None if h0 is None else h0[bi:bi + 1, di:di + 1],
                      delta_softplus=delta_softplus, zoh=zoh, lib=lib)
        ys.append(yc[0, 0])
        hs.append(hc[0, 0])
    return ys, hs


def step(state, u, delta, A, B, C, Dskip=None, z=None, bias=None,
         delta_softplus=True, zoh=False, lib=None):
    """One decode token.  state: (b, D, N) fp64, updated in place (a new fp64
    array is returned if the input was not already a contiguous float64 numpy
    array).  u, delta, z: (b, D); B, C: (b, N).  Returns (y (b, D), state)."""
    lib = lib or load()
    st = _f64(state)
    u, delta, z, B, C, A, Dskip, bias = map(_f64, (u, delta, z, B, C, A, Dskip, bias))
    b, dim, N = st.shape
    assert u.shape == (b, dim) and B.shape == (b, N) and A.shape == (dim, N)
    y = np.empty((b, dim), np.float64)
    rc = lib.oracle_step(b, dim, N, _p(st), _p(u), _p(delta), _p(z), _p(B), _p(C), _p(A),
                         _p(Dskip), _p(bias), int(bool(delta_softplus)), int(bool(zoh)), _p(y))
    if rc != 0:
        raise RuntimeError("oracle_step failed")
    return y, st


def conv1d(x, w, bias=None, state_in=None, silu=True, lib=None):
    """Causal depthwise convolution (+ bias, + SiLU).  x: (b, D, L); w: (D, W);
    bias: (D,); state_in: (b, D, W-1), oldest first.  Returns (u (b, D, L),
    state_out (b, D, W-1)) in fp64."""
    lib = lib or load()
    x, w, bias, state_in = map(_f64, (x, w, bias, state_in))
    b, dim, L = x.shape
    W = w.shape[1]
    assert w.shape == (dim, W) and (state_in is None or state_in.shape == (b, dim, W - 1))
    u = np.empty((b, dim, L), np.float64)
    st = np.empty((b, dim, W - 1), np.float64)
    rc = lib.oracle_conv1d(b, dim, L, W, _p(x), _p(w), _p(bias), int(bool(silu)),
                           _p(state_in), _p(u), _p(st))
    if rc != 0:
        raise RuntimeError("oracle_conv1d failed")
    return u, st


def conv1d_step(state, x, w, bias=None, silu=True, lib=None):
    """One decode token of the convolution.  state: (b, D, W-1) fp64, updated in
    place (a new array is returned if it was not contiguous float64 numpy);
    x: (b, D).  Returns (u (b, D), state)."""
    lib = lib or load()
    st = _f64(state)
    x, w, bias = map(_f64, (x, w, bias))
    b, dim = x.shape
    W = w.shape[1]
    assert st.shape == (b, dim, W - 1) and w.shape == (dim, W)
    u = np.empty((b, dim), np.float64)
    rc = lib.oracle_conv1d_step(b, dim, W, _p(st), _p(x), _p(w), _p(bias), int(bool(silu)), _p(u))
    if rc != 0:
        raise RuntimeError("oracle_conv1d_step failed")
    return u, st


def scan_bwd(u, delta, A, B, C, dy, Dskip=None, z=None, bias=None, h0=None, dhL=None,
             delta_softplus=True, zoh=False, threads: int = 1, lib=None):
    """Gradient of the forward scan for upstream gradients dy (b, D, L) and dhL
    (b, D, N) or None.  Returns a dict of fp64 arrays: du, ddelta, dz (None
    without z), dB, dC, dA, dDskip, dbias, dh0 (None without h0).

    ``threads`` > 1 splits the (b, d) channels over host threads; each range
    adds into its own dB, dC, dA, dDskip, dbias buffers, summed at the end."""
    lib = lib or load()
    u, delta, z, B, C, A, Dskip, bias, h0, dy, dhL = map(
        _f64, (u, delta, z, B, C, A, Dskip, bias, h0, dy, dhL))
    b, dim, L = u.shape
    N = A.shape[1]
    assert dy.shape == u.shape and B.shape == (b, N, L) and C.shape == (b, N, L)
    du = np.empty((b, dim, L))
    ddelta = np.empty((b, dim, L))
    dz = np.empty((b, dim, L)) if z is not None else None
    dh0 = np.empty((b, dim, N)) if h0 is not None else None
    nch = b * dim
    bounds = np.linspace(0, nch, max(1, min(threads, nch)) + 1).astype(np.int64)
    parts = []

    def run(i):
        acc = dict(dB=np.zeros((b, N, L)), dC=np.zeros((b, N, L)), dA=np.zeros((dim, N)),
                   dDskip=np.zeros(dim), dbias=np.zeros(dim))
        rc = lib.oracle_scan_bwd(b, dim, N, L, _p(u), _p(delta), _p(z), _p(B), _p(C), _p(A),
                                 _p(Dskip), _p(bias), int(bool(delta_softplus)), int(bool(zoh)),
                                 _p(h0), _p(dy), _p(dhL), _p(du), _p(ddelta), _p(dz),
                                 _p(acc["dB"]), _p(acc["dC"]), _p(acc["dA"]), _p(acc["dDskip"]),
                                 _p(acc["dbias"]), _p(dh0), int(bounds[i]), int(bounds[i + 1]))
        if rc != 0:
            raise RuntimeError("oracle_scan_bwd failed")
        return acc

    if len(bounds) == 2:
        parts = [run(0)]
    else:
        with ThreadPoolExecutor(len(bounds) - 1) as ex:
            parts = list(ex.map(run, range(len(bounds) - 1)))
    out = {k: sum(p[k] for p in parts) for k in parts[0]}
    out.update(du=du, ddelta=ddelta, dz=dz, dh0=dh0)
    return out


def ssd(x, dt, A, B, C, Dskip=None, dt_bias=None, h0=None, dt_softplus=True, lib=None):
    """Mamba-2 (SSD) forward.  x: (b, L, H, P); dt: (b, L, H); A, Dskip, dt_bias:
    (H,); B, C: (b, L, N); h0: (b, H, P, N).  Returns (y (b, L, H, P), hL
    (b, H, P, N)) in fp64."""
    lib = lib or load()
    x, dt, A, B, C, Dskip, dt_bias, h0 = map(_f64, (x, dt, A, B, C, Dskip, dt_bias, h0))
    b, L, H, P = x.shape
    N = B.shape[2]
    assert dt.shape == (b, L, H) and B.shape == (b, L, N) and C.shape == (b, L, N) and A.shape == (H,)
    y = np.empty((b, L, H, P))
    hL = np.empty((b, H, P, N))
    rc = lib.oracle_ssd(b, L, H, P, N, _p(x), _p(dt), _p(A), _p(B), _p(C), _p(Dskip), _p(dt_bias),
                        int(bool(dt_softplus)), _p(h0), _p(y), _p(hL))
    if rc != 0:
        raise RuntimeError("oracle_ssd failed")
    return y, hL
