"""ctypes view of libssmscan's C ABI (include/ssm_scan.h).

Structs and prototypes mirror the header one to one.  The library is opened on
first use from this package's ``lib/`` directory; if it is missing it is built
in-tree with nvcc, and if that fails the call raises — there is no fallback.
With the environment variable SSM_SCAN_LIBRARY=debug the process opens the
debug build instead (index checks on every store, see ssm_debug_status).
"""

from __future__ import annotations

import ctypes
import os
import threading

from . import build as _build

SSM_OK, SSM_ERR_INVALID_ARG, SSM_ERR_UNSUPPORTED, SSM_ERR_CUDA, SSM_ERR_TIMEOUT, SSM_ERR_BOUNDS = range(6)
SSM_F32, SSM_BF16 = 0, 1
SSM_MAX_DSTATE = 16
SSM_MAX_CONV_WIDTH = 4
SSM_NOALLOC_SCRATCH_BYTES = 16 << 20

_vp = ctypes.c_void_p
_i64 = ctypes.c_int64


class ScanParams(ctypes.Structure):
    _fields_ = [
        ("batch", _i64), ("dim", _i64), ("dstate", _i64), ("seqlen", _i64),
        ("io_dtype", ctypes.c_int),
        ("u", _vp), ("delta", _vp), ("z", _vp), ("B", _vp), ("C", _vp),
        ("A", _vp), ("Dskip", _vp), ("delta_bias", _vp),
        ("delta_softplus", ctypes.c_int), ("zoh", ctypes.c_int),
        ("h0", _vp), ("y", _vp), ("hL", _vp),
        ("workspace", _vp), ("workspace_bytes", ctypes.c_size_t),
        ("chunk_len", _i64),
    ]


class StepParams(ctypes.Structure):
    _fields_ = [
        ("batch", _i64), ("dim", _i64), ("dstate", _i64),
        ("io_dtype", ctypes.c_int),
        ("state", _vp), ("u", _vp), ("delta", _vp), ("z", _vp), ("B", _vp), ("C", _vp),
        ("A", _vp), ("Dskip", _vp), ("delta_bias", _vp),
        ("delta_softplus", ctypes.c_int), ("zoh", ctypes.c_int),
        ("y", _vp),
    ]


class BwdParams(ctypes.Structure):
    _fields_ = [
        ("batch", _i64), ("dim", _i64), ("dstate", _i64), ("seqlen", _i64),
        ("io_dtype", ctypes.c_int),
        ("u", _vp), ("delta", _vp), ("z", _vp), ("B", _vp), ("C", _vp),
        ("A", _vp), ("Dskip", _vp), ("delta_bias", _vp),
        ("delta_softplus", ctypes.c_int), ("zoh", ctypes.c_int),
        ("h0", _vp), ("dy", _vp), ("dhL", _vp),
        ("du", _vp), ("ddelta", _vp), ("dz", _vp), ("dB", _vp), ("dC", _vp), ("dA", _vp),
        ("dDskip", _vp), ("ddelta_bias", _vp), ("dh0", _vp),
        ("workspace", _vp), ("workspace_bytes", ctypes.c_size_t),
        ("chunk_len", _i64),
    ]


class SsdParams(ctypes.Structure):
    _fields_ = [
        ("batch", _i64), ("seqlen", _i64), ("nheads", _i64), ("headdim", _i64), ("dstate", _i64),
        ("io_dtype", ctypes.c_int),
        ("x", _vp), ("dt", _vp), ("A", _vp), ("B", _vp), ("C", _vp),
        ("Dskip", _vp), ("dt_bias", _vp), ("dt_softplus", ctypes.c_int),
        ("h0", _vp), ("y", _vp), ("hL", _vp), ("status", _vp),
        ("workspace", _vp), ("workspace_bytes", ctypes.c_size_t),
    ]


class ConvParams(ctypes.Structure):
    _fields_ = [
        ("batch", _i64), ("dim", _i64), ("seqlen", _i64), ("width", _i64),
        ("io_dtype", ctypes.c_int),
        ("x", _vp), ("weight", _vp), ("bias", _vp), ("silu", ctypes.c_int),
        ("state_in", _vp), ("u", _vp), ("state_out", _vp),
    ]


class ConvStepParams(ctypes.Structure):
    _fields_ = [
        ("batch", _i64), ("dim", _i64), ("width", _i64),
        ("io_dtype", ctypes.c_int),
        ("state", _vp), ("x", _vp), ("weight", _vp), ("bias", _vp), ("silu", ctypes.c_int),
        ("u", _vp),
    ]


_lock = threading.Lock()
_lib = None


def debug_selected() -> bool:
    return os.environ.get("SSM_SCAN_LIBRARY", "") == "debug"


def library_path() -> str:
    return _build.LIB_DEBUG if debug_selected() else _build.LIB


def lib():
    """The loaded library (built in-tree first if absent or stale)."""
    global _lib
    if _lib is not None:
        return _lib
    with _lock:
        if _lib is None:
            debug = debug_selected()
            path = library_path()
            if _build.stale(path):
                _build.build(debug=debug)
            if not os.path.exists(path):
                raise RuntimeError(f"libssmscan is missing at {path} and could not be built")
            L = ctypes.CDLL(path)
            L.ssm_scan_workspace_size.restype = ctypes.c_size_t
            L.ssm_scan_workspace_size.argtypes = [ctypes.POINTER(ScanParams)]
            L.ssm_scan_plan.restype = ctypes.c_int
            L.ssm_scan_plan.argtypes = [ctypes.POINTER(ScanParams), ctypes.POINTER(_i64)]
            L.ssm_scan_fwd.restype = ctypes.c_int
            L.ssm_scan_fwd.argtypes = [ctypes.POINTER(ScanParams), _vp]
            L.ssm_scan_fwd_noalloc.restype = ctypes.c_int
            L.ssm_scan_fwd_noalloc.argtypes = [ctypes.POINTER(ScanParams), _vp]
            L.ssm_state_update.restype = ctypes.c_int
            L.ssm_state_update.argtypes = [ctypes.POINTER(StepParams), _vp]
            L.ssm_scan_bwd_workspace_size.restype = ctypes.c_size_t
            L.ssm_scan_bwd_workspace_size.argtypes = [ctypes.POINTER(BwdParams)]
            L.ssm_scan_bwd.restype = ctypes.c_int
            L.ssm_scan_bwd.argtypes = [ctypes.POINTER(BwdParams), _vp]
            L.ssm_ssd_workspace_size.restype = ctypes.c_size_t
            L.ssm_ssd_workspace_size.argtypes = [ctypes.POINTER(SsdParams)]
            L.ssm_ssd_fwd.restype = ctypes.c_int
            L.ssm_ssd_fwd.argtypes = [ctypes.POINTER(SsdParams), _vp]
            L.ssm_conv1d_fwd.restype = ctypes.c_int
            L.ssm_conv1d_fwd.argtypes = [ctypes.POINTER(ConvParams), _vp]
            L.ssm_conv1d_step.restype = ctypes.c_int
            L.ssm_conv1d_step.argtypes = [ctypes.POINTER(ConvStepParams), _vp]
            L.ssm_workspace_status.restype = ctypes.c_int
            L.ssm_workspace_status.argtypes = [_vp, _vp]
            L.ssm_status_string.restype = ctypes.c_char_p
            L.ssm_status_string.argtypes = [ctypes.c_int]
            L.ssm_bench_mufu_ex2.restype = ctypes.c_int
            L.ssm_bench_mufu_ex2.argtypes = [_vp, ctypes.c_int, ctypes.c_int, _vp]
            L.ssm_selftest_flag_wait.restype = ctypes.c_int
            L.ssm_selftest_flag_wait.argtypes = [_vp, ctypes.c_size_t, ctypes.c_int, _vp]
            L.ssm_version.restype = ctypes.c_char_p
            L.ssm_version.argtypes = []
            L.ssm_debug_status.restype = ctypes.c_int
            L.ssm_debug_status.argtypes = [ctypes.c_int]
            _lib = L
    return _lib


def ssm_debug_status(reset: bool = False) -> int:
    return lib().ssm_debug_status(int(reset))


def status_string(code: int) -> str:
    return lib().ssm_status_string(code).decode()


class SSMError(RuntimeError):
    def __init__(self, code: int, where: str):
        super().__init__(f"{where}: {status_string(code)} (status {code})")
        self.code = code


def check(code: int, where: str) -> None:
    if code != SSM_OK:
        raise SSMError(code, where)


def ssm_scan_workspace_size(p: ScanParams) -> int:
    return lib().ssm_scan_workspace_size(ctypes.byref(p))


def ssm_scan_plan(p: ScanParams) -> dict:
    """The scan's work split: chunk_len, nchunks, chained, groups."""
    out = (_i64 * 4)()
    check(lib().ssm_scan_plan(ctypes.byref(p), out), "ssm_scan_plan")
    return {"chunk_len": out[0], "nchunks": out[1], "chained": bool(out[2]), "groups": out[3]}


def ssm_scan_fwd(p: ScanParams, stream: int) -> int:
    return lib().ssm_scan_fwd(ctypes.byref(p), stream)


def ssm_scan_fwd_noalloc(p: ScanParams, stream: int) -> int:
    return lib().ssm_scan_fwd_noalloc(ctypes.byref(p), stream)


def ssm_state_update(p: StepParams, stream: int) -> int:
    return lib().ssm_state_update(ctypes.byref(p), stream)


def ssm_scan_bwd_workspace_size(p: BwdParams) -> int:
    return lib().ssm_scan_bwd_workspace_size(ctypes.byref(p))


def ssm_scan_bwd(p: BwdParams, stream: int) -> int:
    return lib().ssm_scan_bwd(ctypes.byref(p), stream)


def ssm_ssd_workspace_size(p: SsdParams) -> int:
    return lib().ssm_ssd_workspace_size(ctypes.byref(p))


def ssm_ssd_fwd(p: SsdParams, stream: int) -> int:
    return lib().ssm_ssd_fwd(ctypes.byref(p), stream)


def ssm_conv1d_fwd(p: ConvParams, stream: int) -> int:
    return lib().ssm_conv1d_fwd(ctypes.byref(p), stream)


def ssm_conv1d_step(p: ConvStepParams, stream: int) -> int:
    return lib().ssm_conv1d_step(ctypes.byref(p), stream)


def ssm_workspace_status(workspace: int, stream: int) -> int:
    return lib().ssm_workspace_status(workspace, stream)


def ssm_bench_mufu_ex2(sink: int, blocks: int, iters: int, stream: int) -> int:
    return lib().ssm_bench_mufu_ex2(sink, blocks, iters, stream)


def ssm_selftest_flag_wait(workspace: int, nbytes: int, polls: int, stream: int) -> int:
    return lib().ssm_selftest_flag_wait(workspace, nbytes, polls, stream)
