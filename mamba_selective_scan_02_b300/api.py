"""Torch-facing binding of libssmscan: argument marshalling only.

Every step of the scan runs in the CUDA library; these functions check tensor
placement, fill the C parameter structs with device pointers and the current
stream, and allocate outputs and the workspace with torch when the caller does
not pass them.  They raise if the library cannot be loaded — there is no CPU
or PyTorch fallback.
"""

from __future__ import annotations

import torch

from . import capi

_DT = {torch.float32: capi.SSM_F32, torch.bfloat16: capi.SSM_BF16}


def _ptr(t):
    return None if t is None else t.data_ptr()


def _need(t, name, shape, dtype, device):
    if t is None:
        raise ValueError(f"{name} is required")
    if not t.is_cuda or t.device != device:
        raise ValueError(f"{name} must be on {device}")
    if tuple(t.shape) != tuple(shape):
        raise ValueError(f"{name} has shape {tuple(t.shape)}, expected {tuple(shape)}")
    if t.dtype != dtype:
        raise ValueError(f"{name} has dtype {t.dtype}, expected {dtype}")
    if not t.is_contiguous():
        raise ValueError(f"{name} must be contiguous")


def _opt(t, *args):
    if t is not None:
        _need(t, *args)


def scan_params(u, delta, A, B, C, D=None, z=None, delta_bias=None, h0=None, *, y, hL=None,
                delta_softplus=True, zoh=False, chunk_len=0, workspace=None) -> capi.ScanParams:
    """Validate tensors and build the C parameter struct (workspace may be None to size it)."""
    if u.dtype not in _DT:
        raise ValueError(f"unsupported I/O dtype {u.dtype}")
    dev = u.device
    b, dim, L = u.shape
    N = A.shape[1]
    io = u.dtype
    _need(u, "u", (b, dim, L), io, dev)
    _need(delta, "delta", (b, dim, L), io, dev)
    _opt(z, "z", (b, dim, L), io, dev)
    _need(B, "B", (b, N, L), io, dev)
    _need(C, "C", (b, N, L), io, dev)
    _need(A, "A", (dim, N), torch.float32, dev)
    _opt(D, "D", (dim,), torch.float32, dev)
    _opt(delta_bias, "delta_bias", (dim,), torch.float32, dev)
    _opt(h0, "h0", (b, dim, N), torch.float32, dev)
    _need(y, "y", (b, dim, L), io, dev)
    _opt(hL, "hL", (b, dim, N), torch.float32, dev)
    p = capi.ScanParams()
    p.batch, p.dim, p.dstate, p.seqlen = b, dim, N, L
    p.io_dtype = _DT[io]
    p.u, p.delta, p.z, p.B, p.C = _ptr(u), _ptr(delta), _ptr(z), _ptr(B), _ptr(C)
    p.A, p.Dskip, p.delta_bias = _ptr(A), _ptr(D), _ptr(delta_bias)
    p.delta_softplus = int(bool(delta_softplus))
    p.zoh = int(bool(zoh))
    p.h0, p.y, p.hL = _ptr(h0), _ptr(y), _ptr(hL)
    p.chunk_len = int(chunk_len)
    if workspace is not None:
        p.workspace = workspace.data_ptr()
        p.workspace_bytes = workspace.numel() * workspace.element_size()
    return p


def workspace_bytes(u, delta, A, B, C, chunk_len=0, zoh=False) -> int:
    """Workspace bytes for a scan of these tensors: the plan, and with it the
    workspace, depends on the sizes, the I/O dtype, the discretisation and
    chunk_len."""
    p = capi.ScanParams()
    p.batch, p.dim, p.seqlen = u.shape
    p.dstate = A.shape[1]
    p.io_dtype = capi.SSM_BF16 if u.dtype == torch.bfloat16 else capi.SSM_F32
    p.zoh = 1 if zoh else 0
    p.chunk_len = int(chunk_len)
    n = capi.ssm_scan_workspace_size(p)
    if n == 0:
        raise ValueError("invalid scan sizes")
    return n


def scan_fwd(u, delta, A, B, C, D=None, z=None, delta_bias=None, h0=None, *,
             delta_softplus=True, zoh=False, y=None, hL=None, return_last_state=True,
             chunk_len=0, workspace=None, stream=None):
    """Fused selective scan on the GPU.  Returns (y, hL) (hL None if not requested)."""
    if y is None:
        y = torch.empty_like(u)
    if hL is None and return_last_state:
        hL = torch.empty((u.shape[0], u.shape[1], A.shape[1]), dtype=torch.float32, device=u.device)
    if workspace is None:
        workspace = torch.empty(workspace_bytes(u, delta, A, B, C, chunk_len, zoh), dtype=torch.uint8,
                                device=u.device)
    p = scan_params(u, delta, A, B, C, D, z, delta_bias, h0, y=y, hL=hL,
                    delta_softplus=delta_softplus, zoh=zoh, chunk_len=chunk_len, workspace=workspace)
    st = torch.cuda.current_stream(u.device).cuda_stream if stream is None else stream
    capi.check(capi.ssm_scan_fwd(p, st), "ssm_scan_fwd")
    return y, hL


def step_params(state, u, delta, A, B, C, D=None, z=None, delta_bias=None, *, y,
                delta_softplus=True, zoh=False) -> capi.StepParams:
    if u.dtype not in _DT:
        raise ValueError(f"unsupported I/O dtype {u.dtype}")
    dev = u.device
    b, dim = u.shape
    N = A.shape[1]
    io = u.dtype
    _need(state, "state", (b, dim, N), torch.float32, dev)
    _need(u, "u", (b, dim), io, dev)
    _need(delta, "delta", (b, dim), io, dev)
    _opt(z, "z", (b, dim), io, dev)
    _need(B, "B", (b, N), io, dev)
    _need(C, "C", (b, N), io, dev)
    _need(A, "A", (dim, N), torch.float32, dev)
    _opt(D, "D", (dim,), torch.float32, dev)
    _opt(delta_bias, "delta_bias", (dim,), torch.float32, dev)
    _need(y, "y", (b, dim), io, dev)
    p = capi.StepParams()
    p.batch, p.dim, p.dstate = b, dim, N
    p.io_dtype = _DT[io]
    p.state, p.u, p.delta, p.z = _ptr(state), _ptr(u), _ptr(delta), _ptr(z)
    p.B, p.C, p.A, p.Dskip, p.delta_bias = _ptr(B), _ptr(C), _ptr(A), _ptr(D), _ptr(delta_bias)
    p.delta_softplus = int(bool(delta_softplus))
    p.zoh = int(bool(zoh))
    p.y = _ptr(y)
    return p


def state_update(state, u, delta, A, B, C, D=None, z=None, delta_bias=None, *,
                 delta_softplus=True, zoh=False, y=None, stream=None):
    """One decode token: updates ``state`` (b, D, N) fp32 in place, returns y (b, D)."""
    if y is None:
        y = torch.empty_like(u)
    p = step_params(state, u, delta, A, B, C, D, z, delta_bias, y=y,
                    delta_softplus=delta_softplus, zoh=zoh)
    st = torch.cuda.current_stream(u.device).cuda_stream if stream is None else stream
    capi.check(capi.ssm_state_update(p, st), "ssm_state_update")
    return y


def bwd_params(u, delta, A, B, C, dy, D=None, z=None, delta_bias=None, h0=None, dhL=None, *,
               du, ddelta, dB, dC, dA, dz=None, dD=None, ddelta_bias=None, dh0=None,
               delta_softplus=True, zoh=False, chunk_len=0, workspace=None) -> capi.BwdParams:
    """Validate tensors and build the backward scan's C parameter struct."""
    if u.dtype not in _DT:
        raise ValueError(f"unsupported I/O dtype {u.dtype}")
    dev = u.device
    b, dim, L = u.shape
    N = A.shape[1]
    io = u.dtype
    f32 = torch.float32
    for t, name, shape, dt in ((u, "u", (b, dim, L), io), (delta, "delta", (b, dim, L), io),
                               (B, "B", (b, N, L), io), (C, "C", (b, N, L), io), (dy, "dy", (b, dim, L), io),
                               (A, "A", (dim, N), f32), (du, "du", (b, dim, L), io),
                               (ddelta, "ddelta", (b, dim, L), io), (dB, "dB", (b, N, L), f32),
                               (dC, "dC", (b, N, L), f32), (dA, "dA", (dim, N), f32)):
        _need(t, name, shape, dt, dev)
    for t, name, shape, dt in ((z, "z", (b, dim, L), io), (D, "D", (dim,), f32),
                               (delta_bias, "delta_bias", (dim,), f32), (h0, "h0", (b, dim, N), f32),
                               (dhL, "dhL", (b, dim, N), f32), (dz, "dz", (b, dim, L), io),
                               (dD, "dD", (dim,), f32), (ddelta_bias, "ddelta_bias", (dim,), f32),
                               (dh0, "dh0", (b, dim, N), f32)):
        _opt(t, name, shape, dt, dev)
    p = capi.BwdParams()
    p.batch, p.dim, p.dstate, p.seqlen = b, dim, N, L
    p.io_dtype = _DT[io]
    p.u, p.delta, p.z, p.B, p.C = _ptr(u), _ptr(delta), _ptr(z), _ptr(B), _ptr(C)
    p.A, p.Dskip, p.delta_bias = _ptr(A), _ptr(D), _ptr(delta_bias)
    p.delta_softplus = int(bool(delta_softplus))
    p.zoh = int(bool(zoh))
    p.h0, p.dy, p.dhL = _ptr(h0), _ptr(dy), _ptr(dhL)
    p.du, p.ddelta, p.dz = _ptr(du), _ptr(ddelta), _ptr(dz)
    p.dB, p.dC, p.dA = _ptr(dB), _ptr(dC), _ptr(dA)
    p.dDskip, p.ddelta_bias, p.dh0 = _ptr(dD), _ptr(ddelta_bias), _ptr(dh0)
    p.chunk_len = int(chunk_len)
    if workspace is not None:
        p.workspace = workspace.data_ptr()
        p.workspace_bytes = workspace.numel() * workspace.element_size()
    return p


def bwd_workspace_bytes(batch, dim, dstate, seqlen, chunk_len=0, dtype=torch.bfloat16, zoh=False) -> int:
    """Workspace bytes of ssm_scan_bwd.  The I/O dtype and the discretisation
    matter: bf16 first-order backward passes with enough channel groups take
    their state checkpoints from the forward scan kernel, which needs room of
    its own."""
    p = capi.BwdParams()
    p.batch, p.dim, p.dstate, p.seqlen = batch, dim, dstate, seqlen
    p.chunk_len = int(chunk_len)
    p.io_dtype = _DT[dtype]
    p.zoh = int(bool(zoh))
    n = capi.ssm_scan_bwd_workspace_size(p)
    if n == 0:
        raise ValueError("invalid backward scan sizes")
    return n


def scan_bwd(u, delta, A, B, C, dy, D=None, z=None, delta_bias=None, h0=None, dhL=None, *,
             delta_softplus=True, zoh=False, chunk_len=0, workspace=None, stream=None) -> dict:
    """Gradients of scan_fwd for upstream dy (and dhL).  Returns a dict with du,
    ddelta, dz (None without z), dB, dC, dA, dD, ddelta_bias (None when D /
    delta_bias are None) and dh0 (None without h0); dB, dC, dA, dD and
    ddelta_bias are fp32."""
    b, dim, L = u.shape
    N = A.shape[1]
    dev = u.device
    f32 = torch.float32
    out = dict(du=torch.empty_like(u), ddelta=torch.empty_like(delta),
               dz=torch.empty_like(z) if z is not None else None,
               dB=torch.empty((b, N, L), dtype=f32, device=dev), dC=torch.empty((b, N, L), dtype=f32, device=dev),
               dA=torch.empty((dim, N), dtype=f32, device=dev),
               dD=torch.empty(dim, dtype=f32, device=dev) if D is not None else None,
               ddelta_bias=torch.empty(dim, dtype=f32, device=dev) if delta_bias is not None else None,
               dh0=torch.empty((b, dim, N), dtype=f32, device=dev) if h0 is not None else None)
    if workspace is None:
        workspace = torch.empty(bwd_workspace_bytes(b, dim, N, L, chunk_len, u.dtype, zoh), dtype=torch.uint8,
                                device=dev)
    p = bwd_params(u, delta, A, B, C, dy, D, z, delta_bias, h0, dhL, du=out["du"], ddelta=out["ddelta"],
                   dB=out["dB"], dC=out["dC"], dA=out["dA"], dz=out["dz"], dD=out["dD"],
                   ddelta_bias=out["ddelta_bias"], dh0=out["dh0"], delta_softplus=delta_softplus, zoh=zoh,
                   chunk_len=chunk_len, workspace=workspace)
    st = torch.cuda.current_stream(dev).cuda_stream if stream is None else stream
    capi.check(capi.ssm_scan_bwd(p, st), "ssm_scan_bwd")
    out["workspace"] = workspace
    return out


def ssd_params(x, dt, A, B, C, D=None, dt_bias=None, h0=None, *, y, hL=None,
               dt_softplus=True, status=None, workspace=None) -> capi.SsdParams:
    """Validate tensors and build the Mamba-2 scan's C parameter struct."""
    if x.dtype not in _DT:
        raise ValueError(f"unsupported I/O dtype {x.dtype}")
    dev = x.device
    b, L, H, P = x.shape
    N = B.shape[2]
    io = x.dtype
    f32 = torch.float32
    _need(x, "x", (b, L, H, P), io, dev)
    _need(dt, "dt", (b, L, H), io, dev)
    _need(A, "A", (H,), f32, dev)
    _need(B, "B", (b, L, N), io, dev)
    _need(C, "C", (b, L, N), io, dev)
    _opt(D, "D", (H,), f32, dev)
    _opt(dt_bias, "dt_bias", (H,), f32, dev)
    _opt(h0, "h0", (b, H, P, N), f32, dev)
    _need(y, "y", (b, L, H, P), io, dev)
    _opt(hL, "hL", (b, H, P, N), f32, dev)
    _opt(status, "status", (1,), torch.int32, dev)
    p = capi.SsdParams()
    p.batch, p.seqlen, p.nheads, p.headdim, p.dstate = b, L, H, P, N
    p.io_dtype = _DT[io]
    p.x, p.dt, p.A, p.B, p.C = _ptr(x), _ptr(dt), _ptr(A), _ptr(B), _ptr(C)
    p.Dskip, p.dt_bias, p.dt_softplus = _ptr(D), _ptr(dt_bias), int(bool(dt_softplus))
    p.h0, p.y, p.hL, p.status = _ptr(h0), _ptr(y), _ptr(hL), _ptr(status)
    if workspace is not None:
        p.workspace = workspace.data_ptr()
        p.workspace_bytes = workspace.numel() * workspace.element_size()
    return p


def ssd_workspace_bytes(batch, seqlen, nheads, headdim=64, dstate=128) -> int:
    """Workspace bytes of ssm_ssd_fwd (the segment hand-off of each chain)."""
    p = capi.SsdParams()
    p.batch, p.seqlen, p.nheads, p.headdim, p.dstate = batch, seqlen, nheads, headdim, dstate
    n = capi.ssm_ssd_workspace_size(p)
    if n == 0:
        raise ValueError("invalid SSD sizes")
    return n


def ssd_fwd(x, dt, A, B, C, D=None, dt_bias=None, h0=None, *, dt_softplus=True, y=None, hL=None,
            return_last_state=True, stream=None, status=None, workspace=None, split=True):
    """Mamba-2 layer scan: x (b, L, H, P), dt (b, L, H), A (H,), B, C (b, L, N).
    Returns (y (b, L, H, P), hL (b, H, P, N) fp32 or None).  `status`, an int32
    device tensor of one element, receives SSM_ERR_TIMEOUT if a bounded wait
    inside the kernel ran out.  With `split` (the default) each (sequence,
    head) chain runs as segments handing their state on through `workspace`
    (allocated here if None); split=False runs one CTA per chain."""
    if y is None:
        y = torch.empty_like(x)
    if hL is None and return_last_state:
        b, L, H, P = x.shape
        hL = torch.empty((b, H, P, B.shape[2]), dtype=torch.float32, device=x.device)
    if split and workspace is None:
        b, L, H, P = x.shape
        workspace = torch.empty(ssd_workspace_bytes(b, L, H, P, B.shape[2]), dtype=torch.uint8, device=x.device)
    p = ssd_params(x, dt, A, B, C, D, dt_bias, h0, y=y, hL=hL, dt_softplus=dt_softplus, status=status,
                   workspace=workspace if split else None)
    st = torch.cuda.current_stream(x.device).cuda_stream if stream is None else stream
    capi.check(capi.ssm_ssd_fwd(p, st), "ssm_ssd_fwd")
    return y, hL


def conv_params(x, weight, bias=None, state_in=None, *, u, state_out=None, silu=True) -> capi.ConvParams:
    """Validate tensors and build the convolution's C parameter struct."""
    if x.dtype not in _DT:
        raise ValueError(f"unsupported I/O dtype {x.dtype}")
    dev = x.device
    b, dim, L = x.shape
    W = weight.shape[1]
    io = x.dtype
    _need(x, "x", (b, dim, L), io, dev)
    _need(weight, "weight", (dim, W), torch.float32, dev)
    _opt(bias, "bias", (dim,), torch.float32, dev)
    _opt(state_in, "state_in", (b, dim, W - 1), io, dev)
    _need(u, "u", (b, dim, L), io, dev)
    _opt(state_out, "state_out", (b, dim, W - 1), io, dev)
    p = capi.ConvParams()
    p.batch, p.dim, p.seqlen, p.width = b, dim, L, W
    p.io_dtype = _DT[io]
    p.x, p.weight, p.bias = _ptr(x), _ptr(weight), _ptr(bias)
    p.silu = int(bool(silu))
    p.state_in, p.u, p.state_out = _ptr(state_in), _ptr(u), _ptr(state_out)
    return p


def conv1d(x, weight, bias=None, state_in=None, *, silu=True, u=None, state_out=None,
           return_state=True, stream=None):
    """Causal depthwise convolution (+ bias, + SiLU) of x (b, D, L) with weight
    (D, W).  Returns (u, state_out); state_out (b, D, W-1) holds the last W-1
    inputs (None if not requested)."""
    if u is None:
        u = torch.empty_like(x)
    if state_out is None and return_state:
        state_out = torch.empty((x.shape[0], x.shape[1], weight.shape[1] - 1), dtype=x.dtype, device=x.device)
    p = conv_params(x, weight, bias, state_in, u=u, state_out=state_out, silu=silu)
    st = torch.cuda.current_stream(x.device).cuda_stream if stream is None else stream
    capi.check(capi.ssm_conv1d_fwd(p, st), "ssm_conv1d_fwd")
    return u, state_out


def conv1d_step(state, x, weight, bias=None, *, silu=True, u=None, stream=None):
    """One decode token of the convolution: x (b, D); ``state`` (b, D, W-1) is
    shifted in place.  Returns u (b, D)."""
    if x.dtype not in _DT:
        raise ValueError(f"unsupported I/O dtype {x.dtype}")
    dev = x.device
    b, dim = x.shape
    W = weight.shape[1]
    if u is None:
        u = torch.empty_like(x)
    _need(x, "x", (b, dim), x.dtype, dev)
    _need(weight, "weight", (dim, W), torch.float32, dev)
    _opt(bias, "bias", (dim,), torch.float32, dev)
    if W > 1:
        _need(state, "state", (b, dim, W - 1), x.dtype, dev)
    _need(u, "u", (b, dim), x.dtype, dev)
    p = capi.ConvStepParams()
    p.batch, p.dim, p.width = b, dim, W
    p.io_dtype = _DT[x.dtype]
    p.state = _ptr(state) if W > 1 else None
    p.x, p.weight, p.bias = _ptr(x), _ptr(weight), _ptr(bias)
    p.silu = int(bool(silu))
    p.u = _ptr(u)
    st = torch.cuda.current_stream(dev).cuda_stream if stream is None else stream
    capi.check(capi.ssm_conv1d_step(p, st), "ssm_conv1d_step")
    return u


def workspace_status(workspace, stream=None) -> int:
    """Synchronise and return the device status recorded in a scan workspace."""
    st = torch.cuda.current_stream(workspace.device).cuda_stream if stream is None else stream
    return capi.ssm_workspace_status(workspace.data_ptr(), st)
