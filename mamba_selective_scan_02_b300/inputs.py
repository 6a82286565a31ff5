"""Seeded synthetic inputs for the selective scan and the decode step.

This module only draws random numbers; it holds none of the scan's arithmetic.
Both the CUDA path and the fp64 oracle receive the tensors it returns (the
oracle after widening to fp64), so the two always see identical values.

Draw order is fixed: u, delta_raw, z, B, C, Dskip, the bias draw U, then the
initial state.  Everything is drawn in fp32 with a ``torch.Generator`` seeded on
the target device and rounded (round-to-nearest-even) to bf16 where the
workload says bf16.  Draws on ``cpu`` and on ``cuda`` use different generators,
so a workload is reproducible per device type.

Workloads follow the layer shapes of the pages: Mamba-2.8B has width 2,560 and
5,120 inner channels with N = 16 [Mamba and selective state spaces, from first
principles — "The Mamba block"], A is initialised S4D-Real, A_n = -(n+1)
[same page — "A state space model"].
"""

from __future__ import annotations

from dataclasses import dataclass

import torch


@dataclass(frozen=True)
class Workload:
    name: str
    batch: int
    dim: int
    dstate: int
    seqlen: int          # tokens per sequence (decode: number of consecutive tokens)
    io_dtype: str        # "f32" or "bf16"
    delta_std: float     # std of delta_raw
    bias: str            # "const-1" or "inv-softplus-U[1e-3,1e-1]"
    seed: int
    decode: bool = False
    h0_std: float = 0.0  # >0: draw an initial state N(0, h0_std)

    @property
    def elements(self) -> int:
        return self.batch * self.dim * self.seqlen


WORKLOADS = {
    w.name: w for w in [
        Workload("tiny_fp32", 1, 16, 4, 64, "f32", 1.0, "const-1", 0),
        Workload("small_layer_L2048", 2, 1536, 16, 2048, "bf16", 0.5,
                 "inv-softplus-U[1e-3,1e-1]", 1),
        Workload("mamba2.8b_layer_L2048", 4, 5120, 16, 2048, "bf16", 0.5,
                 "inv-softplus-U[1e-3,1e-1]", 2),
        Workload("long_seq_L131072", 1, 5120, 16, 131072, "bf16", 0.5,
                 "inv-softplus-U[1e-3,1e-1]", 3),
        Workload("decode_b256_64tok", 256, 5120, 16, 64, "bf16", 0.5,
                 "inv-softplus-U[1e-3,1e-1]", 4, decode=True, h0_std=0.1),
    ]
}


def torch_dtype(io_dtype: str) -> torch.dtype:
    return {"f32": torch.float32, "bf16": torch.bfloat16}[io_dtype]


def s4d_real_A(dim: int, dstate: int, device="cpu") -> torch.Tensor:
    """A[d, n] = -(n + 1) for every channel (fp32, dim × dstate)."""
    return -torch.arange(1, dstate + 1, dtype=torch.float32, device=device).repeat(dim, 1).contiguous()


def _bias(w: Workload, dim: int, g: torch.Generator, device) -> torch.Tensor:
    if w.bias == "const-1":
        return torch.full((dim,), -1.0, dtype=torch.float32, device=device)
    # bias_d = log(expm1(U_d)) with U_d ~ Uniform[1e-3, 1e-1]: the inverse of the
    # softplus, so that softplus(bias_d) = U_d is the channel's resting step size.
    U = torch.empty(dim, dtype=torch.float64, device=device)
    U.uniform_(1e-3, 1e-1, generator=g)
    return torch.log(torch.expm1(U)).float()


def make_inputs(w: Workload | str, device="cpu", batch: int | None = None,
                dim: int | None = None, seqlen: int | None = None,
                seed: int | None = None) -> dict:
    """Draw one workload's inputs on ``device``.

    batch / dim / seqlen / seed override the workload's sizes (used for the
    small parity cases drawn with the same distributions).

    Scan workloads return u, delta, z (b, D, L) and B, C (b, N, L) in the I/O
    dtype; A (D, N), Dskip, bias (D,) in fp32; h0 (b, D, N) fp32 or None.
    Decode workloads return the same names with a leading token axis T:
    u, delta, z (T, b, D), B, C (T, b, N), and h0 = the carried state (b, D, N).
    """
    if isinstance(w, str):
        w = WORKLOADS[w]
    b = w.batch if batch is None else batch
    D = w.dim if dim is None else dim
    L = w.seqlen if seqlen is None else seqlen
    N = w.dstate
    g = torch.Generator(device=device)
    g.manual_seed(w.seed if seed is None else seed)
    dt = torch_dtype(w.io_dtype)

    def normal(shape, std=1.0):
        x = torch.randn(shape, generator=g, dtype=torch.float32, device=device)
        if std != 1.0:
            x.mul_(std)
        return x.to(dt)

    if w.decode:
        seq_shape, bc_shape = (L, b, D), (L, b, N)
    else:
        seq_shape, bc_shape = (b, D, L), (b, N, L)
    u = normal(seq_shape)
    delta = normal(seq_shape, w.delta_std)
    z = normal(seq_shape)
    B = normal(bc_shape)
    C = normal(bc_shape)
    Dskip = torch.randn(D, generator=g, dtype=torch.float32, device=device)
    bias = _bias(w, D, g, device)
    h0 = None
    if w.h0_std > 0:
        h0 = torch.randn((b, D, N), generator=g, dtype=torch.float32, device=device) * w.h0_std
    return dict(u=u, delta=delta, z=z, B=B, C=C, A=s4d_real_A(D, N, device),
                Dskip=Dskip, bias=bias, h0=h0, workload=w, batch=b, dim=D, dstate=N,
                seqlen=L)


def make_conv_inputs(batch: int, dim: int, seqlen: int, width: int = 4, io_dtype: str = "bf16",
                     seed: int = 0, device="cpu", with_state: bool = True, decode: bool = False) -> dict:
    """Seeded inputs for the short convolution in front of the scan.

    x ~ N(0, 1) in the I/O dtype (the input projection's output); weight and
    bias ~ U(-1/sqrt(W), 1/sqrt(W)) in fp32, the default initialisation of a
    depthwise convolution whose fan-in is its width; the carried state (the
    W-1 inputs before the sequence) ~ N(0, 1) in the I/O dtype, or None.
    x is (b, D, L), or (T, b, D) for ``decode`` (T = seqlen consecutive tokens).
    Draw order: x, weight, bias, state."""
    g = torch.Generator(device=device)
    g.manual_seed(seed)
    dt = torch_dtype(io_dtype)
    shape = (seqlen, batch, dim) if decode else (batch, dim, seqlen)
    x = torch.randn(shape, generator=g, dtype=torch.float32, device=device).to(dt)
    bound = 1.0 / (width ** 0.5)
    weight = (torch.rand((dim, width), generator=g, dtype=torch.float32, device=device) * 2 - 1) * bound
    bias = (torch.rand(dim, generator=g, dtype=torch.float32, device=device) * 2 - 1) * bound
    state = None
    if with_state:
        state = torch.randn((batch, dim, width - 1), generator=g, dtype=torch.float32, device=device).to(dt)
    return dict(x=x, weight=weight, bias=bias, state=state)


def make_ssd_inputs(batch: int, seqlen: int, nheads: int = 80, headdim: int = 64, dstate: int = 128,
                    seed: int = 0, device="cpu", with_h0: bool = False) -> dict:
    """Seeded bf16 inputs for the Mamba-2 layer scan, shaped like the Mamba-2
    2.7B layer of "Mamba-2: state space duality" (80 heads of 64, N = 128, one
    B/C group).  x, B, C ~ N(0,1); dt ~ N(0, 0.5) with dt_bias =
    log(expm1(U[1e-3, 1e-1])) per head (as the Mamba-1 workloads' Δ); A_h =
    -U[1, 16] per head (Mamba-2 initialises A_log = log U[1, 16]); D ~ N(0,1);
    h0 ~ N(0, 0.1) when asked.  Draw order: x, dt, B, C, A, D, dt_bias, h0."""
    g = torch.Generator(device=device)
    g.manual_seed(seed)
    bf = torch.bfloat16
    x = torch.randn((batch, seqlen, nheads, headdim), generator=g, device=device).to(bf)
    dt = (torch.randn((batch, seqlen, nheads), generator=g, device=device) * 0.5).to(bf)
    B = torch.randn((batch, seqlen, dstate), generator=g, device=device).to(bf)
    C = torch.randn((batch, seqlen, dstate), generator=g, device=device).to(bf)
    A = -(torch.rand(nheads, generator=g, device=device) * 15 + 1)
    D = torch.randn(nheads, generator=g, device=device)
    U = torch.empty(nheads, dtype=torch.float64, device=device)
    U.uniform_(1e-3, 1e-1, generator=g)
    dt_bias = torch.log(torch.expm1(U)).float()
    h0 = None
    if with_h0:
        h0 = torch.randn((batch, nheads, headdim, dstate), generator=g, device=device) * 0.1
    return dict(x=x, dt=dt, A=A, B=B, C=C, D=D, dt_bias=dt_bias, h0=h0)


__all__ = ["Workload", "WORKLOADS", "make_inputs", "make_conv_inputs", "make_ssd_inputs", "s4d_real_A",
           "torch_dtype"]
