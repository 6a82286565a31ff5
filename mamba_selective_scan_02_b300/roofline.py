"""Algorithmic byte and exponential counts for the roofline of each kernel.

These are the minimum the method must move or evaluate, not what a kernel
happens to move: the fused scan never writes the discretised (Ā, B̄) of shape
(batch, L, D, N) nor any intermediate state [Mamba and selective state spaces,
from first principles — "The hardware-aware scan"].
"""


def algorithmic_bytes_scan(batch: int, dim: int, dstate: int, seqlen: int, io_bytes: int,
                           has_z: bool = True, has_h0: bool = False, has_hL: bool = True) -> int:
    """Bytes the fused scan must move at minimum: u, delta (and z) read once and
    y written once per (b, d, t); B and C read once per (b, t) (not per
    channel); A, D and bias once; h0 / hL once per (b, d, n)."""
    per_elem = (3 if has_z else 2) + 1
    n = batch * dim * seqlen * per_elem * io_bytes
    n += 2 * batch * dstate * seqlen * io_bytes
    n += dim * dstate * 4 + 2 * dim * 4
    n += batch * dim * dstate * 4 * (int(has_h0) + int(has_hL))
    return n


def algorithmic_bytes_step(batch: int, dim: int, dstate: int, io_bytes: int,
                           has_z: bool = True) -> int:
    """Bytes per decode token: the fp32 state read and written once, u, delta
    (z) read and y written per (b, d), B and C read per (b, n), A, D, bias once."""
    n = 2 * batch * dim * dstate * 4
    n += batch * dim * ((3 if has_z else 2) + 1) * io_bytes
    n += 2 * batch * dstate * io_bytes
    n += dim * dstate * 4 + 2 * dim * 4
    return n


def algorithmic_bytes_conv(batch: int, dim: int, seqlen: int, width: int, io_bytes: int,
                           has_state_in: bool = True, has_state_out: bool = True) -> int:
    """Bytes the short convolution must move: x read and u written once per
    (b, d, t), the W taps and the bias once per channel, the W-1 carried
    inputs read and written once per (b, d)."""
    n = 2 * batch * dim * seqlen * io_bytes
    n += dim * (width + 1) * 4
    n += batch * dim * (width - 1) * io_bytes * (int(has_state_in) + int(has_state_out))
    return n


def algorithmic_bytes_conv_step(batch: int, dim: int, width: int, io_bytes: int) -> int:
    """Bytes per decode token of the convolution: the W-1 carried inputs read
    and written, x read and u written per (b, d), taps and bias once."""
    return batch * dim * (2 * (width - 1) + 2) * io_bytes + dim * (width + 1) * 4


def algorithmic_bytes_bwd(batch: int, dim: int, dstate: int, seqlen: int, io_bytes: int,
                          has_z: bool = True) -> int:
    """Bytes the backward scan must move at minimum: u, Δraw, (z,) dy read and
    du, dΔraw, (dz) written once per (b, d, t); B, C read and dB, dC (fp32)
    written once per (b, n, t); A, D, bias read and their fp32 gradients
    written once.  The states are recomputed, never read from memory."""
    per_elem = (4 if has_z else 3) + (3 if has_z else 2)
    n = batch * dim * seqlen * per_elem * io_bytes
    n += batch * dstate * seqlen * (2 * io_bytes + 2 * 4)
    n += 2 * (dim * dstate * 4 + 2 * dim * 4)
    return n


def algorithmic_bytes_ssd(batch: int, seqlen: int, nheads: int, headdim: int, dstate: int,
                          io_bytes: int = 2, has_hL: bool = True) -> int:
    """Bytes the Mamba-2 layer scan must move: x read and y written once per
    (b, t, h, p); B and C read once per (b, t, n) (one group for all heads); Δraw
    once per (b, t, h); A, D, Δ bias once; the final state once."""
    n = 2 * batch * seqlen * nheads * headdim * io_bytes
    n += 2 * batch * seqlen * dstate * io_bytes + batch * seqlen * nheads * io_bytes
    n += 3 * nheads * 4
    n += batch * nheads * headdim * dstate * 4 * int(has_hL)
    return n


def flops_ssd(batch: int, seqlen: int, nheads: int, headdim: int, dstate: int, chunk: int = 128) -> int:
    """Multiply-add FLOPs of the chunked SSD algorithm at chunk length Q: per
    chunk and head, the causal half of C·Bᵀ (Q²·N) and of its product with X
    (Q²·P), the inherited state's read-out C·Sᵀ (2·Q·N·P) and the chunk's state
    Xᵀ·B (2·Q·N·P)."""
    nch = -(-seqlen // chunk)
    per = chunk * chunk * dstate + chunk * chunk * headdim + 4 * chunk * dstate * headdim
    return batch * nheads * nch * per


def exps_scan(batch: int, dim: int, dstate: int, seqlen: int) -> int:
    """One exponential Ā = exp(Δ·A) per (b, d, n, t)."""
    return batch * dim * dstate * seqlen
