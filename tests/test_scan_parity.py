"""Forward scan: CUDA path against the fp64 oracle on the same seeded inputs."""

import pytest
import torch

from mamba_selective_scan_02_b300 import api, capi
from mamba_selective_scan_02_b300.inputs import WORKLOADS, make_inputs
from ssm_testutil import (assert_close, gpu_scan, oracle_scan, oracle_scan_sampled,
                          sample_channels, to_device, to_host)

pytestmark = pytest.mark.gpu


def _case(b, D, N, L, dtype, seed, *, z=True, skip=True, bias=True, h0=False):
    g = torch.Generator().manual_seed(seed)

    def rn(*s, std=1.0):
        return (torch.randn(*s, generator=g) * std).to(dtype)
    return dict(u=rn(b, D, L), delta=rn(b, D, L, std=0.5), z=rn(b, D, L) if z else None,
                B=rn(b, N, L), C=rn(b, N, L),
                A=(-torch.arange(1, N + 1, dtype=torch.float32).repeat(D, 1)
                   * (0.5 + torch.rand(D, 1, generator=g))),
                Dskip=torch.randn(D, generator=g) if skip else None,
                bias=(torch.log(torch.expm1(torch.empty(D).uniform_(1e-3, 1e-1, generator=g))).float()
                      if bias else None),
                h0=torch.randn(b, D, N, generator=g) * 0.5 if h0 else None)


def _check(inp, dtype, what, **kw):
    y_ref, h_ref = oracle_scan(inp, delta_softplus=kw.get("delta_softplus", True))
    y, hL = gpu_scan(to_device(inp), **kw)
    assert_close(y.double().cpu().numpy(), y_ref, dtype, what + " y")
    assert_close(hL.double().cpu().numpy(), h_ref, dtype, what + " hL")


def test_tiny_fp32_workload():
    _check(make_inputs("tiny_fp32"), torch.float32, "tiny_fp32")


@pytest.mark.parametrize("b,D,N,L,dtype,opts", [
    (2, 40, 16, 200, torch.bfloat16, {}),                 # TMA path, ragged channel tile and last tile
    (1, 33, 5, 203, torch.bfloat16, {}),                  # row pitch not 16-B aligned: plain loads
    (2, 7, 3, 97, torch.float32, {}),
    (1, 300, 8, 128, torch.float32, dict(chunk_len=64)),  # two chunks joined by look-back
    (2, 64, 16, 1000, torch.bfloat16, dict(chunk_len=128, h0=True)),
    (1, 16, 1, 1, torch.float32, {}),                     # L = 1, N = 1
    (3, 130, 12, 257, torch.bfloat16, dict(z=False)),     # padded state group, no gate
    (1, 128, 4, 64, torch.float32, dict(skip=False, bias=False, softplus=False)),
    (2, 96, 16, 4096, torch.bfloat16, dict(chunk_len=512, h0=True)),
    (1, 8, 2, 33, torch.float32, dict(h0=True)),
])
def test_small_shapes(b, D, N, L, dtype, opts):
    opts = dict(opts)
    chunk = opts.pop("chunk_len", 0)
    softplus = opts.pop("softplus", True)
    inp = _case(b, D, N, L, dtype, seed=b * 1000 + D + N + L, **opts)
    if not softplus:
        inp["delta"] = inp["delta"].float().abs().to(dtype)  # a non-negative step without softplus
    _check(inp, dtype, f"{b}x{D}x{N}x{L} {dtype}", chunk_len=chunk, delta_softplus=softplus)


def test_chained_chunks_every_element():
    """Enough channel groups that chunk k starts from the state chunk k-1 hands
    over (one warp per 16 channels: 225 groups per sequence)."""
    inp = _case(4, 3600, 16, 512, torch.bfloat16, seed=21, h0=True)
    p = capi.ScanParams()
    p.batch, p.dim, p.dstate, p.seqlen, p.chunk_len = 4, 3600, 16, 512, 64
    assert capi.ssm_scan_plan(p)["chained"]
    _check(inp, torch.bfloat16, "chained 4x3600x16x512", chunk_len=64)


@pytest.mark.parametrize("chunk", [64, 0])
def test_chained_ragged_every_element(chunk):
    """The warp-specialised pass in chained mode on a ragged layer: 3,608
    channels (a partial 16-channel group per sequence), 456 tokens (the last
    32-token tile holds 8), with h0 and no gate; chunks of 64 tokens (eight
    hand-offs per group) or the default length (two)."""
    b, D, N, L = 4, 3608, 16, 456
    inp = _case(b, D, N, L, torch.bfloat16, seed=23, z=False, h0=True)
    p = capi.ScanParams()
    p.batch, p.dim, p.dstate, p.seqlen, p.chunk_len = b, D, N, L, chunk
    plan = capi.ssm_scan_plan(p)
    assert plan["chained"] and plan["groups"] == b * 226 and plan["nchunks"] == (8 if chunk else 2)
    _check(inp, torch.bfloat16, f"chained ragged {b}x{D}x{N}x{L} chunk {chunk}", chunk_len=chunk)


def test_small_layer_workload_full():
    """The 2 × 1536 × 16 × 2048 bf16 layer, every channel checked."""
    _check(make_inputs("small_layer_L2048"), torch.bfloat16, "small_layer_L2048")


@pytest.mark.parametrize("chunk", [64, 256, 2048])
def test_small_layer_chunk_sizes(chunk):
    inp = make_inputs("small_layer_L2048", batch=1, dim=256)
    _check(inp, torch.bfloat16, f"small layer chunk {chunk}", chunk_len=chunk)


def _full_size_sampled(name, nsample):
    w = WORKLOADS[name]
    inp = make_inputs(w, device="cuda")
    y, hL = gpu_scan(inp)
    ch = sample_channels(w.batch, w.dim, nsample, seed=w.seed)
    y_ref, h_ref = oracle_scan_sampled(inp, ch)
    yi = torch.stack([y[bi, di] for bi, di in ch]).double().cpu().numpy()
    hi = torch.stack([hL[bi, di] for bi, di in ch]).double().cpu().numpy()
    assert_close(yi, y_ref, torch.bfloat16, name + " y (sampled channels)")
    assert_close(hi, h_ref, torch.bfloat16, name + " hL (sampled channels)")
    assert torch.isfinite(y.float()).all() and torch.isfinite(hL).all()


def test_mamba28b_layer_full_size_sampled():
    _full_size_sampled("mamba2.8b_layer_L2048", 48)


def test_long_sequence_full_size_sampled():
    _full_size_sampled("long_seq_L131072", 12)


def test_deterministic_and_resumable():
    inp = to_device(_case(2, 64, 16, 512, torch.bfloat16, seed=5, h0=True))
    y1, h1 = gpu_scan(inp, chunk_len=128)
    y2, h2 = gpu_scan(inp, chunk_len=128)
    assert torch.equal(y1, y2) and torch.equal(h1, h2)
    cut = 192   # split at a token and resume from the carried state
    part = {k: inp[k][..., :cut].contiguous() for k in ("u", "delta", "z", "B", "C")}
    rest = {k: inp[k][..., cut:].contiguous() for k in ("u", "delta", "z", "B", "C")}
    ya, ha = gpu_scan(dict(inp, **part))
    yb, hb = gpu_scan(dict(inp, **rest, h0=ha))
    assert_close(torch.cat([ya, yb], -1).double().cpu().numpy(), y1.double().cpu().numpy(),
                 torch.bfloat16, "split and resume")
    assert_close(hb.cpu().numpy(), h1.cpu().numpy(), torch.bfloat16, "split and resume state")


def test_final_state_may_alias_initial_state():
    inp = to_device(_case(1, 64, 16, 640, torch.bfloat16, seed=9, h0=True))
    y_ref, h_ref = oracle_scan(to_host(inp))
    for chunk in (0, 64):
        h = inp["h0"].clone()
        y, _ = api.scan_fwd(inp["u"], inp["delta"], inp["A"], inp["B"], inp["C"], inp["Dskip"],
                            inp["z"], inp["bias"], h, hL=h, chunk_len=chunk)
        torch.cuda.synchronize()
        assert_close(y.double().cpu().numpy(), y_ref, torch.bfloat16, f"aliased y chunk={chunk}")
        assert_close(h.cpu().numpy(), h_ref, torch.bfloat16, f"aliased hL chunk={chunk}")


def test_output_guard_bands_untouched():
    inp = to_device(_case(2, 40, 16, 200, torch.bfloat16, seed=3))
    n = inp["u"].numel()
    buf = torch.full((n + 4096,), 7.0, dtype=torch.bfloat16, device="cuda")
    y = buf[:n].view(inp["u"].shape)
    hbuf = torch.full((2 * 40 * 16 + 1024,), -3.0, device="cuda")
    hL = hbuf[:2 * 40 * 16].view(2, 40, 16)
    api.scan_fwd(inp["u"], inp["delta"], inp["A"], inp["B"], inp["C"], inp["Dskip"], inp["z"],
                 inp["bias"], y=y, hL=hL)
    torch.cuda.synchronize()
    assert torch.all(buf[n:] == 7.0)
    assert torch.all(hbuf[2 * 40 * 16:] == -3.0)


def test_workspace_status_ok_and_errors():
    inp = to_device(_case(1, 32, 16, 256, torch.bfloat16, seed=4))
    ws = torch.empty(api.workspace_bytes(inp["u"], inp["delta"], inp["A"], inp["B"], inp["C"], 64),
                     dtype=torch.uint8, device="cuda")
    api.scan_fwd(inp["u"], inp["delta"], inp["A"], inp["B"], inp["C"], inp["Dskip"], inp["z"],
                 inp["bias"], chunk_len=64, workspace=ws)
    assert api.workspace_status(ws) == capi.SSM_OK
    with pytest.raises(capi.SSMError) as e:
        api.scan_fwd(inp["u"], inp["delta"], inp["A"], inp["B"], inp["C"], chunk_len=64, workspace=ws[:64])
    assert e.value.code == capi.SSM_ERR_INVALID_ARG
    odd = torch.empty(inp["u"].numel() + 8, dtype=torch.bfloat16, device="cuda")[1:1 + inp["u"].numel()]
    with pytest.raises(capi.SSMError):
        api.scan_fwd(odd.view(inp["u"].shape), inp["delta"], inp["A"], inp["B"], inp["C"])
