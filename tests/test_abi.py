"""The C-ABI library loads, exports every declared entry point, and rejects bad
arguments before touching the GPU (these run without a GPU: every call below
returns from host-side validation)."""

import ctypes
import os
import re

import pytest

from mamba_selective_scan_02_b300 import capi

ROOT = os.path.dirname(os.path.dirname(os.path.abspath(__file__)))
HEADER = os.path.join(ROOT, "include", "ssm_scan.h")


def declared_functions():
    text = open(HEADER).read()
    text = re.sub(r"/\*.*?\*/", "", text, flags=re.S)
    return sorted(set(re.findall(r"\b(ssm_[a-z0-9_]+)\s*\(", text)))


def test_header_declares_the_boundary():
    names = declared_functions()
    for must in ("ssm_scan_fwd", "ssm_state_update", "ssm_scan_workspace_size",
                 "ssm_workspace_status", "ssm_status_string"):
        assert must in names


def test_library_exports_every_declared_symbol():
    lib = capi.lib()
    for name in declared_functions():
        assert hasattr(lib, name), f"{name} declared in include/ssm_scan.h but not exported"


def test_library_is_in_tree():
    assert os.path.dirname(capi.library_path()).startswith(ROOT)
    assert capi.lib().ssm_version().decode().endswith("sm_103a")


def test_status_strings():
    for code in range(5):
        assert capi.status_string(code)
    assert capi.status_string(99) == "unknown status"


FAKE = 0x10000000  # never dereferenced: every case below fails validation first


def valid_scan(**over):
    p = capi.ScanParams()
    p.batch, p.dim, p.dstate, p.seqlen = 2, 64, 16, 256
    p.io_dtype = capi.SSM_BF16
    step = 1 << 20
    p.u, p.delta, p.z, p.B, p.C = FAKE, FAKE + step, FAKE + 2 * step, FAKE + 3 * step, FAKE + 4 * step
    p.A, p.Dskip, p.delta_bias = FAKE + 5 * step, FAKE + 6 * step, FAKE + 7 * step
    p.delta_softplus = 1
    p.y, p.hL, p.workspace = FAKE + 8 * step, FAKE + 9 * step, FAKE + 10 * step
    p.workspace_bytes = 1 << 20
    for k, v in over.items():
        setattr(p, k, v)
    return p


@pytest.mark.parametrize("over,code", [
    (dict(batch=0), capi.SSM_ERR_INVALID_ARG),
    (dict(seqlen=0), capi.SSM_ERR_INVALID_ARG),
    (dict(dstate=0), capi.SSM_ERR_INVALID_ARG),
    (dict(dstate=17), capi.SSM_ERR_UNSUPPORTED),
    (dict(io_dtype=7), capi.SSM_ERR_INVALID_ARG),
    (dict(u=None), capi.SSM_ERR_INVALID_ARG),
    (dict(A=None), capi.SSM_ERR_INVALID_ARG),
    (dict(workspace=None), capi.SSM_ERR_INVALID_ARG),
    (dict(u=FAKE + 2), capi.SSM_ERR_INVALID_ARG),           # not 16-byte aligned
    (dict(hL=FAKE + 9 * (1 << 20) + 8), capi.SSM_ERR_INVALID_ARG),
    (dict(A=FAKE + 5 * (1 << 20) + 1), capi.SSM_ERR_INVALID_ARG),
    (dict(y=FAKE + 64), capi.SSM_ERR_INVALID_ARG),          # y overlaps u
    (dict(workspace_bytes=16), capi.SSM_ERR_INVALID_ARG),   # smaller than the status word header
    (dict(chunk_len=100), capi.SSM_ERR_INVALID_ARG),        # not a multiple of 64
    (dict(chunk_len=-64), capi.SSM_ERR_INVALID_ARG),
    (dict(delta_softplus=2), capi.SSM_ERR_INVALID_ARG),
    (dict(zoh=2), capi.SSM_ERR_INVALID_ARG),
])
def test_scan_rejects_before_launch(over, code):
    assert capi.ssm_scan_fwd(valid_scan(**over), None) == code


def test_scan_rejects_null_params():
    assert capi.lib().ssm_scan_fwd(None, None) == capi.SSM_ERR_INVALID_ARG
    assert capi.lib().ssm_scan_workspace_size(None) == 0


def _bc_bytes(b, L, np_):
    """B and C widened to fp32 token-major rows: two [b][L][np] arrays."""
    return 2 * (-(-b * L * np_ * 4 // 256) * 256)


def test_workspace_size():
    p = valid_scan(chunk_len=256)
    assert capi.ssm_scan_workspace_size(p) == 256 + _bc_bytes(2, 256, 16)   # one chunk
    p = valid_scan(chunk_len=64)                             # 4 chunks of 64 tokens, look-back
    bdn = 2 * 64 * 16
    flags = -(-(2 * 64 // 16) * 4 * 4 // 256) * 256           # one per (group of 16 channels, chunk)
    agg = -(-bdn * 3 * 8 // 256) * 256
    carry = -(-bdn * 4 * 4 // 256) * 256
    assert capi.ssm_scan_workspace_size(p) == 256 + flags + agg + carry + _bc_bytes(2, 256, 16)
    # the small-model layer shape is split into chunks automatically
    p = valid_scan(batch=2, dim=1536, seqlen=2048)
    assert capi.ssm_scan_workspace_size(p) > 256 + _bc_bytes(2, 2048, 16)
    # enough channel groups to fill the GPU: chunks are chained, and the
    # workspace holds one flag per group of 16 channels and one hand-off state
    p = valid_scan(batch=4, dim=5120, seqlen=2048)
    groups = 4 * 5120 // 16
    flags = -(-groups * 4 // 256) * 256
    assert capi.ssm_scan_workspace_size(p) == 256 + flags + 4 * 5120 * 16 * 4 + _bc_bytes(4, 2048, 16)
    # small state sizes widen B and C to rows of 4 or 8
    p = valid_scan(batch=1, dim=64, dstate=4, seqlen=256, chunk_len=256)
    assert capi.ssm_scan_workspace_size(p) == 256 + _bc_bytes(1, 256, 4)
    # too small a workspace is rejected
    p = valid_scan(chunk_len=64, workspace_bytes=300)
    assert capi.ssm_scan_fwd(p, None) == capi.SSM_ERR_INVALID_ARG


def test_scan_plan():
    plan = capi.ssm_scan_plan(valid_scan(batch=4, dim=5120, seqlen=2048))
    assert plan == {"chunk_len": 384, "nchunks": 6, "chained": True, "groups": 1280}
    plan = capi.ssm_scan_plan(valid_scan(batch=1, dim=5120, seqlen=131072))
    assert not plan["chained"] and plan["nchunks"] > 1 and plan["chunk_len"] % 64 == 0
    plan = capi.ssm_scan_plan(valid_scan(batch=1, dim=64, seqlen=64))
    assert plan["nchunks"] == 1 and not plan["chained"]
    # few channel groups on a long sequence: chunks sized so that both passes
    # fill the resident warps (320 groups, 131072 tokens -> dozens of chunks)
    plan = capi.ssm_scan_plan(valid_scan(batch=1, dim=5120, seqlen=131072))
    assert plan["nchunks"] * plan["groups"] >= 8 * 1184
    assert capi.lib().ssm_scan_plan(None, None) == capi.SSM_ERR_INVALID_ARG


def valid_step(**over):
    p = capi.StepParams()
    p.batch, p.dim, p.dstate = 4, 64, 16
    p.io_dtype = capi.SSM_BF16
    step = 1 << 20
    p.state, p.u, p.delta, p.z = FAKE, FAKE + step, FAKE + 2 * step, FAKE + 3 * step
    p.B, p.C, p.A = FAKE + 4 * step, FAKE + 5 * step, FAKE + 6 * step
    p.delta_softplus = 1
    p.y = FAKE + 7 * step
    for k, v in over.items():
        setattr(p, k, v)
    return p


@pytest.mark.parametrize("over,code", [
    (dict(batch=0), capi.SSM_ERR_INVALID_ARG),
    (dict(dstate=17), capi.SSM_ERR_UNSUPPORTED),
    (dict(state=None), capi.SSM_ERR_INVALID_ARG),
    (dict(state=FAKE + 2), capi.SSM_ERR_INVALID_ARG),      # fp32 state not 4-byte aligned
    (dict(u=FAKE + (1 << 20) + 1), capi.SSM_ERR_INVALID_ARG),  # bf16 input at an odd address
    (dict(y=FAKE + 1 * (1 << 20)), capi.SSM_ERR_INVALID_ARG),  # y is u
    (dict(io_dtype=3), capi.SSM_ERR_INVALID_ARG),
    (dict(zoh=2), capi.SSM_ERR_INVALID_ARG),
])
def test_step_rejects_before_launch(over, code):
    assert capi.ssm_state_update(valid_step(**over), None) == code


def test_misc_rejections():
    lib = capi.lib()
    assert lib.ssm_state_update(None, None) == capi.SSM_ERR_INVALID_ARG
    assert lib.ssm_workspace_status(None, None) == capi.SSM_ERR_INVALID_ARG
    assert lib.ssm_bench_mufu_ex2(None, 1, 1, None) == capi.SSM_ERR_INVALID_ARG
    assert lib.ssm_bench_mufu_ex2(ctypes.c_void_p(FAKE), 0, 1, None) == capi.SSM_ERR_INVALID_ARG


def valid_conv(**over):
    p = capi.ConvParams()
    p.batch, p.dim, p.seqlen, p.width = 2, 64, 256, 4
    p.io_dtype = capi.SSM_BF16
    step = 1 << 20
    p.x, p.weight, p.bias = FAKE, FAKE + step, FAKE + 2 * step
    p.silu = 1
    p.state_in, p.u, p.state_out = FAKE + 3 * step, FAKE + 4 * step, FAKE + 5 * step
    for k, v in over.items():
        setattr(p, k, v)
    return p


@pytest.mark.parametrize("over,code", [
    (dict(batch=0), capi.SSM_ERR_INVALID_ARG),
    (dict(seqlen=0), capi.SSM_ERR_INVALID_ARG),
    (dict(width=0), capi.SSM_ERR_INVALID_ARG),
    (dict(width=5), capi.SSM_ERR_UNSUPPORTED),
    (dict(io_dtype=9), capi.SSM_ERR_INVALID_ARG),
    (dict(silu=3), capi.SSM_ERR_INVALID_ARG),
    (dict(x=None), capi.SSM_ERR_INVALID_ARG),
    (dict(weight=None), capi.SSM_ERR_INVALID_ARG),
    (dict(u=None), capi.SSM_ERR_INVALID_ARG),
    (dict(x=FAKE + 1), capi.SSM_ERR_INVALID_ARG),                     # bf16 at an odd address
    (dict(weight=FAKE + (1 << 20) + 2), capi.SSM_ERR_INVALID_ARG),    # fp32 weight not 4-byte aligned
    (dict(u=FAKE + 512), capi.SSM_ERR_INVALID_ARG),                   # u overlaps x
    (dict(state_out=FAKE + 3 * (1 << 20) + 2), capi.SSM_ERR_INVALID_ARG),  # state_out overlaps state_in
    (dict(state_out=FAKE + 4 * (1 << 20) + 64), capi.SSM_ERR_INVALID_ARG),  # state_out inside u
])
def test_conv_rejects_before_launch(over, code):
    assert capi.ssm_conv1d_fwd(valid_conv(**over), None) == code


def valid_conv_step(**over):
    p = capi.ConvStepParams()
    p.batch, p.dim, p.width = 4, 64, 4
    p.io_dtype = capi.SSM_F32
    step = 1 << 20
    p.state, p.x, p.weight, p.bias, p.u = FAKE, FAKE + step, FAKE + 2 * step, FAKE + 3 * step, FAKE + 4 * step
    p.silu = 1
    for k, v in over.items():
        setattr(p, k, v)
    return p


@pytest.mark.parametrize("over,code", [
    (dict(batch=0), capi.SSM_ERR_INVALID_ARG),
    (dict(width=0), capi.SSM_ERR_INVALID_ARG),
    (dict(width=8), capi.SSM_ERR_UNSUPPORTED),
    (dict(state=None), capi.SSM_ERR_INVALID_ARG),                     # W > 1 needs a state
    (dict(x=FAKE + (1 << 20) + 2), capi.SSM_ERR_INVALID_ARG),         # fp32 at a 2-byte offset
    (dict(u=FAKE + (1 << 20)), capi.SSM_ERR_INVALID_ARG),             # u is x
    (dict(u=FAKE + 16), capi.SSM_ERR_INVALID_ARG),                    # u inside the state
    (dict(silu=-1), capi.SSM_ERR_INVALID_ARG),
])
def test_conv_step_rejects_before_launch(over, code):
    assert capi.ssm_conv1d_step(valid_conv_step(**over), None) == code


def test_conv_null_params():
    assert capi.lib().ssm_conv1d_fwd(None, None) == capi.SSM_ERR_INVALID_ARG
    assert capi.lib().ssm_conv1d_step(None, None) == capi.SSM_ERR_INVALID_ARG


def valid_bwd(**over):
    p = capi.BwdParams()
    p.batch, p.dim, p.dstate, p.seqlen = 2, 64, 16, 256
    p.io_dtype = capi.SSM_BF16
    step = 1 << 20
    names = ["u", "delta", "z", "B", "C", "A", "Dskip", "delta_bias", "dy", "du", "ddelta", "dz",
             "dB", "dC", "dA", "workspace"]
    for i, n in enumerate(names):
        setattr(p, n, FAKE + i * step)
    p.delta_softplus = 1
    p.workspace_bytes = 1 << 30
    for k, v in over.items():
        setattr(p, k, v)
    return p


@pytest.mark.parametrize("over,code", [
    (dict(batch=0), capi.SSM_ERR_INVALID_ARG),
    (dict(dstate=17), capi.SSM_ERR_UNSUPPORTED),
    (dict(io_dtype=5), capi.SSM_ERR_INVALID_ARG),
    (dict(dy=None), capi.SSM_ERR_INVALID_ARG),
    (dict(dA=None), capi.SSM_ERR_INVALID_ARG),
    (dict(workspace=None), capi.SSM_ERR_INVALID_ARG),
    (dict(workspace_bytes=1024), capi.SSM_ERR_INVALID_ARG),
    (dict(chunk_len=24), capi.SSM_ERR_INVALID_ARG),            # not a multiple of 16
    (dict(u=FAKE + 1), capi.SSM_ERR_INVALID_ARG),               # bf16 at an odd address
    (dict(dB=FAKE + 12 * (1 << 20) + 2), capi.SSM_ERR_INVALID_ARG),
    (dict(workspace=FAKE + 15 * (1 << 20) + 4), capi.SSM_ERR_INVALID_ARG),  # not 16-byte aligned
    (dict(du=FAKE + 64), capi.SSM_ERR_INVALID_ARG),             # du overlaps u
    (dict(zoh=3), capi.SSM_ERR_INVALID_ARG),
])
def test_bwd_rejects_before_launch(over, code):
    assert capi.ssm_scan_bwd(valid_bwd(**over), None) == code


def test_bwd_workspace_size():
    p = valid_bwd()
    groups = 2 * 64 // 16
    ntiles = 256 // 16
    flags = -(-groups * 4 // 256) * 256
    bdn = -(-2 * 64 * 16 * 4 // 256) * 256
    assert capi.ssm_scan_bwd_workspace_size(p) == 256 + 2 * flags + 2 * bdn + groups * ntiles * 1024
    assert capi.ssm_scan_bwd_workspace_size(valid_bwd(seqlen=0)) == 0
    assert capi.lib().ssm_scan_bwd(None, None) == capi.SSM_ERR_INVALID_ARG


def test_bwd_workspace_size_with_forward_checkpoints():
    # Enough channel groups for a chained forward plan (bf16, first order): the
    # checkpoint pass runs on the forward scan kernel, which adds its own flags,
    # hand-off state and fp32 B, C rows to the workspace.
    b, d, n, L = 4, 5120, 16, 2048
    groups, ntiles = b * d // 16, L // 16
    flags = -(-groups * 4 // 256) * 256
    bdn = -(-b * d * n * 4 // 256) * 256
    bt = -(-b * L * 16 * 4 // 256) * 256
    base = 256 + 2 * flags + 2 * bdn + groups * ntiles * 1024
    p = valid_bwd(batch=b, dim=d, seqlen=L)
    assert capi.ssm_scan_bwd_workspace_size(p) == base + flags + bdn + 2 * bt
    # the zero-order hold keeps the backward's own checkpoint pass, as do fp32
    # I/O, too few channel groups for a chained forward plan, and a row pitch
    # TMA cannot describe
    assert capi.ssm_scan_bwd_workspace_size(valid_bwd(batch=b, dim=d, seqlen=L, zoh=1)) == base
    assert capi.ssm_scan_bwd_workspace_size(valid_bwd(batch=b, dim=d, seqlen=L, io_dtype=capi.SSM_F32)) == base
    small = valid_bwd(batch=1, dim=d, seqlen=L)                # 320 groups: a look-back forward plan
    g1 = d // 16
    assert capi.ssm_scan_bwd_workspace_size(small) == (
        256 + 2 * (-(-g1 * 4 // 256) * 256) + 2 * (-(-d * n * 4 // 256) * 256) + g1 * ntiles * 1024)
    odd = valid_bwd(batch=b, dim=d, seqlen=L - 1)              # 2·L bytes not a multiple of 16
    assert capi.ssm_scan_bwd_workspace_size(odd) == (
        256 + 2 * flags + 2 * bdn + groups * -(-(L - 1) // 16) * 1024)


def valid_ssd(**over):
    p = capi.SsdParams()
    p.batch, p.seqlen, p.nheads, p.headdim, p.dstate = 2, 256, 4, 64, 128
    p.io_dtype = capi.SSM_BF16
    step = 1 << 22
    for i, n in enumerate(["x", "dt", "A", "B", "C", "Dskip", "dt_bias", "y"]):
        setattr(p, n, FAKE + i * step)
    p.dt_softplus = 1
    for k, v in over.items():
        setattr(p, k, v)
    return p


def test_ssd_workspace_size_and_rejections():
    p = valid_ssd()
    n = capi.ssm_ssd_workspace_size(p)
    chains = 2 * 4
    assert n == 256 + (-(-chains * 4 // 256) * 256) + chains * 64 * 128 * 4
    assert capi.lib().ssm_ssd_workspace_size(None) == 0
    assert capi.ssm_ssd_workspace_size(valid_ssd(batch=0)) == 0
    small = valid_ssd(workspace=FAKE + (1 << 26), workspace_bytes=n - 1)
    assert capi.ssm_ssd_fwd(small, None) == capi.SSM_ERR_INVALID_ARG
    odd = valid_ssd(workspace=FAKE + (1 << 26) + 16, workspace_bytes=n)
    assert capi.ssm_ssd_fwd(odd, None) == capi.SSM_ERR_INVALID_ARG


@pytest.mark.parametrize("over,code", [
    (dict(batch=0), capi.SSM_ERR_INVALID_ARG),
    (dict(nheads=0), capi.SSM_ERR_INVALID_ARG),
    (dict(headdim=32), capi.SSM_ERR_UNSUPPORTED),
    (dict(dstate=64), capi.SSM_ERR_UNSUPPORTED),
    (dict(io_dtype=capi.SSM_F32), capi.SSM_ERR_UNSUPPORTED),
    (dict(io_dtype=4), capi.SSM_ERR_INVALID_ARG),
    (dict(x=None), capi.SSM_ERR_INVALID_ARG),
    (dict(A=None), capi.SSM_ERR_INVALID_ARG),
    (dict(x=FAKE + 8), capi.SSM_ERR_INVALID_ARG),                # not 16-byte aligned
    (dict(dt=FAKE + (1 << 22) + 1), capi.SSM_ERR_INVALID_ARG),
    (dict(y=FAKE + 4096), capi.SSM_ERR_INVALID_ARG),             # y overlaps x
    (dict(dt_softplus=2), capi.SSM_ERR_INVALID_ARG),
])
def test_ssd_rejects_before_launch(over, code):
    assert capi.ssm_ssd_fwd(valid_ssd(**over), None) == code
    assert capi.lib().ssm_ssd_fwd(None, None) == capi.SSM_ERR_INVALID_ARG


def test_selftest_flag_wait_rejects_before_launch():
    lib = capi.lib()
    assert lib.ssm_selftest_flag_wait(None, 256, 10, None) == capi.SSM_ERR_INVALID_ARG
    assert lib.ssm_selftest_flag_wait(ctypes.c_void_p(FAKE), 100, 10, None) == capi.SSM_ERR_INVALID_ARG
    assert lib.ssm_selftest_flag_wait(ctypes.c_void_p(FAKE + 8), 256, 10, None) == capi.SSM_ERR_INVALID_ARG
    assert lib.ssm_selftest_flag_wait(ctypes.c_void_p(FAKE), 256, 0, None) == capi.SSM_ERR_INVALID_ARG
    assert lib.ssm_selftest_flag_wait(ctypes.c_void_p(FAKE), 256, (1 << 24) + 1, None) == capi.SSM_ERR_INVALID_ARG
