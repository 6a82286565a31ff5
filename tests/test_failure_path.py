"""The device-side failure path, exercised without a fault: a bounded wait on a
flag that nothing sets records SSM_ERR_TIMEOUT in the workspace status word,
the host reads it, and the context stays usable for the next scan."""

import pytest
import torch

from mamba_selective_scan_02_b300 import api, capi
from mamba_selective_scan_02_b300.inputs import make_inputs


@pytest.mark.gpu
def test_bounded_wait_times_out_and_reports():
    ws = torch.zeros(1024, dtype=torch.uint8, device="cuda")
    st = torch.cuda.current_stream().cuda_stream
    assert capi.ssm_selftest_flag_wait(ws.data_ptr(), ws.numel(), 1 << 12, st) == capi.SSM_OK
    assert api.workspace_status(ws) == capi.SSM_ERR_TIMEOUT
    # the context still runs a scan, and a fresh workspace reports no error
    inp = make_inputs("small_layer_L2048", device="cuda", batch=1, dim=64, seqlen=512, seed=9)
    y, hL = api.scan_fwd(inp["u"], inp["delta"], inp["A"], inp["B"], inp["C"], inp["Dskip"], inp["z"],
                         inp["bias"], chunk_len=64, workspace=None)
    torch.cuda.synchronize()
    assert torch.isfinite(y.float()).all() and torch.isfinite(hL).all()
    ws2 = torch.zeros(4 << 20, dtype=torch.uint8, device="cuda")
    p = api.scan_params(inp["u"], inp["delta"], inp["A"], inp["B"], inp["C"], inp["Dskip"], inp["z"], inp["bias"],
                        None, y=torch.empty_like(inp["u"]), workspace=ws2)
    assert capi.ssm_scan_fwd(p, st) == capi.SSM_OK
    assert api.workspace_status(ws2) == capi.SSM_OK
