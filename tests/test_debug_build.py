"""The debug build (libssmscan_debug.so, -DSSM_DEBUG): every global store
checks its element range against the buffer it writes and records, instead of
trapping, any that falls outside.

A child process opens the debug build (SSM_SCAN_LIBRARY=debug) and runs
small, ragged calls of every entry point (tests/debug_cases.py); its debug
status must stay SSM_OK, and its outputs must match the release library's on
the same calls: bit for bit, except the backward's fp32 atomic sums, held to a
tight tolerance.
"""

import os
import subprocess
import sys

import pytest
import torch

from mamba_selective_scan_02_b300 import capi

HERE = os.path.dirname(os.path.abspath(__file__))


def test_release_build_has_no_debug_words():
    # the release library answers without touching the device
    if capi.debug_selected():
        pytest.skip("this process runs the debug build")
    assert capi.ssm_debug_status(False) == capi.SSM_ERR_UNSUPPORTED


@pytest.mark.gpu
def test_debug_build_index_checks_stay_clean_and_match_release(tmp_path):
    sys.path.insert(0, HERE)
    import debug_cases

    out = tmp_path / "debug_outputs.pt"
    env = dict(os.environ, SSM_SCAN_LIBRARY="debug")
    r = subprocess.run([sys.executable, os.path.join(HERE, "debug_cases.py"), str(out)], env=env,
                       capture_output=True, text=True, timeout=1200)
    assert r.returncode == 0, r.stdout[-3000:] + r.stderr[-3000:]
    res = torch.load(out)
    assert res["library"].endswith("libssmscan_debug.so")
    assert res["before"] == capi.SSM_OK, capi.status_string(res["before"])
    assert res["after"] == capi.SSM_OK, capi.status_string(res["after"])
    want = debug_cases.run_cases()
    assert set(res["outputs"]) == set(want)
    for case, outs in want.items():
        for k, v in outs.items():
            got = res["outputs"][case][k]
            if case.startswith("bwd"):
                g, w = got.double(), v.double()
                scale = 1.0 + w.abs() + w.pow(2).mean().sqrt()
                assert torch.all((g - w).abs() <= 1e-5 * scale), f"{case} {k}"
            else:
                assert torch.equal(got, v), f"{case} {k}: debug and release builds differ"
