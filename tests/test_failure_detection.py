"""Failure detection without a GPU fault: a bounded device-side wait that
nothing completes must expire, record SSD_ERR_TIMEOUT in the status word and
leave the context usable for the next call."""
import ctypes

import numpy as np
import pytest

import oracle
from parity_util import assert_close, to_np
from state_space_model_sm_gb300 import _native
from state_space_model_sm_gb300.inputs import SSDShape, make_inputs, to_torch

pytestmark = pytest.mark.gpu


def test_bounded_wait_reports_timeout_and_context_survives(cuda_lib):
    import torch
    lib = _native.load()
    assert cuda_lib.device_status() == 0
    stream = torch.cuda.current_stream().cuda_stream
    assert lib.ssd_selftest_timeout(ctypes.c_void_p(stream)) == 0
    assert cuda_lib.device_status() == 5           # SSD_ERR_TIMEOUT, read and cleared
    assert cuda_lib.device_status() == 0
    # the suspending wait of the gated-norm row ring ends the same way
    assert lib.ssd_selftest_timeout_suspend(ctypes.c_void_p(stream)) == 0
    assert cuda_lib.device_status() == 5
    assert cuda_lib.device_status() == 0
    # the context still runs kernels correctly
    inp = make_inputs(SSDShape(1, 300, 4, 64, 128, 1, 256), seed=8, dtype="bf16")
    t = to_torch(inp)
    y, _ = cuda_lib.ssd_fwd(t["x"], t["dt"], t["dt_bias"], t["A"], t["B"], t["C"], t["D"],
                            chunk_size=256)
    torch.cuda.synchronize()
    y_ref, _ = oracle.ssd_fwd(*oracle.from_inputs(inp))
    assert_close("y", to_np(y), y_ref, "bf16")
    assert cuda_lib.device_status() == 0


def test_nonfinite_outputs_are_reported_when_the_check_is_on(cuda_lib):
    """The opt-in NaN / Inf scan: an input NaN (made on the host) propagates to
    the outputs and the scan records SSD_ERR_NONFINITE (6); clean inputs
    leave the status at 0; with the scan off nothing is recorded."""
    import torch
    inp = make_inputs(SSDShape(1, 300, 4, 64, 128, 1, 128), seed=9, dtype="bf16", with_dy=True)
    t = to_torch(inp)
    prev = cuda_lib.set_check_finite(True)
    try:
        cuda_lib.ssd_fwd(t["x"], t["dt"], t["dt_bias"], t["A"], t["B"], t["C"], t["D"],
                         chunk_size=128)
        cuda_lib.ssd_bwd(t["x"], t["dt"], t["dt_bias"], t["A"], t["B"], t["C"], t["D"], 128,
                         None, t["dy"])
        assert cuda_lib.device_status() == 0
        x_bad = t["x"].clone()
        x_bad[0, 17, 2, 5] = float("nan")
        cuda_lib.ssd_fwd(x_bad, t["dt"], t["dt_bias"], t["A"], t["B"], t["C"], t["D"],
                         chunk_size=128)
        assert cuda_lib.device_status() == 6        # SSD_ERR_NONFINITE, read and cleared
        assert cuda_lib.device_status() == 0
        dy_bad = t["dy"].clone()
        dy_bad[0, 250, 1, 0] = float("inf")
        with pytest.raises(cuda_lib.SSDError) as err:
            cuda_lib.ssd_bwd(t["x"], t["dt"], t["dt_bias"], t["A"], t["B"], t["C"], t["D"],
                             128, None, dy_bad, check=True)
        assert err.value.status == 6
        cuda_lib.set_check_finite(False)
        cuda_lib.ssd_fwd(x_bad, t["dt"], t["dt_bias"], t["A"], t["B"], t["C"], t["D"],
                         chunk_size=128)
        torch.cuda.synchronize()
        assert cuda_lib.device_status() == 0        # off: not scanned
    finally:
        cuda_lib.set_check_finite(prev)
