"""ssd_fwd_noalloc: the forward for callers that cannot allocate device memory.

It must give the results of ssd_fwd (which takes a caller-allocated
workspace) on consecutive calls that share its fixed internal scratch, and
refuse shapes whose workspace does not fit that scratch.  Collected last so
that a failure here cannot hide the other tests' results.
"""
import ctypes

import numpy as np
import pytest

import oracle
from parity_util import assert_close, stats, to_np
from state_space_model_sm_gb300 import _native
from state_space_model_sm_gb300.inputs import SSDShape, make_inputs, to_torch

pytestmark = pytest.mark.gpu


def _p(t):
    return None if t is None else ctypes.c_void_p(t.data_ptr())


def _call_noalloc(ssd, inp):
    import torch
    t = to_torch(inp)
    s = inp.shape
    shape = ssd.make_shape(s.batch, s.seqlen, s.nheads, s.headdim, s.dstate, s.ngroups,
                           s.chunk_size, ssd.SSD_BF16 if inp.dtype == "bf16" else ssd.SSD_F32,
                           ssd.SSD_F32)
    y = torch.full((s.batch, s.seqlen, s.nheads, s.headdim), float("nan"), device="cuda")
    final = torch.full((s.batch, s.nheads, s.headdim, s.dstate), float("nan"), device="cuda")
    stream = torch.cuda.current_stream().cuda_stream
    st = _native.load().ssd_fwd_noalloc(ctypes.byref(shape), _p(t["x"]), _p(t["dt"]),
                                        _p(t["dt_bias"]), _p(t["A"]), _p(t["B"]), _p(t["C"]),
                                        _p(t["D"]), _p(t["init"]), _p(y), _p(final),
                                        ctypes.c_void_p(stream))
    torch.cuda.synchronize()
    return st, y, final


def _call_with_workspace(ssd, inp):
    import torch
    t = to_torch(inp)
    y, final = ssd.ssd_fwd(t["x"], t["dt"], t["dt_bias"], t["A"], t["B"], t["C"], t["D"],
                           chunk_size=inp.shape.chunk_size, init_states=t["init"])
    torch.cuda.synchronize()
    return y, final


def test_noalloc_matches_workspace_forward_on_consecutive_calls(cuda_lib):
    cases = [make_inputs(SSDShape(2, 1000, 8, 64, 128, 2, 128), seed=21, dtype="bf16",
                         init_std=0.1),
             make_inputs(SSDShape(1, 300, 4, 16, 16, 1, 64), seed=22, dtype="f32", init_std=0.5)]
    for inp in cases:     # two calls in a row, different shapes, one scratch
        st, y, final = _call_noalloc(cuda_lib, inp)
        assert st == 0, cuda_lib.load_library().ssd_strerror(st)
        y_ref, f_ref = _call_with_workspace(cuda_lib, inp)
        tol = 1e-4 if inp.dtype == "f32" else 1e-2
        for got, ref in ((y, y_ref), (final, f_ref)):
            s = stats(to_np(got), to_np(ref))
            assert np.isfinite(to_np(got)).all()
            assert s["rel_l2"] <= tol and (inp.dtype == "f32" or s["max_abs"] <= 2e-2), s
        # and against the CPU oracle itself, at the library's parity bars
        y_or, f_or = oracle.ssd_fwd(*oracle.from_inputs(inp))
        assert_close("y", to_np(y), y_or, inp.dtype)
        assert_close("final", to_np(final), f_or, inp.dtype)
    assert cuda_lib.device_status() == 0


def test_noalloc_rejects_shapes_beyond_its_scratch(cuda_lib):
    lib = _native.load()
    cap = lib.ssd_noalloc_scratch_bytes()
    assert cap == 64 << 20
    s = cuda_lib.make_shape(4, 4096, 24, 64, 128, 1, 256, cuda_lib.SSD_BF16, cuda_lib.SSD_F32)
    assert lib.ssd_fwd_workspace_size(ctypes.byref(s)) > cap
    dummy = ctypes.c_void_p(256)
    st = lib.ssd_fwd_noalloc(ctypes.byref(s), dummy, dummy, None, dummy, dummy, dummy, None,
                             None, dummy, None, None)
    assert st == 3  # SSD_ERR_WORKSPACE, nothing launched
