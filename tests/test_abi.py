"""C-ABI checks that need no GPU: the library loads, exports every symbol
include/ssd.h declares, and rejects bad arguments on the host before any
launch."""
import ctypes
import os
import re

import pytest

import state_space_model_sm_gb300 as ssd
from state_space_model_sm_gb300 import _native

ROOT = os.path.dirname(os.path.dirname(os.path.abspath(__file__)))


def header_functions():
    text = open(os.path.join(ROOT, "include", "ssd.h")).read()
    text = re.sub(r"/\*.*?\*/", "", text, flags=re.S)
    return sorted(set(re.findall(r"\b(ssd_[a-z_]+)\s*\(", text)))


@pytest.fixture(scope="module")
def lib():
    ssd.build()
    return ssd.load_library()


def test_header_lists_the_entry_points():
    fns = header_functions()
    for name in ("ssd_fwd", "ssd_bwd", "ssd_fwd_workspace_size", "ssd_bwd_workspace_size",
                 "ssd_get_device_status", "ssd_strerror"):
        assert name in fns


def test_library_exports_every_declared_symbol(lib):
    for name in header_functions():
        assert hasattr(lib, name), name
        assert name in _native.SIGNATURES, name


def test_status_strings(lib):
    for code in range(7):
        assert lib.ssd_strerror(code) and lib.ssd_strerror(code) != b"unknown status"
    assert b"NaN" in lib.ssd_strerror(6)   # SSD_ERR_NONFINITE
    assert lib.ssd_strerror(99) == b"unknown status"


def test_check_finite_setting_round_trips(lib):
    # host-only: the process-wide switch of the opt-in NaN / Inf output scan
    assert lib.ssd_set_check_finite(1) == 0
    assert lib.ssd_set_check_finite(0) == 1
    assert ssd.set_check_finite(False) is False


def test_noalloc_scratch_size_matches_header_macro(lib):
    text = open(os.path.join(ROOT, "include", "ssd.h")).read()
    m = re.search(r"#define SSD_NOALLOC_SCRATCH_BYTES \(\(size_t\)(\d+) << (\d+)\)", text)
    assert m, "SSD_NOALLOC_SCRATCH_BYTES missing from ssd.h"
    assert lib.ssd_noalloc_scratch_bytes() == int(m.group(1)) << int(m.group(2))


def shape(**kw):
    base = dict(batch=4, seqlen=4096, nheads=24, headdim=64, dstate=128, ngroups=1,
                chunk_size=256, in_dtype=ssd.SSD_BF16, out_dtype=ssd.SSD_F32)
    base.update(kw)
    return ssd.make_shape(**base)


def test_workspace_sizes(lib):
    s = shape()
    fwd, bwd = ssd.fwd_workspace_bytes(s), ssd.bwd_workspace_bytes(s)
    assert fwd > 0 and bwd > fwd
    lay = ssd.fwd_workspace_layout(s)
    nc = 16
    assert lay["dA_cumsum"] >= 4 * 24 * nc * 256 * 4
    assert lay["hprev"] - lay["states"] >= 4 * nc * 24 * 64 * 128 * 4
    assert lay["total"] == fwd
    assert all(lay[k] % 256 == 0 for k in ("delta", "dA_cumsum", "states", "hprev"))
    # grows with the problem
    assert ssd.fwd_workspace_bytes(shape(seqlen=8192)) > fwd


@pytest.mark.parametrize("kw,code", [
    (dict(batch=0), 1), (dict(nheads=24, ngroups=5), 1), (dict(chunk_size=0), 1),
    (dict(chunk_size=512), 2), (dict(headdim=256, dstate=128), 2), (dict(in_dtype=7), 1)])
def test_bad_shapes_are_rejected(lib, kw, code):
    s = shape(**kw)
    assert lib.ssd_fwd_workspace_size(ctypes.byref(s)) == 0
    dummy = ctypes.c_void_p(256)
    st = lib.ssd_fwd(ctypes.byref(s), dummy, dummy, None, dummy, dummy, dummy, None, None, dummy,
                     None, dummy, ctypes.c_size_t(1 << 40), None)
    assert st == code


def test_null_and_workspace_errors_before_launch(lib):
    s = shape()
    dummy = ctypes.c_void_p(256)
    # missing x
    assert lib.ssd_fwd(ctypes.byref(s), None, dummy, None, dummy, dummy, dummy, None, None, dummy,
                       None, dummy, ctypes.c_size_t(1 << 40), None) == 1
    # workspace too small
    assert lib.ssd_fwd(ctypes.byref(s), dummy, dummy, None, dummy, dummy, dummy, None, None, dummy,
                       None, dummy, ctypes.c_size_t(16), None) == 3
    # misaligned bf16 pointer
    odd = ctypes.c_void_p(257)
    assert lib.ssd_fwd(ctypes.byref(s), odd, dummy, None, dummy, dummy, dummy, None, None, dummy,
                       None, dummy, ctypes.c_size_t(1 << 40), None) == 1
    # backward without dy
    assert lib.ssd_bwd(ctypes.byref(s), dummy, dummy, None, dummy, dummy, dummy, None, None, None,
                       None, dummy, dummy, dummy, dummy, dummy, None, None, None, dummy,
                       ctypes.c_size_t(1 << 40), None) == 1
