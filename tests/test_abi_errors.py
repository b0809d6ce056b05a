"""Host-side argument checking of the entry points beyond ssd_fwd / ssd_bwd:
every error below is returned before anything is launched, so these run on
a machine without a GPU (the status codes of include/ssd.h)."""
import ctypes

import pytest

import state_space_model_sm_gb300 as ssd
from state_space_model_sm_gb300 import _native

OK, INVALID, UNSUPPORTED, WORKSPACE = 0, 1, 2, 3
D = ctypes.c_void_p(256)  # a 256-byte-aligned stand-in address, never dereferenced
BIG = ctypes.c_size_t(1 << 40)


@pytest.fixture(scope="module")
def lib():
    return ssd.load_library()


def shape(**kw):
    a = dict(batch=1, seqlen=512, nheads=4, headdim=64, dstate=128, ngroups=1, chunk_size=256,
             in_dtype=ssd.SSD_BF16, out_dtype=ssd.SSD_F32)
    a.update(kw)
    return ssd.make_shape(**a)


def norm_shape(rows=64, features=512, group_size=128, eps=1e-5, in_dtype=1, out_dtype=1):
    return _native.NormShape(rows, features, group_size, eps, in_dtype, out_dtype)


# ------------------------------------------------------ context parallel

@pytest.mark.parametrize("kw", [dict(batch=0), dict(seqlen=0), dict(nheads=0), dict(in_dtype=5),
                                dict(seqlen=1 << 30)])
def test_segment_decay_bad_shape(lib, kw):
    s = shape(**kw)
    assert lib.ssd_segment_decay_workspace_size(ctypes.byref(s)) == 0
    assert lib.ssd_segment_decay(ctypes.byref(s), D, None, D, D, D, BIG, None) == INVALID


def test_segment_decay_null_and_workspace(lib):
    s = shape()
    assert lib.ssd_segment_decay_workspace_size(ctypes.byref(s)) > 0
    assert lib.ssd_segment_decay(ctypes.byref(s), None, None, D, D, D, BIG, None) == INVALID
    assert lib.ssd_segment_decay(ctypes.byref(s), D, None, None, D, D, BIG, None) == INVALID
    assert lib.ssd_segment_decay(ctypes.byref(s), D, None, D, None, D, BIG, None) == INVALID
    assert lib.ssd_segment_decay(ctypes.byref(s), D, None, D, D, None, BIG, None) == WORKSPACE
    assert lib.ssd_segment_decay(ctypes.byref(s), D, None, D, D, D, ctypes.c_size_t(8),
                                 None) == WORKSPACE
    odd = ctypes.c_void_p(260)  # workspace holds doubles: 8-byte alignment
    assert lib.ssd_segment_decay(ctypes.byref(s), D, None, D, D, odd, BIG, None) == WORKSPACE


@pytest.mark.parametrize("R,rank,direction,bh,pn", [
    (0, 0, 0, 4, 8), (2, 2, 0, 4, 8), (2, -1, 1, 4, 8), (2, 0, 2, 4, 8), (2, 0, 0, 0, 8),
    (2, 0, 0, 4, 0)])
def test_state_scan_bad_arguments(lib, R, rank, direction, bh, pn):
    assert lib.ssd_state_scan(R, rank, direction, bh, pn, D, D, D, None) == INVALID


def test_state_scan_null_pointers(lib):
    assert lib.ssd_state_scan(2, 0, 0, 4, 8, None, D, D, None) == INVALID
    assert lib.ssd_state_scan(2, 0, 0, 4, 8, D, None, D, None) == INVALID
    assert lib.ssd_state_scan(2, 0, 0, 4, 8, D, D, None, None) == INVALID


@pytest.mark.parametrize("kw,code", [(dict(batch=0), INVALID), (dict(chunk_size=512), UNSUPPORTED),
                                     (dict(nheads=4, ngroups=3), INVALID)])
def test_first_passes_bad_shape(lib, kw, code):
    s = shape(**kw)
    assert lib.ssd_fwd_final_state(ctypes.byref(s), D, D, None, D, D, None, D, D, BIG,
                                   None) == code
    assert lib.ssd_bwd_dinit(ctypes.byref(s), D, None, D, D, D, None, D, D, BIG, None) == code


def test_first_passes_null_and_workspace(lib):
    s = shape()
    # final state: x, dt, A, B and the output are required
    for i in (0, 1, 3, 4, 6):
        args = [D, D, None, D, D, None, D]
        args[i] = None
        assert lib.ssd_fwd_final_state(ctypes.byref(s), *args, D, BIG, None) == INVALID, i
    assert lib.ssd_fwd_final_state(ctypes.byref(s), D, D, None, D, D, None, D, D,
                                   ctypes.c_size_t(16), None) == WORKSPACE
    odd = ctypes.c_void_p(257)
    assert lib.ssd_fwd_final_state(ctypes.byref(s), odd, D, None, D, D, None, D, D, BIG,
                                   None) == INVALID
    # initial-state gradient: dt, A, C, dy and the output are required
    for i in (0, 2, 3, 4, 6):
        args = [D, None, D, D, D, None, D]
        args[i] = None
        assert lib.ssd_bwd_dinit(ctypes.byref(s), *args, D, BIG, None) == INVALID, i
    assert lib.ssd_bwd_dinit(ctypes.byref(s), D, None, D, D, D, None, D, None, BIG,
                             None) == WORKSPACE


# ------------------------------------------------------------ gated norm

@pytest.mark.parametrize("kw,code", [
    (dict(features=20), INVALID),                 # not a multiple of 8
    (dict(group_size=96), INVALID),               # does not divide 512
    (dict(eps=-1.0), INVALID), (dict(in_dtype=3), INVALID), (dict(rows=-1), INVALID),
    (dict(rows=1 << 30), INVALID),
    (dict(features=8192, group_size=512), UNSUPPORTED),   # more than 512 threads a row
    (dict(features=24, group_size=8), UNSUPPORTED),       # 3 threads a row
    (dict(features=96, group_size=24), UNSUPPORTED),      # groups of 3 threads
])
def test_gated_norm_bad_shapes(lib, kw, code):
    s = norm_shape(**kw)
    assert lib.ssd_gated_norm_fwd(ctypes.byref(s), D, D, D, D, None, None) == code
    assert lib.ssd_gated_norm_bwd(ctypes.byref(s), D, D, D, None, D, D, D, D, D, BIG,
                                  None) == code
    if code == INVALID or code == UNSUPPORTED:
        assert lib.ssd_gated_norm_workspace_size(ctypes.byref(s)) == 0


def test_gated_norm_null_alignment_workspace(lib):
    s = norm_shape()
    assert lib.ssd_gated_norm_fwd(ctypes.byref(s), None, D, D, D, None, None) == INVALID
    assert lib.ssd_gated_norm_fwd(ctypes.byref(s), D, D, None, D, None, None) == INVALID
    odd = ctypes.c_void_p(264)  # 8-byte but not 16-byte aligned
    assert lib.ssd_gated_norm_fwd(ctypes.byref(s), odd, D, D, D, None, None) == INVALID
    assert lib.ssd_gated_norm_bwd(ctypes.byref(s), D, D, D, None, D, D, D, None, D, BIG,
                                  None) == INVALID          # no dw
    assert lib.ssd_gated_norm_bwd(ctypes.byref(s), D, D, D, None, D, D, D, D, None, BIG,
                                  None) == WORKSPACE
    assert lib.ssd_gated_norm_bwd(ctypes.byref(s), D, D, D, None, D, D, D, D, D,
                                  ctypes.c_size_t(64), None) == WORKSPACE


def test_gated_norm_zero_rows_forward_launches_nothing(lib):
    s = norm_shape(rows=0)
    assert lib.ssd_gated_norm_fwd(ctypes.byref(s), None, None, None, None, None, None) == OK
