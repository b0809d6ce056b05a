"""Gated RMSNorm kernels (``ssd_gated_norm_fwd`` / ``_bwd``) against the fp64
oracle (``oracle/gated_norm.py``) on identical seeded inputs.

Tolerances: fp32 inputs and outputs, relative L2 <= 1e-4; bf16 inputs with
fp32 outputs, the SSD path's bar (max-abs <= 2e-2, relative L2 <= 1e-2);
bf16 outputs additionally carry one rounding to bf16 (8 significant bits),
so each element must lie within 2^-8 |ref| + 1e-5 of the oracle.
"""
import numpy as np
import pytest

from oracle import gated_norm as gn
from parity_util import assert_close, to_np
from state_space_model_sm_gb300.inputs import (NORM_WORKLOADS, NormShape, make_norm_inputs,
                                               make_norm_workload)

pytestmark = pytest.mark.gpu


def _dev(inp):
    import torch
    tdt = torch.bfloat16 if inp.dtype == "bf16" else torch.float32

    def cv(a, dt=tdt):
        return torch.from_numpy(np.ascontiguousarray(a)).to("cuda", dt)
    return cv(inp.y), cv(inp.z), cv(inp.w, torch.float32), cv(inp.dout)


def _check(name, got, ref, in_dtype, out_bf16):
    if out_bf16:
        d = np.abs(got - ref)
        bound = 2.0 ** -8 * np.abs(ref) + 1e-5
        worst = int(np.argmax(d - bound))
        assert np.all(d <= bound), f"{name}: |d|={d.flat[worst]} > {bound.flat[worst]}"
        return
    assert_close(name, got, ref, in_dtype)


CASES = [
    # rows, features, group_size, dtype
    (37, 64, 16, "f32"),        # 2 threads per group, 64 rows per item: one ragged item
    (1000, 128, 8, "f32"),      # one thread per group
    (515, 256, 256, "bf16"),    # one warp per group, ragged last item
    (301, 1536, 1536, "bf16"),  # a group of 6 warps (layer width), 2 rows per item
    (129, 4096, 512, "bf16"),   # groups of 2 warps (hybrid width), 1 row per item
    (70, 4096, 4096, "f32"),    # one group of 16 warps
]


@pytest.mark.parametrize("rows,features,gs,dtype", CASES)
@pytest.mark.parametrize("out_bf16", [False, True])
def test_forward_backward_match_oracle(cuda_lib, rows, features, gs, dtype, out_bf16):
    import torch
    inp = make_norm_inputs(NormShape(rows, features, gs), seed=rows + features, dtype=dtype)
    y, z, w, dout = _dev(inp)
    odt = torch.bfloat16 if out_bf16 else torch.float32
    out, rstd = cuda_lib.gated_norm_fwd(y, z, w, gs, eps=inp.shape.eps, out_dtype=odt)
    ref, rstd_ref = gn.gated_rmsnorm_fwd(inp.y, inp.z, inp.w, gs, eps=inp.shape.eps)
    _check("out", to_np(out), ref, dtype, out_bf16)
    assert_close("rstd", to_np(rstd), rstd_ref, "f32")
    g_ref = gn.gated_rmsnorm_bwd(inp.y, inp.z, inp.w, inp.dout, gs, eps=inp.shape.eps)
    for saved in (rstd, None):
        g = cuda_lib.gated_norm_bwd(y, z, w, dout, gs, eps=inp.shape.eps, rstd=saved,
                                    out_dtype=odt)
        _check("dy", to_np(g["dy"]), g_ref["dy"], dtype, out_bf16)
        _check("dz", to_np(g["dz"]), g_ref["dz"], dtype, out_bf16)
        assert_close("dw", to_np(g["dw"]), g_ref["dw"], "f32")
    assert cuda_lib.device_status() == 0


@pytest.mark.parametrize("name", ["norm_layer_bf16", "norm_hybrid_bf16"])
def test_full_size_sampled_rows_and_dw(cuda_lib, name):
    """The full workload in the configuration the benchmark times: out, dy,
    dz on 256 sampled rows against the oracle of those rows; dw (a sum over
    every row) against the oracle summed over row blocks."""
    import torch
    inp = make_norm_workload(name)
    sh = inp.shape
    y, z, w, dout = _dev(inp)
    out, rstd = cuda_lib.gated_norm_fwd(y, z, w, sh.group_size, eps=sh.eps)
    g = cuda_lib.gated_norm_bwd(y, z, w, dout, sh.group_size, eps=sh.eps, rstd=rstd)
    torch.cuda.synchronize()
    rows = np.sort(np.random.default_rng(7).choice(sh.rows, 256, replace=False))
    ref, _ = gn.gated_rmsnorm_fwd(inp.y[rows], inp.z[rows], inp.w, sh.group_size, eps=sh.eps)
    _check("out", to_np(out[torch.from_numpy(rows).cuda()]), ref, "bf16", True)
    gr = gn.gated_rmsnorm_bwd(inp.y[rows], inp.z[rows], inp.w, inp.dout[rows], sh.group_size,
                              eps=sh.eps)
    idx = torch.from_numpy(rows).cuda()
    _check("dy", to_np(g["dy"][idx]), gr["dy"], "bf16", True)
    _check("dz", to_np(g["dz"][idx]), gr["dz"], "bf16", True)
    dw_ref = np.zeros(sh.features)
    for r0 in range(0, sh.rows, 2048):
        sl = slice(r0, r0 + 2048)
        dw_ref += gn.gated_rmsnorm_bwd(inp.y[sl], inp.z[sl], inp.w, inp.dout[sl], sh.group_size,
                                       eps=sh.eps)["dw"]
    assert_close("dw", to_np(g["dw"]), dw_ref, "f32")
    assert cuda_lib.device_status() == 0


def test_dw_is_deterministic(cuda_lib):
    import torch
    inp = make_norm_inputs(NormShape(3000, 1536, 1536), seed=9, dtype="bf16")
    y, z, w, dout = _dev(inp)
    a = cuda_lib.gated_norm_bwd(y, z, w, dout, 1536)["dw"].clone()
    b = cuda_lib.gated_norm_bwd(y, z, w, dout, 1536)["dw"]
    assert torch.equal(a, b)


def test_zero_rows(cuda_lib):
    import torch
    y = torch.empty((0, 256), dtype=torch.bfloat16, device="cuda")
    w = torch.ones(256, device="cuda")
    out, _ = cuda_lib.gated_norm_fwd(y, y, w, 64)
    assert out.shape == (0, 256)
    g = cuda_lib.gated_norm_bwd(y, y, w, y, 64)
    assert torch.count_nonzero(g["dw"]) == 0


@pytest.mark.parametrize("features,gs,status", [
    (24, 8, 2),       # a row of 3 threads does not tile a warp: unsupported
    (8192, 512, 2),   # wider than one CTA row: unsupported
    (96, 24, 2),      # groups of 3 threads: unsupported
    (64, 24, 1),      # group does not divide the row: invalid
])
def test_rejected_shapes(cuda_lib, features, gs, status):
    import torch
    y = torch.zeros((4, features), dtype=torch.float32, device="cuda")
    w = torch.ones(features, device="cuda")
    with pytest.raises(cuda_lib.SSDError) as e:
        cuda_lib.gated_norm_fwd(y, y, w, gs)
    assert e.value.status == status
