"""Pins of the gated RMSNorm oracle (``oracle/gated_norm.py``) to facts
outside itself: PyTorch's own rms_norm and silu (library routines) and
autograd through them, central finite differences, and closed forms."""
import numpy as np
import pytest

from oracle import gated_norm as gn


def _data(M=6, D=24, gs=8, seed=0, zscale=2.0):
    rng = np.random.default_rng(seed)
    y = rng.standard_normal((M, D))
    z = rng.standard_normal((M, D)) * zscale
    w = 1.0 + 0.3 * rng.standard_normal(D)
    dout = rng.standard_normal((M, D))
    return y, z, w, dout, gs


def _torch_ref(y, z, w, gs, eps):
    import torch
    import torch.nn.functional as F
    yt, zt, wt = (torch.tensor(a, dtype=torch.float64, requires_grad=True) for a in (y, z, w))
    M, D = y.shape
    u = (yt * F.silu(zt)).reshape(M, D // gs, gs)
    out = F.rms_norm(u, (gs,), eps=eps).reshape(M, D) * wt
    return out, (yt, zt, wt)


@pytest.mark.parametrize("gs", [8, 24, 4])
def test_forward_matches_torch_rms_norm_of_gated_input(gs):
    y, z, w, _, _ = _data(gs=gs)
    out, rstd = gn.gated_rmsnorm_fwd(y, z, w, gs, eps=1e-5)
    ref, _ = _torch_ref(y, z, w, gs, 1e-5)
    np.testing.assert_allclose(out, ref.detach().numpy(), rtol=1e-12, atol=1e-13)
    assert rstd.shape == (y.shape[0], y.shape[1] // gs)


@pytest.mark.parametrize("gs", [8, 24])
def test_backward_matches_torch_autograd(gs):
    import torch
    y, z, w, dout, _ = _data(gs=gs, seed=1)
    g = gn.gated_rmsnorm_bwd(y, z, w, dout, gs, eps=1e-5)
    out, (yt, zt, wt) = _torch_ref(y, z, w, gs, 1e-5)
    out.backward(torch.tensor(dout))
    np.testing.assert_allclose(g["dy"], yt.grad.numpy(), rtol=1e-10, atol=1e-12)
    np.testing.assert_allclose(g["dz"], zt.grad.numpy(), rtol=1e-10, atol=1e-12)
    np.testing.assert_allclose(g["dw"], wt.grad.numpy(), rtol=1e-10, atol=1e-12)


def test_backward_matches_central_finite_differences():
    y, z, w, dout, gs = _data(M=3, D=8, gs=4, seed=2)
    eps = 1e-3

    def loss(y_, z_, w_):
        return float(np.sum(dout * gn.gated_rmsnorm_fwd(y_, z_, w_, gs, eps=eps)[0]))

    g = gn.gated_rmsnorm_bwd(y, z, w, dout, gs, eps=eps)
    h = 1e-6
    for name, arr in (("dy", y), ("dz", z), ("dw", w)):
        fd = np.zeros_like(arr)
        for idx in np.ndindex(arr.shape):
            p, m = arr.copy(), arr.copy()
            p[idx] += h
            m[idx] -= h
            args_p = dict(y_=y, z_=z, w_=w)
            args_m = dict(y_=y, z_=z, w_=w)
            key = {"dy": "y_", "dz": "z_", "dw": "w_"}[name]
            args_p[key], args_m[key] = p, m
            fd[idx] = (loss(**args_p) - loss(**args_m)) / (2 * h)
        np.testing.assert_allclose(g[name], fd, rtol=1e-6, atol=1e-7, err_msg=name)


def test_zero_gate_closed_form():
    """z = 0: silu = 0 so u = 0, out = 0, rstd = 1/sqrt(eps); the gradient
    reaches z only: dz = rstd * dout * w * y * silu'(0), silu'(0) = 1/2."""
    y, _, w, dout, gs = _data(seed=3)
    z = np.zeros_like(y)
    eps = 1e-5
    out, rstd = gn.gated_rmsnorm_fwd(y, z, w, gs, eps=eps)
    assert np.all(out == 0.0)
    np.testing.assert_allclose(rstd, 1.0 / np.sqrt(eps), rtol=1e-15)
    g = gn.gated_rmsnorm_bwd(y, z, w, dout, gs, eps=eps)
    assert np.all(g["dy"] == 0.0) and np.all(g["dw"] == 0.0)
    np.testing.assert_allclose(g["dz"], dout * w * y * 0.5 / np.sqrt(eps), rtol=1e-13)


def test_group_mean_square_closed_form():
    """With w = 1 each group of out has mean square ms / (ms + eps)."""
    y, z, _, _, gs = _data(seed=4)
    eps = 0.25
    out, _ = gn.gated_rmsnorm_fwd(y, z, np.ones(y.shape[1]), gs, eps=eps)
    u = (y * gn.silu(z)).reshape(y.shape[0], -1, gs)
    ms = np.mean(u * u, axis=2)
    got = np.mean(out.reshape(y.shape[0], -1, gs) ** 2, axis=2)
    np.testing.assert_allclose(got, ms / (ms + eps), rtol=1e-13)


def test_scale_invariance_without_eps():
    y, z, w, _, gs = _data(seed=5)
    a, _ = gn.gated_rmsnorm_fwd(y, z, w, gs, eps=0.0)
    b, _ = gn.gated_rmsnorm_fwd(3.7 * y, z, w, gs, eps=0.0)
    np.testing.assert_allclose(a, b, rtol=1e-13)


def test_silu_and_its_derivative():
    z = np.linspace(-30.0, 30.0, 601)
    np.testing.assert_allclose(gn.sigmoid(z), 1.0 / (1.0 + np.exp(-z)), rtol=1e-14, atol=1e-300)
    h = 1e-6
    fd = (gn.silu(z + h) - gn.silu(z - h)) / (2 * h)
    np.testing.assert_allclose(gn.silu_grad(z), fd, rtol=1e-7, atol=1e-9)
    assert gn.silu(0.0) == 0.0 and gn.silu_grad(0.0) == 0.5


def test_group_size_must_divide():
    y, z, w, _, _ = _data(D=24)
    with pytest.raises(ValueError):
        gn.gated_rmsnorm_fwd(y, z, w, 5)


def test_random_shapes_match_torch_autograd():
    """Property check over random shapes, group sizes, eps and gate scales:
    forward and backward equal torch's rms_norm / silu with autograd."""
    hyp = pytest.importorskip("hypothesis")
    st = pytest.importorskip("hypothesis.strategies")
    import torch

    @hyp.settings(max_examples=40, deadline=None, derandomize=True)
    @hyp.given(rows=st.integers(1, 9), groups=st.integers(1, 4), gs=st.integers(1, 12),
               eps=st.sampled_from([0.0, 1e-5, 0.3]), zscale=st.floats(0.1, 8.0),
               seed=st.integers(0, 2 ** 16))
    def check(rows, groups, gs, eps, zscale, seed):
        D = groups * gs
        rng = np.random.default_rng(seed)
        y = rng.standard_normal((rows, D))
        z = rng.standard_normal((rows, D)) * zscale
        w = 1.0 + 0.3 * rng.standard_normal(D)
        dout = rng.standard_normal((rows, D))
        out, rstd = gn.gated_rmsnorm_fwd(y, z, w, gs, eps=eps)
        g = gn.gated_rmsnorm_bwd(y, z, w, dout, gs, eps=eps)
        ref, (yt, zt, wt) = _torch_ref(y, z, w, gs, eps)
        ref.backward(torch.tensor(dout))
        np.testing.assert_allclose(out, ref.detach().numpy(), rtol=1e-10, atol=1e-12)
        # the backward subtracts terms of size rstd |dout w| (times |y| or |z|
        # factors) that cancel exactly in degenerate groups (one element: xhat
        # = +-1, du = 0); rounding there is relative to that size
        scale = (float(rstd.max()) * float(np.abs(dout * w).max()) *
                 max(1.0, float(np.abs(y).max())) * max(1.0, float(np.abs(z).max())))
        for name, t in (("dy", yt), ("dz", zt), ("dw", wt)):
            np.testing.assert_allclose(g[name], t.grad.numpy(), rtol=1e-8,
                                       atol=1e-12 * scale + 1e-12, err_msg=name)
    check()


def test_norm_inputs_recipe():
    """The norm workloads' seeded inputs: shapes, exact bf16 values, the
    weight's spread around one, and determinism across calls."""
    from state_space_model_sm_gb300.inputs import (NORM_WORKLOADS, NormShape,
                                                   make_norm_inputs)
    a = make_norm_inputs(NormShape(33, 64, 16), seed=3, dtype="bf16")
    b = make_norm_inputs(NormShape(33, 64, 16), seed=3, dtype="bf16")
    for x in (a.y, a.z, a.dout):
        assert x.shape == (33, 64) and x.dtype == np.float32
        assert (x.view(np.uint32) & 0xFFFF == 0).all()      # exactly representable in bf16
    assert a.w.shape == (64,) and abs(float(a.w.mean()) - 1.0) < 0.1
    for k in ("y", "z", "w", "dout"):
        np.testing.assert_array_equal(getattr(a, k), getattr(b, k))
    f = make_norm_inputs(NormShape(5, 16, 8), seed=3, dtype="f32")
    assert (f.y.view(np.uint32) & 0xFFFF != 0).any()       # fp32 keeps its low bits
    with pytest.raises(ValueError):
        make_norm_inputs(NormShape(5, 16, 8), seed=0, dtype="fp16")
    for name, (shape, dtype, _) in NORM_WORKLOADS.items():
        assert shape.features % shape.group_size == 0, name
        assert dtype in ("bf16", "f32"), name
