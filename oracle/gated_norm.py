"""Gated RMSNorm in fp64 numpy -- TEST INFRASTRUCTURE (see ``oracle``).

The step that follows the SSD output in a Mamba-2 layer: its backward is the
kernel ``_layer_norm_bwd`` (step bwd_2 in the per-kernel table of
"Optimizing Mamba-2 kernels for the B200", section "Latency and speedup by
kernel"; the 3.18x case discussed under "The highway got wider, but we
didn't add any cars").  The pages name the kernel but do not write out its
arithmetic.  The reading taken here is the Mamba-2 block's output
normalisation: the SSD output y is gated by silu(z) and then RMS-normalised
over groups of ``group_size`` consecutive features, scaled by a per-feature
weight, with no bias (the gate applied before the norm):

  u       = y * silu(z),             silu(z) = z * sigmoid(z)
  rstd_g  = 1 / sqrt(mean_{j in g} u_j^2 + eps)       per row and group g
  out_j   = u_j * rstd_g * w_j

and its backward for an upstream gradient dout:

  xhat_j  = u_j * rstd_g,  gx_j = dout_j * w_j
  dw_j    = sum over rows of dout_j * xhat_j
  du_j    = rstd_g * (gx_j - xhat_j * mean_{k in g}(gx_k * xhat_k))
  dy_j    = du_j * silu(z_j)
  dz_j    = du_j * y_j * silu'(z_j),  silu'(z) = sigmoid(z) (1 + z (1 - sigmoid(z)))

Rows are the flattened (batch, seqlen) positions; features the flattened
(nheads, headdim).  Pins: ``tests/test_oracle_gated_norm.py``.
"""
from __future__ import annotations

import numpy as np


def sigmoid(z):
    # 1 / (1 + e^-z), taken as e^z / (1 + e^z) for z < 0 (no overflow, no
    # cancellation in either tail)
    z = np.asarray(z, dtype=np.float64)
    e = np.exp(-np.abs(z))
    return np.where(z >= 0, 1.0 / (1.0 + e), e / (1.0 + e))


def silu(z):
    z = np.asarray(z, dtype=np.float64)
    return z * sigmoid(z)


def silu_grad(z):
    z = np.asarray(z, dtype=np.float64)
    s = sigmoid(z)
    return s * (1.0 + z * (1.0 - s))


def _grouped(a, group_size):
    M, D = a.shape
    if D % group_size != 0:
        raise ValueError("group_size must divide the feature count")
    return a.reshape(M, D // group_size, group_size)


def gated_rmsnorm_fwd(y, z, w, group_size, eps=1e-5):
    """Returns (out (M, D), rstd (M, D // group_size)), fp64."""
    y = np.asarray(y, dtype=np.float64)
    z = np.asarray(z, dtype=np.float64)
    w = np.asarray(w, dtype=np.float64)
    M, D = y.shape
    u = _grouped(y * silu(z), group_size)
    rstd = 1.0 / np.sqrt(np.mean(u * u, axis=2) + eps)
    out = (u * rstd[:, :, None]).reshape(M, D) * w[None, :]
    return out, rstd


def gated_rmsnorm_bwd(y, z, w, dout, group_size, eps=1e-5):
    """Returns dict dy, dz (M, D) and dw (D,), fp64."""
    y = np.asarray(y, dtype=np.float64)
    z = np.asarray(z, dtype=np.float64)
    w = np.asarray(w, dtype=np.float64)
    dout = np.asarray(dout, dtype=np.float64)
    M, D = y.shape
    g = silu(z)
    u = _grouped(y * g, group_size)
    rstd = 1.0 / np.sqrt(np.mean(u * u, axis=2) + eps)
    xhat = u * rstd[:, :, None]
    gx = _grouped(dout * w[None, :], group_size)
    c = np.mean(gx * xhat, axis=2)
    du = (rstd[:, :, None] * (gx - xhat * c[:, :, None])).reshape(M, D)
    dw = np.sum(dout * xhat.reshape(M, D), axis=0)
    return dict(dy=du * g, dz=du * y * silu_grad(z), dw=dw)
