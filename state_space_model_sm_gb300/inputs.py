"""Seeded synthetic inputs for the Mamba-2 SSD chunked scan.

This module only draws random numbers and rounds them to the storage
precision; it holds none of the SSD arithmetic.  Both the CUDA path and the
CPU oracle are fed from the arrays it returns, so they see bit-identical
inputs.

Recipe (Mamba-2 layer shapes; value distributions of the workload):
  * draw order: dt_bias, A, D, init, dt, x, B, C, dy, dfinal (fixed);
  * x, B, C, dy ~ N(0, 1);
  * the effective step size softplus(dt + dt_bias) is log-uniform on
    [1e-3, 1e-1]: a per-head target v_h and a per-element target u are drawn
    log-uniform, dt_bias[h] = softplus^-1(v_h) and dt = softplus^-1(u) - dt_bias[h];
  * A[h] = -exp(U[0, ln 16]);  D[h] ~ U(0, 1);
  * init ~ N(0, init_std^2) (std reading), zero when init_std == 0.
The generator is numpy's PCG64, whose streams are identical on x86-64 and
aarch64.  Tensors that the kernels read in bf16 (x, dt, B, C, dy) are rounded
to bf16 here (round to nearest even) and returned as float32 arrays holding
exactly representable bf16 values; dt_bias, A, D, init and dfinal stay fp32.
"""
from __future__ import annotations

import dataclasses
from typing import Optional

import numpy as np

DT_MIN, DT_MAX = 1e-3, 1e-1


def round_to_bf16(a: np.ndarray) -> np.ndarray:
    """Round float32 values to the nearest bf16 (ties to even); returns float32."""
    a = np.ascontiguousarray(a, dtype=np.float32)
    u = a.view(np.uint32).astype(np.uint64)
    lsb = (u >> np.uint64(16)) & np.uint64(1)
    u = (u + np.uint64(0x7FFF) + lsb) & np.uint64(0xFFFF0000)
    return u.astype(np.uint32).view(np.float32)


def _inv_softplus(v: np.ndarray) -> np.ndarray:
    # Input preparation only: pick the pre-activation that yields a given step.
    return np.log(np.expm1(v))


@dataclasses.dataclass
class SSDShape:
    batch: int
    seqlen: int
    nheads: int
    headdim: int
    dstate: int
    ngroups: int
    chunk_size: int

    @property
    def nchunks(self) -> int:
        return -(-self.seqlen // self.chunk_size)


@dataclasses.dataclass
class SSDInputs:
    shape: SSDShape
    dtype: str              # "bf16" or "f32": storage type of x, dt, B, C, dy
    x: np.ndarray           # (batch, seqlen, nheads, headdim)
    dt: np.ndarray          # (batch, seqlen, nheads)
    dt_bias: np.ndarray     # (nheads,) fp32
    A: np.ndarray           # (nheads,) fp32
    B: np.ndarray           # (batch, seqlen, ngroups, dstate)
    C: np.ndarray           # (batch, seqlen, ngroups, dstate)
    D: np.ndarray           # (nheads,) fp32
    init: Optional[np.ndarray]    # (batch, nheads, headdim, dstate) fp32 or None
    dy: Optional[np.ndarray] = None       # (batch, seqlen, nheads, headdim)
    dfinal: Optional[np.ndarray] = None   # (batch, nheads, headdim, dstate) fp32


def make_inputs(shape: SSDShape, *, seed: int, dtype: str = "bf16",
                init_std: float = 0.0, with_dy: bool = False,
                dfinal_std: float = 0.0) -> SSDInputs:
    if dtype not in ("bf16", "f32"):
        raise ValueError(f"dtype must be 'bf16' or 'f32', got {dtype!r}")
    Bt, T, H, P = shape.batch, shape.seqlen, shape.nheads, shape.headdim
    N, G = shape.dstate, shape.ngroups
    rng = np.random.Generator(np.random.PCG64(seed))
    lo, hi = np.log(DT_MIN), np.log(DT_MAX)

    v = np.exp(rng.uniform(lo, hi, size=H))
    dt_bias = _inv_softplus(v).astype(np.float32)
    A = (-np.exp(rng.uniform(0.0, np.log(16.0), size=H))).astype(np.float32)
    D = rng.uniform(0.0, 1.0, size=H).astype(np.float32)
    init = None
    if init_std > 0.0:
        init = (rng.standard_normal((Bt, H, P, N), dtype=np.float32)
                * np.float32(init_std)).astype(np.float32)
    u = np.exp(rng.uniform(lo, hi, size=(Bt, T, H)))
    dt = (_inv_softplus(u) - dt_bias.astype(np.float64)[None, None, :]).astype(np.float32)
    x = rng.standard_normal((Bt, T, H, P), dtype=np.float32)
    Bm = rng.standard_normal((Bt, T, G, N), dtype=np.float32)
    Cm = rng.standard_normal((Bt, T, G, N), dtype=np.float32)
    dy = rng.standard_normal((Bt, T, H, P), dtype=np.float32) if with_dy else None
    dfinal = None
    if dfinal_std > 0.0:
        dfinal = (rng.standard_normal((Bt, H, P, N), dtype=np.float32)
                  * np.float32(dfinal_std)).astype(np.float32)

    if dtype == "bf16":
        x, dt, Bm, Cm = (round_to_bf16(a) for a in (x, dt, Bm, Cm))
        if dy is not None:
            dy = round_to_bf16(dy)
    return SSDInputs(shape, dtype, x, dt, dt_bias, A, Bm, Cm, D, init, dy, dfinal)


# Workloads (sizes and seeds).  Each entry: shape, input dtype, init std, seed,
# and whether the backward runs.
WORKLOADS = {
    "tiny_f32": (SSDShape(1, 256, 4, 16, 16, 1, 64), "f32", 0.0, 0, False),
    "layer_bf16": (SSDShape(4, 4096, 24, 64, 128, 1, 256), "bf16", 0.0, 1, False),
    "hybrid_bf16": (SSDShape(2, 8192, 64, 64, 128, 8, 128), "bf16", 0.1, 2, False),
    "long_bf16": (SSDShape(1, 131072, 32, 64, 128, 1, 256), "bf16", 0.0, 3, False),
    "layer_fwdbwd_bf16": (SSDShape(4, 4096, 24, 64, 128, 1, 256), "bf16", 0.0, 4, True),
    # long context with few heads (8 heads of 64: the chunk loop of state
    # passing has few (batch, head) pairs to run in parallel)
    "long_h8_bf16": (SSDShape(1, 131072, 8, 64, 128, 1, 256), "bf16", 0.0, 5, True),
    # the layer with headdim 128 (same d_inner 1536: 12 heads of 128)
    "layer_p128_fwdbwd_bf16": (SSDShape(4, 4096, 12, 128, 128, 1, 256), "bf16", 0.0, 6, True),
}


def make_workload(name: str) -> SSDInputs:
    shape, dtype, init_std, seed, bwd = WORKLOADS[name]
    return make_inputs(shape, seed=seed, dtype=dtype, init_std=init_std, with_dy=bwd)


def to_torch(inp: SSDInputs, device="cuda") -> dict:
    """Copy an input bundle to torch tensors (bf16 or fp32 storage as drawn)."""
    import torch
    tdt = torch.bfloat16 if inp.dtype == "bf16" else torch.float32

    def cv(a, dt=tdt):
        return None if a is None else torch.from_numpy(np.ascontiguousarray(a)).to(
            device=device, dtype=dt)
    f32 = torch.float32
    return dict(x=cv(inp.x), dt=cv(inp.dt), dt_bias=cv(inp.dt_bias, f32), A=cv(inp.A, f32),
                B=cv(inp.B), C=cv(inp.C), D=cv(inp.D, f32), init=cv(inp.init, f32),
                dy=cv(inp.dy), dfinal=cv(inp.dfinal, f32))


# ------------------------------------------------------------ gated norm
@dataclasses.dataclass
class NormShape:
    rows: int          # batch * seqlen
    features: int      # nheads * headdim (d_inner)
    group_size: int    # d_inner / ngroups
    eps: float = 1e-5


@dataclasses.dataclass
class NormInputs:
    shape: NormShape
    dtype: str         # "bf16" or "f32": storage type of y, z, dout
    y: np.ndarray      # (rows, features): the SSD output
    z: np.ndarray      # (rows, features): the gate
    w: np.ndarray      # (features,) fp32 weight
    dout: np.ndarray   # (rows, features): upstream gradient


def make_norm_inputs(shape: NormShape, *, seed: int, dtype: str = "bf16") -> NormInputs:
    """Draw order y, z, w, dout (PCG64): y, z, dout ~ N(0, 1); w = 1 + 0.1 N(0, 1)
    (the weight starts at one in the layer; the spread exercises it).  y, z
    and dout are rounded to bf16 for dtype "bf16"."""
    if dtype not in ("bf16", "f32"):
        raise ValueError(f"dtype must be 'bf16' or 'f32', got {dtype!r}")
    M, D = shape.rows, shape.features
    rng = np.random.Generator(np.random.PCG64(seed))
    y = rng.standard_normal((M, D), dtype=np.float32)
    z = rng.standard_normal((M, D), dtype=np.float32)
    w = (1.0 + 0.1 * rng.standard_normal(D, dtype=np.float32)).astype(np.float32)
    dout = rng.standard_normal((M, D), dtype=np.float32)
    if dtype == "bf16":
        y, z, dout = (round_to_bf16(a) for a in (y, z, dout))
    return NormInputs(shape, dtype, y, z, w, dout)


# rows = batch * seqlen, features = nheads * headdim, group = features / ngroups
NORM_WORKLOADS = {
    "norm_tiny_f32": (NormShape(37, 64, 16), "f32", 0),
    "norm_layer_bf16": (NormShape(4 * 4096, 24 * 64, 24 * 64), "bf16", 1),
    "norm_hybrid_bf16": (NormShape(2 * 8192, 64 * 64, 64 * 64 // 8), "bf16", 2),
}


def make_norm_workload(name: str) -> NormInputs:
    shape, dtype, seed = NORM_WORKLOADS[name]
    return make_norm_inputs(shape, seed=seed, dtype=dtype)
