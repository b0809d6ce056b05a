"""Mamba-2 SSD chunked selective scan for GB300 (sm_103a).

Thin binding over the C ABI in ``include/ssd.h``: it checks torch tensors,
allocates outputs and workspace with torch's caching allocator, and passes
raw device pointers plus the current CUDA stream to libssd.  Every step of
the computation runs in the library's CUDA kernels; there is no fallback.
"""
from __future__ import annotations

import ctypes
from typing import Optional

from . import _native
from ._native import build  # noqa: F401

SSD_F32, SSD_BF16 = 0, 1


class SSDError(RuntimeError):
    def __init__(self, fn, status):
        lib = _native.load()
        super().__init__(f"{fn} failed: status {status} ({lib.ssd_strerror(status).decode()})")
        self.status = status


def load_library():
    return _native.load()


def _torch():
    import torch
    return torch


def _dtype_code(t) -> int:
    torch = _torch()
    if t == torch.float32:
        return SSD_F32
    if t == torch.bfloat16:
        return SSD_BF16
    raise TypeError(f"unsupported dtype {t}; use float32 or bfloat16")


def make_shape(batch, seqlen, nheads, headdim, dstate, ngroups, chunk_size, in_dtype=SSD_BF16,
               out_dtype=SSD_F32) -> _native.Shape:
    return _native.Shape(batch, seqlen, nheads, headdim, dstate, ngroups, chunk_size, in_dtype,
                         out_dtype)


def _ptr(t):
    return None if t is None else ctypes.c_void_p(t.data_ptr())


def _check(t, name, shape, dtype, device):
    if t is None:
        return
    if tuple(t.shape) != tuple(shape):
        raise ValueError(f"{name}: expected shape {tuple(shape)}, got {tuple(t.shape)}")
    if t.dtype != dtype:
        raise TypeError(f"{name}: expected {dtype}, got {t.dtype}")
    if t.device != device:
        raise ValueError(f"{name}: expected device {device}, got {t.device}")
    if not t.is_contiguous():
        raise ValueError(f"{name}: must be contiguous")


def _shape_from(x, B, chunk_size, out_dtype):
    Bt, T, H, P = x.shape
    G, N = B.shape[2], B.shape[3]
    return make_shape(Bt, T, H, P, N, G, chunk_size, _dtype_code(x.dtype), _dtype_code(out_dtype))


def _validate(x, dt, dt_bias, A, B, C, D, init_states):
    torch = _torch()
    if x.dim() != 4 or B.dim() != 4:
        raise ValueError("x must be (batch, seqlen, nheads, headdim), B/C (batch, seqlen, ngroups, dstate)")
    dev = x.device
    if dev.type != "cuda":
        raise ValueError("tensors must live on a CUDA device")
    Bt, T, H, P = x.shape
    G, N = B.shape[2], B.shape[3]
    _check(x, "x", (Bt, T, H, P), x.dtype, dev)
    _check(dt, "dt", (Bt, T, H), x.dtype, dev)
    _check(B, "B", (Bt, T, G, N), x.dtype, dev)
    _check(C, "C", (Bt, T, G, N), x.dtype, dev)
    _check(A, "A", (H,), torch.float32, dev)
    _check(dt_bias, "dt_bias", (H,), torch.float32, dev)
    _check(D, "D", (H,), torch.float32, dev)
    _check(init_states, "init_states", (Bt, H, P, N), torch.float32, dev)
    return Bt, T, H, P, N, G


def fwd_workspace_bytes(shape) -> int:
    return int(_native.load().ssd_fwd_workspace_size(ctypes.byref(shape)))


def bwd_workspace_bytes(shape) -> int:
    return int(_native.load().ssd_bwd_workspace_size(ctypes.byref(shape)))


def fwd_workspace_layout(shape) -> dict:
    lay = _native.FwdLayout()
    st = _native.load().ssd_fwd_workspace_layout(ctypes.byref(shape), ctypes.byref(lay))
    if st != 0:
        raise SSDError("ssd_fwd_workspace_layout", st)
    return dict(delta=lay.delta, dA_cumsum=lay.dA_cumsum, states=lay.states, hprev=lay.hprev,
                total=lay.total)


def _workspace(nbytes, device, workspace):
    torch = _torch()
    if workspace is not None:
        if workspace.numel() * workspace.element_size() < nbytes:
            raise ValueError("workspace too small")
        return workspace
    return torch.empty(max(nbytes, 1), dtype=torch.uint8, device=device)


def _raise_on_device_status(fn, device):
    """Synchronise and raise SSDError if the device status word is set."""
    torch = _torch()
    st = int(_native.load().ssd_get_device_status(
        ctypes.c_void_p(torch.cuda.current_stream(device).cuda_stream)))
    if st != 0:
        raise SSDError(fn, st)


def ssd_fwd(x, dt, dt_bias, A, B, C, D=None, chunk_size: int = 256, init_states=None,
            out_dtype=None, return_final_states: bool = True, workspace=None, y=None,
            final_states=None, check: bool = False):
    """y, final_states = SSD(x, dt, A, B, C, D, init_states) by the chunked scan.

    x (b, t, h, p), dt (b, t, h), B/C (b, t, g, n) in float32 or bfloat16 (one
    dtype for all four); dt_bias, A, D (h,) and init_states (b, h, p, n) float32.
    y is float32 by default (``out_dtype=torch.bfloat16`` for bf16).

    The call is asynchronous: y and final_states are only meaningful once the
    library's device status word reads 0 (``device_status()``), since a
    kernel whose bounded wait expired skips its remaining work.  With
    ``check=True`` the call synchronises and raises SSDError when the word is
    set (a timeout, or NaN / Inf in an output when ``set_check_finite(True)``)."""
    torch = _torch()
    lib = _native.load()
    Bt, T, H, P, N, G = _validate(x, dt, dt_bias, A, B, C, D, init_states)
    out_dtype = torch.float32 if out_dtype is None else out_dtype
    shape = _shape_from(x, B, chunk_size, out_dtype)
    if y is None:
        y = torch.empty((Bt, T, H, P), dtype=out_dtype, device=x.device)
    _check(y, "y", (Bt, T, H, P), out_dtype, x.device)
    if return_final_states and final_states is None:
        final_states = torch.empty((Bt, H, P, N), dtype=torch.float32, device=x.device)
    ws_bytes = lib.ssd_fwd_workspace_size(ctypes.byref(shape))
    if ws_bytes == 0:
        raise ValueError("invalid SSD shape")
    ws = _workspace(ws_bytes, x.device, workspace)
    stream = torch.cuda.current_stream(x.device).cuda_stream
    st = lib.ssd_fwd(ctypes.byref(shape), _ptr(x), _ptr(dt), _ptr(dt_bias), _ptr(A), _ptr(B),
                     _ptr(C), _ptr(D), _ptr(init_states), _ptr(y),
                     _ptr(final_states) if return_final_states else None, _ptr(ws),
                     ctypes.c_size_t(ws.numel()), ctypes.c_void_p(stream))
    if st != 0:
        raise SSDError("ssd_fwd", st)
    if check:
        _raise_on_device_status("ssd_fwd", x.device)
    return y, (final_states if return_final_states else None)


def ssd_bwd(x, dt, dt_bias, A, B, C, D, chunk_size: int, init_states, dy, dfinal_states=None,
            workspace=None, out=None, check: bool = False):
    """Gradients of <dy, y> + <dfinal, final> w.r.t. every input of ssd_fwd.

    Returns a dict with dx, ddt, dA, dB, dC (float32, shapes of the inputs)
    and dD, ddt_bias, dinit_states (when D / init_states are given; dD and
    ddt_bias are always returned).  As for ssd_fwd, the gradients are only
    meaningful once the device status word reads 0; ``check=True``
    synchronises and raises SSDError otherwise."""
    torch = _torch()
    lib = _native.load()
    Bt, T, H, P, N, G = _validate(x, dt, dt_bias, A, B, C, D, init_states)
    _check(dy, "dy", (Bt, T, H, P), x.dtype, x.device)
    _check(dfinal_states, "dfinal_states", (Bt, H, P, N), torch.float32, x.device)
    shape = _shape_from(x, B, chunk_size, torch.float32)
    f32 = dict(dtype=torch.float32, device=x.device)
    if out is None:
        out = dict(dx=torch.empty((Bt, T, H, P), **f32), ddt=torch.empty((Bt, T, H), **f32),
                   dA=torch.empty((H,), **f32), dB=torch.empty((Bt, T, G, N), **f32),
                   dC=torch.empty((Bt, T, G, N), **f32), dD=torch.empty((H,), **f32),
                   ddt_bias=torch.empty((H,), **f32))
        if init_states is not None:
            out["dinit_states"] = torch.empty((Bt, H, P, N), **f32)
    ws_bytes = lib.ssd_bwd_workspace_size(ctypes.byref(shape))
    if ws_bytes == 0:
        raise ValueError("invalid SSD shape")
    ws = _workspace(ws_bytes, x.device, workspace)
    stream = torch.cuda.current_stream(x.device).cuda_stream
    st = lib.ssd_bwd(ctypes.byref(shape), _ptr(x), _ptr(dt), _ptr(dt_bias), _ptr(A), _ptr(B),
                     _ptr(C), _ptr(D), _ptr(init_states), _ptr(dy), _ptr(dfinal_states),
                     _ptr(out["dx"]), _ptr(out["ddt"]), _ptr(out["dA"]), _ptr(out["dB"]),
                     _ptr(out["dC"]), _ptr(out.get("dD")), _ptr(out.get("ddt_bias")),
                     _ptr(out.get("dinit_states")), _ptr(ws), ctypes.c_size_t(ws.numel()),
                     ctypes.c_void_p(stream))
    if st != 0:
        raise SSDError("ssd_bwd", st)
    if check:
        _raise_on_device_status("ssd_bwd", x.device)
    return out


def ssd_final_state(x, dt, dt_bias, A, B, chunk_size: int = 256, init_states=None,
                    workspace=None, final_states=None):
    """The state after the whole sequence from ``init_states`` (None: zero),
    without the outputs: chunk_cumsum, chunk_state, state_passing
    (``ssd_fwd_final_state``)."""
    torch = _torch()
    lib = _native.load()
    Bt, T, H, P, N, G = _validate(x, dt, dt_bias, A, B, B, None, init_states)
    shape = _shape_from(x, B, chunk_size, torch.float32)
    if final_states is None:
        final_states = torch.empty((Bt, H, P, N), dtype=torch.float32, device=x.device)
    _check(final_states, "final_states", (Bt, H, P, N), torch.float32, x.device)
    ws = _workspace(lib.ssd_fwd_workspace_size(ctypes.byref(shape)), x.device, workspace)
    stream = torch.cuda.current_stream(x.device).cuda_stream
    st = lib.ssd_fwd_final_state(ctypes.byref(shape), _ptr(x), _ptr(dt), _ptr(dt_bias), _ptr(A),
                                 _ptr(B), _ptr(init_states), _ptr(final_states), _ptr(ws),
                                 ctypes.c_size_t(ws.numel()), ctypes.c_void_p(stream))
    if st != 0:
        raise SSDError("ssd_fwd_final_state", st)
    return final_states


def ssd_dinit(x, dt, dt_bias, A, C, dy, chunk_size: int = 256, dfinal_states=None,
              workspace=None, dinit_states=None):
    """Gradient of <dy, y> + <dfinal, final> w.r.t. the initial state alone
    (``ssd_bwd_dinit``); x is read for its shape only."""
    torch = _torch()
    lib = _native.load()
    Bt, T, H, P, N, G = _validate(x, dt, dt_bias, A, C, C, None, None)
    _check(dy, "dy", (Bt, T, H, P), x.dtype, x.device)
    _check(dfinal_states, "dfinal_states", (Bt, H, P, N), torch.float32, x.device)
    shape = _shape_from(x, C, chunk_size, torch.float32)
    if dinit_states is None:
        dinit_states = torch.empty((Bt, H, P, N), dtype=torch.float32, device=x.device)
    _check(dinit_states, "dinit_states", (Bt, H, P, N), torch.float32, x.device)
    ws = _workspace(lib.ssd_fwd_workspace_size(ctypes.byref(shape)), x.device, workspace)
    stream = torch.cuda.current_stream(x.device).cuda_stream
    st = lib.ssd_bwd_dinit(ctypes.byref(shape), _ptr(dt), _ptr(dt_bias), _ptr(A), _ptr(C),
                           _ptr(dy), _ptr(dfinal_states), _ptr(dinit_states), _ptr(ws),
                           ctypes.c_size_t(ws.numel()), ctypes.c_void_p(stream))
    if st != 0:
        raise SSDError("ssd_bwd_dinit", st)
    return dinit_states


def _norm_shape(y, group_size, eps, out_dtype):
    D = y.shape[-1]
    rows = y.numel() // D if D else 0
    return _native.NormShape(rows, D, group_size, float(eps), _dtype_code(y.dtype),
                             _dtype_code(out_dtype))


def _norm_check(name, t, like, dtype=None):
    if t is None:
        raise ValueError(f"{name} is required")
    _check(t, name, tuple(like.shape), like.dtype if dtype is None else dtype, like.device)


def gated_norm_fwd(y, z, w, group_size: int, eps: float = 1e-5, out_dtype=None,
                   return_rstd: bool = True, out=None, rstd=None):
    """out = rmsnorm over groups of ``group_size`` of (y * silu(z)), times w
    (``ssd_gated_norm_fwd``).  y, z (..., features) float32 or bfloat16 (one
    dtype), w (features,) float32.  Returns (out, rstd (rows, groups) or None)."""
    torch = _torch()
    lib = _native.load()
    if y.dim() < 1 or y.device.type != "cuda":
        raise ValueError("y must be a CUDA tensor (..., features)")
    _norm_check("z", z, y)
    D = y.shape[-1]
    _check(w, "w", (D,), torch.float32, y.device)
    out_dtype = y.dtype if out_dtype is None else out_dtype
    shape = _norm_shape(y, group_size, eps, out_dtype)
    if out is None:
        out = torch.empty(y.shape, dtype=out_dtype, device=y.device)
    _check(out, "out", tuple(y.shape), out_dtype, y.device)
    if return_rstd and rstd is None:
        rstd = torch.empty((shape.rows, max(D // max(group_size, 1), 1)), dtype=torch.float32,
                           device=y.device)
    stream = torch.cuda.current_stream(y.device).cuda_stream
    st = lib.ssd_gated_norm_fwd(ctypes.byref(shape), _ptr(y), _ptr(z), _ptr(w), _ptr(out),
                                _ptr(rstd) if return_rstd else None, ctypes.c_void_p(stream))
    if st != 0:
        raise SSDError("ssd_gated_norm_fwd", st)
    return out, (rstd if return_rstd else None)


def gated_norm_workspace_bytes(y, group_size: int, eps: float = 1e-5, out_dtype=None) -> int:
    shape = _norm_shape(y, group_size, eps, y.dtype if out_dtype is None else out_dtype)
    return int(_native.load().ssd_gated_norm_workspace_size(ctypes.byref(shape)))


def gated_norm_bwd(y, z, w, dout, group_size: int, eps: float = 1e-5, rstd=None,
                   out_dtype=None, workspace=None, out=None):
    """Gradients of <dout, out> (``ssd_gated_norm_bwd``): dict dy, dz (shape of
    y, ``out_dtype``: y's dtype by default) and dw (features,) float32.  rstd
    as ``gated_norm_fwd`` returned it, or None to recompute it."""
    torch = _torch()
    lib = _native.load()
    _norm_check("z", z, y)
    _norm_check("dout", dout, y)
    D = y.shape[-1]
    _check(w, "w", (D,), torch.float32, y.device)
    out_dtype = y.dtype if out_dtype is None else out_dtype
    shape = _norm_shape(y, group_size, eps, out_dtype)
    if out is None:
        out = dict(dy=torch.empty(y.shape, dtype=out_dtype, device=y.device),
                   dz=torch.empty(y.shape, dtype=out_dtype, device=y.device),
                   dw=torch.empty((D,), dtype=torch.float32, device=y.device))
    nbytes = lib.ssd_gated_norm_workspace_size(ctypes.byref(shape))
    if nbytes == 0:
        raise SSDError("ssd_gated_norm_workspace_size", 2)
    ws = _workspace(nbytes, y.device, workspace)
    stream = torch.cuda.current_stream(y.device).cuda_stream
    st = lib.ssd_gated_norm_bwd(ctypes.byref(shape), _ptr(y), _ptr(z), _ptr(w), _ptr(rstd),
                                _ptr(dout), _ptr(out["dy"]), _ptr(out["dz"]), _ptr(out["dw"]),
                                _ptr(ws), ctypes.c_size_t(ws.numel()), ctypes.c_void_p(stream))
    if st != 0:
        raise SSDError("ssd_gated_norm_bwd", st)
    return out


def segment_decay(dt, dt_bias, A):
    """decay (b, h) = exp(A[h] * sum_t softplus(dt[b, t, h] + dt_bias[h])) over
    the whole of dt's sequence: the factor by which a state entering this
    segment is carried to its end (context parallelism, ``ssd_segment_decay``)."""
    torch = _torch()
    lib = _native.load()
    if dt.dim() != 3:
        raise ValueError("dt: expected (batch, seqlen, nheads)")
    Bt, T, H = dt.shape
    _check(A, "A", (H,), torch.float32, dt.device)
    _check(dt_bias, "dt_bias", (H,), torch.float32, dt.device)
    dt = dt.contiguous()
    out = torch.empty((Bt, H), dtype=torch.float32, device=dt.device)
    shape = make_shape(Bt, T, H, 1, 1, 1, 1, _dtype_code(dt.dtype), SSD_F32)
    ws = _workspace(lib.ssd_segment_decay_workspace_size(ctypes.byref(shape)), dt.device, None)
    stream = torch.cuda.current_stream(dt.device).cuda_stream
    st = lib.ssd_segment_decay(ctypes.byref(shape), _ptr(dt), _ptr(dt_bias), _ptr(A), _ptr(out),
                               _ptr(ws), ctypes.c_size_t(ws.numel()), ctypes.c_void_p(stream))
    if st != 0:
        raise SSDError("ssd_segment_decay", st)
    return out


def state_scan(decays, states, rank: int, direction: int):
    """Exclusive scan over ranks of S -> D_k * S + S_k (``ssd_state_scan``):
    decays (R, b, h), states (R, b, h, p, n) float32 -> (b, h, p, n) for
    ``rank``; direction 0 over the ranks before it (incoming state),
    1 over the ranks after it (gradient of the outgoing state)."""
    torch = _torch()
    lib = _native.load()
    R = decays.shape[0]
    if states.dim() != 5 or states.shape[0] != R or tuple(decays.shape) != tuple(states.shape[:3]):
        raise ValueError("state_scan: expected decays (R, b, h) and states (R, b, h, p, n)")
    if decays.dtype != torch.float32 or states.dtype != torch.float32:
        raise TypeError("state_scan: float32 tensors expected")
    decays, states = decays.contiguous(), states.contiguous()
    bh = states.shape[1] * states.shape[2]
    pn = states.shape[3] * states.shape[4]
    out = torch.empty(states.shape[1:], dtype=torch.float32, device=states.device)
    stream = torch.cuda.current_stream(states.device).cuda_stream
    st = lib.ssd_state_scan(int(R), int(rank), int(direction), int(bh), int(pn), _ptr(decays),
                            _ptr(states), _ptr(out), ctypes.c_void_p(stream))
    if st != 0:
        raise SSDError("ssd_state_scan", st)
    return out


def device_status(stream=None) -> int:
    """Synchronise and read/clear the library's device status word."""
    torch = _torch()
    s = torch.cuda.current_stream().cuda_stream if stream is None else stream
    return int(_native.load().ssd_get_device_status(ctypes.c_void_p(s)))


def set_check_finite(on: bool = True) -> bool:
    """Turn the library's opt-in NaN / Inf scan of every output on or off
    (process-wide); returns the previous setting.  A non-finite output shows
    as status 6 (SSD_ERR_NONFINITE) in ``device_status()``."""
    return bool(_native.load().ssd_set_check_finite(1 if on else 0))


def last_path() -> int:
    """0 = generic SIMT kernels, 1 = tcgen05 tensor-core kernels (last call, this thread)."""
    return int(_native.load().ssd_last_path())


def profile_enable(on: bool = True) -> None:
    """Start (clearing previous totals) or stop per-kernel CUDA-event timing."""
    _native.load().ssd_profile_enable(1 if on else 0)


def profile_read(max_kernels: int = 64) -> dict:
    """{kernel name: (total device ms, launches)} since profile_enable(True)."""
    lib = _native.load()
    names = ctypes.create_string_buffer(64 * max_kernels)
    ms = (ctypes.c_double * max_kernels)()
    cnt = (ctypes.c_int64 * max_kernels)()
    n = lib.ssd_profile_read(max_kernels, names, ms, cnt)
    if n < 0:
        raise SSDError("ssd_profile_read", -n)
    out = {}
    for i in range(n):
        nm = names.raw[64 * i:64 * (i + 1)].split(b"\0", 1)[0].decode()
        out[nm] = (ms[i], cnt[i])
    return out


def launch_count() -> int:
    """Kernels launched by libssd in this process so far."""
    return int(_native.load().ssd_launch_count())
