"""CPU oracle for the Mamba-2 SSD chunked selective scan -- TEST INFRASTRUCTURE.

Only ``tests/``, ``__graft_entry__.smoke()`` and the CPU-baseline leg of
``bench.py`` may import this package.  The product path (the CUDA library and
its binding) never calls it; it shares no code with it.

Contents
  * ``ssd_fwd`` / ``ssd_bwd``: the plain fp64 per-token recurrence and its
    reverse sweep (``ssd_oracle.cpp``), threaded over (batch, head) pairs.
  * ``chunked``: the chunked algorithm (chunk_cumsum, chunk_state,
    state_passing, chunk_scan) written step by step in fp64 numpy; it exposes
    the intermediate tensors the GPU kernels also produce.
  * ``gated_norm``: the gated RMSNorm that follows the SSD output in the
    layer (forward and backward), fp64 numpy.

Parity pins for every function here live in ``tests/test_oracle.py``.
"""
from __future__ import annotations

import ctypes
import os
import subprocess
import threading
from typing import Optional

import numpy as np

_HERE = os.path.dirname(os.path.abspath(__file__))
_SRC = os.path.join(_HERE, "ssd_oracle.cpp")
_LIB_DIR = os.path.join(_HERE, "_build")
_LIB = os.path.join(_LIB_DIR, "libssd_oracle.so")
_lock = threading.Lock()
_lib = None


def build(force: bool = False) -> str:
    """Compile the oracle with g++ (plain -O2, no fast-math, no FMA contraction)."""
    os.makedirs(_LIB_DIR, exist_ok=True)
    if force or not os.path.exists(_LIB) or os.path.getmtime(_LIB) < os.path.getmtime(_SRC):
        tmp = _LIB + f".tmp{os.getpid()}"
        cmd = ["g++", "-O2", "-std=c++17", "-ffp-contract=off", "-fno-fast-math", "-shared",
               "-fPIC", "-pthread", "-o", tmp, _SRC]
        subprocess.run(cmd, check=True)
        os.replace(tmp, _LIB)
    return _LIB


def _load():
    global _lib
    with _lock:
        if _lib is None:
            lib = ctypes.CDLL(build())
            dp = ctypes.POINTER(ctypes.c_double)
            i64p = ctypes.POINTER(ctypes.c_int64)
            lib.ssd_oracle_fwd.argtypes = [i64p] + [dp] * 10 + [ctypes.c_int]
            lib.ssd_oracle_fwd.restype = ctypes.c_int
            lib.ssd_oracle_bwd.argtypes = [i64p] + [dp] * 18 + [ctypes.c_int]
            lib.ssd_oracle_bwd.restype = ctypes.c_int
            lib.ssd_oracle_hardware_threads.restype = ctypes.c_int
            _lib = lib
    return _lib


def hardware_threads() -> int:
    return int(_load().ssd_oracle_hardware_threads())


def _f64(a):
    if a is None:
        return None
    return np.ascontiguousarray(a, dtype=np.float64)


def _ptr(a):
    if a is None:
        return None
    return a.ctypes.data_as(ctypes.POINTER(ctypes.c_double))


def _dims(x, Bm):
    Bt, T, H, P = x.shape
    G, N = Bm.shape[2], Bm.shape[3]
    return np.array([Bt, T, H, P, N, G], dtype=np.int64)


def ssd_fwd(x, dt, dt_bias, A, B, C, D=None, init=None, nthreads: int = 0):
    """Sequential fp64 recurrence.  Returns (y, final_state)."""
    x, dt, dt_bias, A, B, C, D, init = map(_f64, (x, dt, dt_bias, A, B, C, D, init))
    dims = _dims(x, B)
    Bt, T, H, P = x.shape
    N = B.shape[3]
    y = np.empty_like(x)
    final = np.empty((Bt, H, P, N), dtype=np.float64)
    rc = _load().ssd_oracle_fwd(dims.ctypes.data_as(ctypes.POINTER(ctypes.c_int64)), _ptr(x),
                                _ptr(dt), _ptr(dt_bias), _ptr(A), _ptr(B), _ptr(C), _ptr(D),
                                _ptr(init), _ptr(y), _ptr(final), int(nthreads))
    if rc != 0:
        raise ValueError("ssd_oracle_fwd: bad dimensions")
    return y, final


def ssd_bwd(x, dt, dt_bias, A, B, C, D, init, dy, dfinal=None, nthreads: int = 0):
    """Reverse sweep of the recurrence.  Returns a dict of fp64 gradients:
    dx, ddt, dA, dB, dC, dD, ddt_bias, dinit."""
    x, dt, dt_bias, A, B, C, D, init, dy, dfinal = map(
        _f64, (x, dt, dt_bias, A, B, C, D, init, dy, dfinal))
    dims = _dims(x, B)
    Bt, T, H, P = x.shape
    N = B.shape[3]
    out = dict(dx=np.empty_like(x), ddt=np.empty_like(dt), dA=np.empty(H), dB=np.empty_like(B),
               dC=np.empty_like(C), dD=np.empty(H), ddt_bias=np.empty(H),
               dinit=np.empty((Bt, H, P, N)))
    rc = _load().ssd_oracle_bwd(
        dims.ctypes.data_as(ctypes.POINTER(ctypes.c_int64)), _ptr(x), _ptr(dt), _ptr(dt_bias),
        _ptr(A), _ptr(B), _ptr(C), _ptr(D), _ptr(init), _ptr(dy), _ptr(dfinal), _ptr(out["dx"]),
        _ptr(out["ddt"]), _ptr(out["dA"]), _ptr(out["dB"]), _ptr(out["dC"]), _ptr(out["dD"]),
        _ptr(out["ddt_bias"]), _ptr(out["dinit"]), int(nthreads))
    if rc != 0:
        raise ValueError("ssd_oracle_bwd: bad dimensions")
    return out


def from_inputs(inp, fields=("x", "dt", "dt_bias", "A", "B", "C", "D", "init")):
    """fp64 copies of an ``SSDInputs`` bundle's arrays, in oracle argument order."""
    return tuple(_f64(getattr(inp, f)) for f in fields)
