"""Build and load libssd (the CUDA library behind include/ssd.h).

The library is compiled in-tree with nvcc for sm_103a only; each .cu file is a
separate translation unit compiled in parallel, then linked into one shared
object.  Loading fails loudly when the library is missing: there is no other
implementation to fall back to.
"""
from __future__ import annotations

import concurrent.futures as cf
import ctypes
import glob
import os
import shutil
import subprocess
import threading

PKG = os.path.dirname(os.path.abspath(__file__))
ROOT = os.path.dirname(PKG)
CSRC = os.path.join(PKG, "csrc")
INCLUDE = os.path.join(ROOT, "include")
BUILD = os.path.join(PKG, "_build")
LIB = os.path.join(BUILD, "libssd.so")

ARCH = ["-gencode", "arch=compute_103a,code=sm_103a"]
NVCC_FLAGS = ["-O3", "-lineinfo", "-std=c++17", "-Xcompiler", "-fPIC", "-Xcompiler", "-O2",
              "--expt-relaxed-constexpr", "-I", INCLUDE]


def _nvcc() -> str:
    for cand in (shutil.which("nvcc"), "/usr/local/cuda/bin/nvcc"):
        if cand and os.path.exists(cand):
            return cand
    raise RuntimeError("nvcc not found: the CUDA toolkit is required to build libssd")


def _sources():
    return sorted(glob.glob(os.path.join(CSRC, "*.cu")))


def _deps():
    return _sources() + sorted(glob.glob(os.path.join(CSRC, "*.h"))) + \
        sorted(glob.glob(os.path.join(CSRC, "*.cuh"))) + [os.path.join(INCLUDE, "ssd.h")]


def build(force: bool = False, verbose: bool = False) -> str:
    """Compile every CUDA source for sm_103a and link libssd.so in-tree."""
    os.makedirs(BUILD, exist_ok=True)
    if not force and os.path.exists(LIB):
        newest = max(os.path.getmtime(p) for p in _deps())
        if os.path.getmtime(LIB) >= newest:
            return LIB
    nvcc = _nvcc()
    objs = []

    def compile_one(src):
        obj = os.path.join(BUILD, os.path.basename(src)[:-3] + ".o")
        cmd = [nvcc] + ARCH + NVCC_FLAGS + ["-c", src, "-o", obj]
        if verbose:
            cmd.insert(1, "-Xptxas=-v")
        r = subprocess.run(cmd, capture_output=True, text=True)
        if r.returncode != 0:
            raise RuntimeError(f"nvcc failed on {src}:\n{r.stdout}\n{r.stderr}")
        return obj, r.stderr

    with cf.ThreadPoolExecutor(max_workers=min(8, os.cpu_count() or 1)) as ex:
        for obj, log in ex.map(compile_one, _sources()):
            objs.append(obj)
            if verbose and log:
                print(log)
    tmp = LIB + f".tmp{os.getpid()}"
    cmd = [nvcc] + ARCH + ["-shared", "-cudart", "static", "-o", tmp] + objs
    r = subprocess.run(cmd, capture_output=True, text=True)
    if r.returncode != 0:
        raise RuntimeError(f"nvcc link failed:\n{r.stdout}\n{r.stderr}")
    os.replace(tmp, LIB)
    return LIB


class Shape(ctypes.Structure):
    _fields_ = [("batch", ctypes.c_int64), ("seqlen", ctypes.c_int64),
                ("nheads", ctypes.c_int64), ("headdim", ctypes.c_int64),
                ("dstate", ctypes.c_int64), ("ngroups", ctypes.c_int64),
                ("chunk_size", ctypes.c_int64), ("in_dtype", ctypes.c_int32),
                ("out_dtype", ctypes.c_int32)]


class FwdLayout(ctypes.Structure):
    _fields_ = [("delta", ctypes.c_size_t), ("dA_cumsum", ctypes.c_size_t),
                ("states", ctypes.c_size_t), ("hprev", ctypes.c_size_t),
                ("total", ctypes.c_size_t)]


# Every symbol include/ssd.h declares, with its ctypes signature.
class NormShape(ctypes.Structure):
    _fields_ = [("rows", ctypes.c_int64), ("features", ctypes.c_int64),
                ("group_size", ctypes.c_int64), ("eps", ctypes.c_float),
                ("in_dtype", ctypes.c_int32), ("out_dtype", ctypes.c_int32)]


class ScanConfig(ctypes.Structure):
    _fields_ = [("scan_head_blocks", ctypes.c_int32), ("bc_head_blocks", ctypes.c_int32),
                ("scan_head_blocks_light", ctypes.c_int32),
                ("bc_head_blocks_light", ctypes.c_int32)]


class NormConfig(ctypes.Structure):
    _fields_ = [("rows_per_item", ctypes.c_int32), ("ring_kb", ctypes.c_int32),
                ("ctas_per_sm", ctypes.c_int32)]


_VP = ctypes.c_void_p
_SP = ctypes.POINTER(Shape)
_NP = ctypes.POINTER(NormShape)
SIGNATURES = {
    "ssd_fwd_workspace_size": ([_SP], ctypes.c_size_t),
    "ssd_bwd_workspace_size": ([_SP], ctypes.c_size_t),
    "ssd_fwd_workspace_layout": ([_SP, ctypes.POINTER(FwdLayout)], ctypes.c_int),
    "ssd_fwd": ([_SP] + [_VP] * 10 + [_VP, ctypes.c_size_t, _VP], ctypes.c_int),
    "ssd_bwd": ([_SP] + [_VP] * 18 + [_VP, ctypes.c_size_t, _VP], ctypes.c_int),
    "ssd_get_device_status": ([_VP], ctypes.c_int),
    "ssd_last_path": ([], ctypes.c_int),
    "ssd_set_check_finite": ([ctypes.c_int], ctypes.c_int),
    "ssd_scan_set_config": ([_SP, ctypes.POINTER(ScanConfig)], ctypes.c_int),
    "ssd_scan_get_config": ([_SP, ctypes.POINTER(ScanConfig)], ctypes.c_int),
    "ssd_strerror": ([ctypes.c_int], ctypes.c_char_p),
    "ssd_profile_enable": ([ctypes.c_int], ctypes.c_int),
    "ssd_profile_read": ([ctypes.c_int, ctypes.c_char_p, ctypes.POINTER(ctypes.c_double),
                          ctypes.POINTER(ctypes.c_int64)], ctypes.c_int),
    "ssd_launch_count": ([], ctypes.c_int64),
    "ssd_selftest_mma": ([ctypes.c_int] * 5 + [_VP] * 4, ctypes.c_int),
    "ssd_selftest_timeout": ([_VP], ctypes.c_int),
    "ssd_selftest_timeout_suspend": ([_VP], ctypes.c_int),
    "ssd_fwd_noalloc": ([_SP] + [_VP] * 10 + [_VP], ctypes.c_int),
    "ssd_noalloc_scratch_bytes": ([], ctypes.c_size_t),
    "ssd_segment_decay_workspace_size": ([_SP], ctypes.c_size_t),
    "ssd_segment_decay": ([_SP, _VP, _VP, _VP, _VP, _VP, ctypes.c_size_t, _VP], ctypes.c_int),
    "ssd_gated_norm_workspace_size": ([_NP], ctypes.c_size_t),
    "ssd_gated_norm_set_config": ([_NP, ctypes.POINTER(NormConfig)], ctypes.c_int),
    "ssd_gated_norm_get_config": ([_NP, ctypes.POINTER(NormConfig)], ctypes.c_int),
    "ssd_gated_norm_fwd": ([_NP] + [_VP] * 5 + [_VP], ctypes.c_int),
    "ssd_gated_norm_bwd": ([_NP] + [_VP] * 9 + [ctypes.c_size_t, _VP], ctypes.c_int),
    "ssd_fwd_final_state": ([_SP] + [_VP] * 7 + [_VP, ctypes.c_size_t, _VP], ctypes.c_int),
    "ssd_bwd_dinit": ([_SP] + [_VP] * 7 + [_VP, ctypes.c_size_t, _VP], ctypes.c_int),
    "ssd_state_scan": ([ctypes.c_int, ctypes.c_int, ctypes.c_int, ctypes.c_int64, ctypes.c_int64,
                        _VP, _VP, _VP, _VP], ctypes.c_int),
}

_lock = threading.Lock()
_lib = None


def load(path: str = LIB):
    """Load libssd.so (built by ``build()``); raises if it is missing."""
    global _lib
    with _lock:
        if _lib is None:
            if not os.path.exists(path):
                raise RuntimeError(
                    f"libssd is not built ({path} missing); run __graft_entry__.build() "
                    "or state_space_model_sm_gb300.build()")
            lib = ctypes.CDLL(path)
            for name, (args, res) in SIGNATURES.items():
                fn = getattr(lib, name)
                fn.argtypes = args
                fn.restype = res
            from . import tuning  # the offline launch table, applied once at load
            tuning.apply_default(lib)
            _lib = lib
    return _lib
