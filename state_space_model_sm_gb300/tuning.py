"""Offline launch-configuration tables for the gated-norm and SSD chunk kernels.

The pages' config generator ("Cutting autotuning overhead with an automated
config generator", Fig. 4) separates the search from the run: the best
launch parameters for each environment are found ahead of time, written to a
file, and loaded when training starts.  The same split here:

  * ``sweep_gated_norm`` times every candidate launch of the forward +
    backward for one shape on the current GPU (CUDA events, L2 flushed
    between steps) and returns the best;
  * ``python -m state_space_model_sm_gb300.tuning --sweep F:G[,F:G...]
    --out table.json`` writes the table for several (features, group_size)
    shapes;
  * the library applies a table when it is loaded: the one named by the
    environment variable ``SSD_TUNING_TABLE`` (``none`` disables), else the
    packaged ``tuning_tables/gated_norm_gb300.json``.

The parameters (``ssd_norm_config`` in ``include/ssd.h``): rows per CTA work
item, the shared-memory ring size aimed at, and the persistent CTAs per SM.

The SSD chunk kernels have a table of their own (``ssd_scan_config``): how
many blocks of heads the chunk_scan and the dC / dB CTAs split each group
into, for the chunk's heavy row tile (more column panels) and its light one.
``sweep_scan`` times the forward + backward step of a workload for each
candidate pair, ``--sweep-scan W[,W...] --out`` writes the table, and the
packaged ``tuning_tables/ssd_scan_gb300.json`` is applied at load like the
norm's (``SSD_SCAN_TABLE`` names another table or ``none``).
"""
from __future__ import annotations

import argparse
import ctypes
import json
import os
from typing import Iterable, Optional

from . import _native

TABLE_KIND = "gated_norm_launch_table"
DEFAULT_TABLE = os.path.join(os.path.dirname(os.path.abspath(__file__)), "tuning_tables",
                             "gated_norm_gb300.json")
SCAN_TABLE_KIND = "ssd_scan_launch_table"
DEFAULT_SCAN_TABLE = os.path.join(os.path.dirname(os.path.abspath(__file__)), "tuning_tables",
                                  "ssd_scan_gb300.json")
_SCAN_KEYS = ("batch", "seqlen", "nheads", "headdim", "dstate", "ngroups", "chunk_size")
_SCAN_FIELDS = ("scan_head_blocks", "bc_head_blocks", "scan_head_blocks_light",
                "bc_head_blocks_light")
_DTYPES = {"f32": 0, "bf16": 1}
_FIELDS = ("rows_per_item", "ring_kb", "ctas_per_sm")


def _shape(features, group_size, in_dtype, out_dtype, rows=1, eps=1e-5):
    return _native.NormShape(int(rows), int(features), int(group_size), float(eps),
                             _DTYPES[in_dtype], _DTYPES[out_dtype])


def validate_table(table: dict) -> None:
    """Raises ValueError unless ``table`` is a well-formed launch table
    (field ranges as ``ssd_gated_norm_set_config`` accepts them)."""
    if table.get("kind") != TABLE_KIND:
        raise ValueError(f"not a {TABLE_KIND}")
    entries = table.get("entries")
    if not isinstance(entries, list):
        raise ValueError("entries must be a list")
    seen = set()
    for e in entries:
        for k in ("features", "group_size", "in_dtype", "out_dtype") + _FIELDS:
            if k not in e:
                raise ValueError(f"entry misses {k!r}: {e}")
        if e["in_dtype"] not in _DTYPES or e["out_dtype"] not in _DTYPES:
            raise ValueError(f"bad dtype in {e}")
        F, G = int(e["features"]), int(e["group_size"])
        if F % 8 or G % 8 or F % G or F < 8:
            raise ValueError(f"bad shape in {e}")
        rpc, ring, ctas = (int(e[k]) for k in _FIELDS)
        tpr = F // 8
        if rpc < 0 or (rpc > 0 and (rpc * tpr > 512 or (rpc * tpr) % 32)):
            raise ValueError(f"bad rows_per_item in {e}")
        if ring < 0 or (ring > 0 and not 8 <= ring <= 200):
            raise ValueError(f"bad ring_kb in {e}")
        if not 0 <= ctas <= 8:
            raise ValueError(f"bad ctas_per_sm in {e}")
        key = (F, G, e["in_dtype"], e["out_dtype"])
        if key in seen:
            raise ValueError(f"duplicate entry {key}")
        seen.add(key)
    if len(entries) > 64:
        raise ValueError("at most 64 entries")


def set_norm_config(features, group_size, in_dtype="bf16", out_dtype=None, rows_per_item=0,
                    ring_kb=0, ctas_per_sm=0, lib=None) -> None:
    """Sets the table entry of one shape (zero fields keep the built-in choice)."""
    lib = lib or _native.load()
    cfg = _native.NormConfig(int(rows_per_item), int(ring_kb), int(ctas_per_sm))
    sh = _shape(features, group_size, in_dtype, out_dtype or in_dtype)
    st = lib.ssd_gated_norm_set_config(ctypes.byref(sh), ctypes.byref(cfg))
    if st != 0:
        raise ValueError(f"ssd_gated_norm_set_config: status {st}")


def clear_norm_config(features, group_size, in_dtype="bf16", out_dtype=None, lib=None) -> None:
    lib = lib or _native.load()
    sh = _shape(features, group_size, in_dtype, out_dtype or in_dtype)
    st = lib.ssd_gated_norm_set_config(ctypes.byref(sh), None)
    if st != 0:
        raise ValueError(f"ssd_gated_norm_set_config: status {st}")


def get_norm_config(features, group_size, in_dtype="bf16", out_dtype=None, lib=None):
    """(config dict the next call will use, True if it comes from the table)."""
    lib = lib or _native.load()
    cfg = _native.NormConfig()
    sh = _shape(features, group_size, in_dtype, out_dtype or in_dtype)
    st = lib.ssd_gated_norm_get_config(ctypes.byref(sh), ctypes.byref(cfg))
    if st < 0:
        raise ValueError(f"ssd_gated_norm_get_config: status {-st}")
    return {k: int(getattr(cfg, k)) for k in _FIELDS}, st == 1


def apply_table(table: dict, lib=None) -> int:
    """Sets every entry of a validated table; returns the number applied."""
    validate_table(table)
    for e in table["entries"]:
        set_norm_config(e["features"], e["group_size"], e["in_dtype"], e["out_dtype"],
                        e["rows_per_item"], e["ring_kb"], e["ctas_per_sm"], lib=lib)
    return len(table["entries"])


def apply_default(lib) -> Optional[str]:
    """Called once when the library is loaded: applies the norm table named by
    SSD_TUNING_TABLE (``none``: no table), else the packaged one if present,
    and likewise the SSD chunk-kernel table (SSD_SCAN_TABLE).  Returns the
    norm table's path, or None."""
    scan_path = os.environ.get("SSD_SCAN_TABLE", DEFAULT_SCAN_TABLE)
    if scan_path.lower() != "none" and os.path.exists(scan_path):
        with open(scan_path) as f:
            apply_scan_table(json.load(f), lib=lib)
    path = os.environ.get("SSD_TUNING_TABLE", DEFAULT_TABLE)
    if path.lower() == "none" or not os.path.exists(path):
        return None
    with open(path) as f:
        apply_table(json.load(f), lib=lib)
    return path


# ------------------------------------------------------ SSD chunk kernels
def _scan_shape(e: dict):
    return _native.Shape(*(int(e[k]) for k in _SCAN_KEYS), 1, 0)


def _kernel_heads_per_group(shape: dict) -> int:
    """Heads per group as the chunk kernels count them: a head of headdim 128
    runs as two 64-wide heads."""
    hpg = int(shape["nheads"]) // int(shape["ngroups"])
    return 2 * hpg if int(shape["headdim"]) == 128 else hpg


def validate_scan_table(table: dict) -> None:
    """Raises ValueError unless ``table`` is a well-formed SSD launch table
    (field ranges as ``ssd_scan_set_config`` accepts them)."""
    if table.get("kind") != SCAN_TABLE_KIND:
        raise ValueError(f"not a {SCAN_TABLE_KIND}")
    entries = table.get("entries")
    if not isinstance(entries, list) or len(entries) > 64:
        raise ValueError("entries must be a list of at most 64")
    seen = set()
    for e in entries:
        for k in _SCAN_KEYS + _SCAN_FIELDS[:2]:
            if k not in e:
                raise ValueError(f"entry misses {k!r}: {e}")
        H, G = int(e["nheads"]), int(e["ngroups"])
        if min(int(e[k]) for k in _SCAN_KEYS) < 1 or H % G:
            raise ValueError(f"bad shape in {e}")
        hpg = _kernel_heads_per_group(e)
        for k in _SCAN_FIELDS:
            v = int(e.get(k, 0))
            if v < 0 or v > 32 or (v > 0 and hpg % v):
                raise ValueError(f"bad {k} in {e}")
        key = tuple(int(e[k]) for k in _SCAN_KEYS)
        if key in seen:
            raise ValueError(f"duplicate entry {key}")
        seen.add(key)


def set_scan_config(shape: dict, scan_head_blocks=0, bc_head_blocks=0, scan_head_blocks_light=0,
                    bc_head_blocks_light=0, lib=None) -> None:
    """Sets the table entry of one SSD shape (``shape``: the _SCAN_KEYS);
    zero fields keep the built-in rule's count."""
    lib = lib or _native.load()
    cfg = _native.ScanConfig(int(scan_head_blocks), int(bc_head_blocks),
                             int(scan_head_blocks_light), int(bc_head_blocks_light))
    st = lib.ssd_scan_set_config(ctypes.byref(_scan_shape(shape)), ctypes.byref(cfg))
    if st != 0:
        raise ValueError(f"ssd_scan_set_config: status {st}")


def clear_scan_config(shape: dict, lib=None) -> None:
    lib = lib or _native.load()
    st = lib.ssd_scan_set_config(ctypes.byref(_scan_shape(shape)), None)
    if st != 0:
        raise ValueError(f"ssd_scan_set_config: status {st}")


def get_scan_config(shape: dict, lib=None):
    """(head blocks the next call will use, True if they come from the table)."""
    lib = lib or _native.load()
    cfg = _native.ScanConfig()
    st = lib.ssd_scan_get_config(ctypes.byref(_scan_shape(shape)), ctypes.byref(cfg))
    if st < 0:
        raise ValueError(f"ssd_scan_get_config: status {-st}")
    return {k: int(getattr(cfg, k)) for k in _SCAN_FIELDS}, st == 1


def apply_scan_table(table: dict, lib=None) -> int:
    validate_scan_table(table)
    for e in table["entries"]:
        set_scan_config({k: e[k] for k in _SCAN_KEYS}, lib=lib,
                        **{k: int(e.get(k, 0)) for k in _SCAN_FIELDS})
    return len(table["entries"])


def sweep_scan(workload: str, steps: int = 10, warmup: int = 3, max_blocks: int = 12) -> dict:
    """Times the forward + backward step of a workload (CUDA events, a 512 MB
    L2 flush before each step) for every head-block count of chunk_scan, then
    of dC / dB with chunk_scan's best, on the current GPU; returns the best
    entry with the built-in rule's time."""
    import torch

    from . import ssd_bwd, ssd_fwd
    from .inputs import WORKLOADS, make_inputs, to_torch
    lib = _native.load()
    shape, dtype, init_std, seed, _ = WORKLOADS[workload]
    inp = make_inputs(shape, seed=seed, dtype=dtype, init_std=init_std, with_dy=True)
    s = inp.shape
    key = dict(batch=s.batch, seqlen=s.seqlen, nheads=s.nheads, headdim=s.headdim,
               dstate=s.dstate, ngroups=s.ngroups, chunk_size=s.chunk_size)
    t = to_torch(inp)
    dev = t["x"].device
    flush = torch.empty(512 * 1024 * 1024 // 4, device=dev)
    stream = torch.cuda.current_stream(dev)

    def step():
        ssd_fwd(t["x"], t["dt"], t["dt_bias"], t["A"], t["B"], t["C"], t["D"],
                chunk_size=s.chunk_size, init_states=t["init"])
        ssd_bwd(t["x"], t["dt"], t["dt_bias"], t["A"], t["B"], t["C"], t["D"], s.chunk_size,
                t["init"], t["dy"], t["dfinal"])

    def time_us():
        for _ in range(warmup):
            step()
        ev = [(torch.cuda.Event(enable_timing=True), torch.cuda.Event(enable_timing=True))
              for _ in range(steps)]
        for a, b in ev:
            flush.fill_(1.0)
            a.record(stream)
            step()
            b.record(stream)
        torch.cuda.synchronize()
        return 1e3 * sum(a.elapsed_time(b) for a, b in ev) / steps

    hpg = _kernel_heads_per_group(key)
    blocks = [nb for nb in range(1, min(hpg, max_blocks) + 1) if hpg % nb == 0]
    # (heavy, light) pairs; with chunk 128 there is one row tile
    pairs = [(h, l) for h in blocks for l in blocks] if s.chunk_size > 128 else \
        [(h, h) for h in blocks]
    saved, had = get_scan_config(key, lib=lib)
    clear_scan_config(key, lib=lib)
    default_cfg, _ = get_scan_config(key, lib=lib)
    default_us = time_us()
    try:
        scan_t = []
        for h, l in pairs:
            set_scan_config(key, h, default_cfg["bc_head_blocks"], l,
                            default_cfg["bc_head_blocks_light"], lib=lib)
            scan_t.append((time_us(), (h, l)))
        best_scan = min(scan_t)[1]
        timings = []
        for h, l in pairs:
            set_scan_config(key, best_scan[0], h, best_scan[1], l, lib=lib)
            timings.append((time_us(), (h, l)))
    finally:
        if had:
            set_scan_config(key, lib=lib, **saved)
        else:
            clear_scan_config(key, lib=lib)
    best_us, best_bc = min(timings)
    best = dict(scan_head_blocks=best_scan[0], bc_head_blocks=best_bc[0],
                scan_head_blocks_light=best_scan[1], bc_head_blocks_light=best_bc[1])
    return dict(**key, **best, workload=workload, tuned_us=round(best_us, 2),
                default_us=round(default_us, 2), default=default_cfg,
                scan_sweep={f"{h},{l}": round(us, 2) for us, (h, l) in scan_t},
                bc_sweep={f"{h},{l}": round(us, 2) for us, (h, l) in timings})


def main(argv=None):
    ap = argparse.ArgumentParser(description=__doc__.split("\n")[0])
    ap.add_argument("--sweep", default=None,
                    help="comma-separated features:group_size shapes, e.g. 4096:512,1536:1536")
    ap.add_argument("--sweep-scan", default=None,
                    help="comma-separated SSD workloads, e.g. layer_fwdbwd_bf16,hybrid_bf16")
    ap.add_argument("--dtype", default="bf16", choices=sorted(_DTYPES))
    ap.add_argument("--rows", type=int, default=16384)
    ap.add_argument("--out", required=True)
    args = ap.parse_args(argv)
    import torch
    if args.sweep_scan:
        os.environ.setdefault("SSD_SCAN_TABLE", "none")
        entries = []
        for w in args.sweep_scan.split(","):
            e = sweep_scan(w)
            print(json.dumps(e))
            entries.append(e)
        table = {"kind": SCAN_TABLE_KIND, "gpu": torch.cuda.get_device_name(),
                 "sms": torch.cuda.get_device_properties(0).multi_processor_count,
                 "generated_by": "SSD_SCAN_TABLE=none python -m state_space_model_sm_gb300.tuning "
                                 "--sweep-scan " + args.sweep_scan + " --out <table>",
                 "entries": entries}
        validate_scan_table(table)
        with open(args.out, "w") as f:
            json.dump(table, f, indent=1)
        return
    if not args.sweep:
        ap.error("--sweep or --sweep-scan is required")
    entries = []
    for item in args.sweep.split(","):
        F, G = (int(v) for v in item.split(":"))
        e = sweep_gated_norm(F, G, args.dtype, rows=args.rows)
        print(json.dumps(e))
        entries.append(e)
    table = {"kind": TABLE_KIND, "gpu": torch.cuda.get_device_name(),
             "sms": torch.cuda.get_device_properties(0).multi_processor_count,
             "generated_by": "python -m state_space_model_sm_gb300.tuning --sweep " + args.sweep
                             + f" --dtype {args.dtype} --rows {args.rows}",
             "entries": entries}
    validate_table(table)
    with open(args.out, "w") as f:
        json.dump(table, f, indent=1)


if __name__ == "__main__":
    main()
