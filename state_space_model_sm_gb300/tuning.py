"""Offline launch-configuration table for the gated-norm kernels.

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
    """Called once when the library is loaded: applies the table named by
    SSD_TUNING_TABLE (``none``: no table), else the packaged one if present.
    Returns the path applied, or None."""
    path = os.environ.get("SSD_TUNING_TABLE", DEFAULT_TABLE)
    if path.lower() == "none" or not os.path.exists(path):
        return None
    with open(path) as f:
        apply_table(json.load(f), lib=lib)
    return path


def candidates(features: int) -> Iterable[dict]:
    """Launch configurations worth timing for a row of ``features``."""
    tpr = features // 8
    rpcs = sorted({r for r in (1, 2, 4, 8, 16, 32, 64, 512 // max(tpr, 1))
                   if r >= 1 and r * tpr <= 512 and (r * tpr) % 32 == 0})
    for rpc in rpcs:
        for ring in (32, 64, 96, 128):
            for ctas in (1, 2, 3, 4):
                yield dict(rows_per_item=rpc, ring_kb=ring, ctas_per_sm=ctas)


def sweep_gated_norm(features: int, group_size: int, dtype: str = "bf16", rows: int = 16384,
                     steps: int = 10, warmup: int = 3, seed: int = 0, configs=None) -> dict:
    """Times forward + backward for every candidate configuration of one
    shape on the current GPU (CUDA events around each step, a 512 MB L2
    flush before each) and returns the best entry with the default's time."""
    import torch

    from . import gated_norm_bwd, gated_norm_fwd, gated_norm_workspace_bytes
    lib = _native.load()
    configs = list(configs if configs is not None else candidates(features))
    if not configs:
        raise ValueError(f"no launch configuration for {features} features (at most 4096)")
    dev = torch.device("cuda", torch.cuda.current_device())
    tdt = torch.bfloat16 if dtype == "bf16" else torch.float32
    g = torch.Generator(device="cpu").manual_seed(seed)
    y, z, dout = (torch.randn(rows, features, generator=g).to(dev, tdt) for _ in range(3))
    w = (1.0 + 0.1 * torch.randn(features, generator=g)).to(dev)
    flush = torch.empty(512 * 1024 * 1024 // 4, device=dev)
    ws = torch.empty(gated_norm_workspace_bytes(y, group_size), dtype=torch.uint8, device=dev)
    out, rstd = gated_norm_fwd(y, z, w, group_size)
    grads = gated_norm_bwd(y, z, w, dout, group_size, rstd=rstd, workspace=ws)
    stream = torch.cuda.current_stream(dev)

    def time_us():
        for _ in range(warmup):
            gated_norm_fwd(y, z, w, group_size, out=out, rstd=rstd)
            gated_norm_bwd(y, z, w, dout, group_size, rstd=rstd, workspace=ws, out=grads)
        ev = [(torch.cuda.Event(enable_timing=True), torch.cuda.Event(enable_timing=True))
              for _ in range(steps)]
        for a, b in ev:
            flush.fill_(1.0)
            a.record(stream)
            gated_norm_fwd(y, z, w, group_size, out=out, rstd=rstd)
            gated_norm_bwd(y, z, w, dout, group_size, rstd=rstd, workspace=ws, out=grads)
            b.record(stream)
        torch.cuda.synchronize()
        return 1e3 * sum(a.elapsed_time(b) for a, b in ev) / steps

    saved, had = get_norm_config(features, group_size, dtype, lib=lib)
    clear_norm_config(features, group_size, dtype, lib=lib)
    default_us = time_us()
    default_cfg, _ = get_norm_config(features, group_size, dtype, lib=lib)
    timings = []
    try:
        for cfg in configs:
            set_norm_config(features, group_size, dtype, dtype, lib=lib, **cfg)
            timings.append((time_us(), cfg))
    finally:
        if had:
            set_norm_config(features, group_size, dtype, dtype, lib=lib, **saved)
        else:
            clear_norm_config(features, group_size, dtype, lib=lib)
    best_us, best = min(timings, key=lambda t: t[0])
    return dict(features=features, group_size=group_size, in_dtype=dtype, out_dtype=dtype,
                **best, rows=rows, tuned_us=round(best_us, 2), default_us=round(default_us, 2),
                default=default_cfg, candidates=len(timings))


def main(argv=None):
    ap = argparse.ArgumentParser(description=__doc__.split("\n")[0])
    ap.add_argument("--sweep", required=True,
                    help="comma-separated features:group_size shapes, e.g. 4096:512,1536:1536")
    ap.add_argument("--dtype", default="bf16", choices=sorted(_DTYPES))
    ap.add_argument("--rows", type=int, default=16384)
    ap.add_argument("--out", required=True)
    args = ap.parse_args(argv)
    import torch
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
