"""Host-side pieces of bench.py and roofline.py (no GPU): the measured-traffic
lookup and its staleness check, the roofline arithmetic, the peaks file and
its fallback, and the algorithmic byte counts of the gated norm."""
import hashlib
import json
import os
import sys

import pytest

ROOT = os.path.dirname(os.path.dirname(os.path.abspath(__file__)))
sys.path.insert(0, ROOT)

import bench  # noqa: E402
from state_space_model_sm_gb300 import roofline  # noqa: E402


def _fake_root(tmp_path, src_text="kernel v1", workload="wl"):
    (tmp_path / "profiles").mkdir()
    (tmp_path / "k.cu").write_text(src_text)
    sha = hashlib.sha256(src_text.encode()).hexdigest()
    entry = {"k_x": {"bytes_per_launch": 1234, "workload": workload, "sources": ["k.cu"],
                     "sources_sha256": sha}}
    (tmp_path / "profiles" / "dram_traffic.json").write_text(json.dumps(entry))
    return tmp_path


def test_measured_traffic_current_sources(tmp_path, monkeypatch):
    monkeypatch.setattr(bench, "ROOT", str(_fake_root(tmp_path)))
    assert bench.measured_traffic("k_x", "wl") == 1234


def test_measured_traffic_stale_or_other_workload(tmp_path, monkeypatch):
    root = _fake_root(tmp_path)
    monkeypatch.setattr(bench, "ROOT", str(root))
    assert bench.measured_traffic("k_x", "other") is None      # another workload
    assert bench.measured_traffic("k_y", "wl") is None         # never captured
    (root / "k.cu").write_text("kernel v2")                      # the kernel changed
    assert bench.measured_traffic("k_x", "wl") is None


def test_committed_traffic_entries_name_existing_sources():
    with open(os.path.join(ROOT, "profiles", "dram_traffic.json")) as f:
        table = json.load(f)
    for name, e in table.items():
        assert e["bytes_per_launch"] == e["dram_bytes_read"] + e["dram_bytes_write"], name
        for src in e["sources"]:
            assert os.path.exists(os.path.join(ROOT, src)), (name, src)
        assert os.path.exists(os.path.join(ROOT, e["summary"])), name


def test_peaks_file_and_fallback(tmp_path, monkeypatch):
    monkeypatch.setattr(bench, "ROOT", str(tmp_path))
    p = bench.load_peaks()
    assert p["source"] == "fallback" and p["hbm"] == 6800.0 and p["bf16"] == 1900.0
    (tmp_path / "MEASURED_PEAKS.json").write_text(
        json.dumps({"hbm_gbs": 7000.0, "bf16_tflops": 2000.0, "bf16_tflops_sustained": 1800.0}))
    p = bench.load_peaks()
    assert p["source"] == "measured" and p["hbm"] == 7000.0 and p["bf16_sustained"] == 1800.0


def test_kernel_roofline_hbm_arithmetic():
    d = roofline.Dims(4, 4096, 24, 64, 128, 1, 256)
    nbytes = roofline.kernel_bytes("k_state_passing", d)
    peaks = {"hbm": 8000.0, "bf16": 2000.0, "source": "test"}
    r = bench.kernel_roofline("k_state_passing", {"us_per_launch": 10.0}, d, peaks, roofline)
    assert r["bound"] == "hbm" and r["unit"] == "GB/s"
    assert r["achieved"] == pytest.approx(nbytes / 10e-6 / 1e9, rel=1e-3)
    assert r["frac"] == pytest.approx(r["hbm_GBps"] / 8000.0)


def test_norm_kernel_bytes():
    d = roofline.NormDims(rows=16384, features=4096, group_size=512, ib=2, ob=2)
    md = 16384 * 4096
    rstd = 16384 * 8 * 4
    assert roofline.norm_kernel_bytes("k_gated_norm_fwd", d) == md * 6 + rstd
    assert roofline.norm_kernel_bytes("k_gated_norm_bwd", d) == md * 10 + rstd
    assert roofline.norm_kernel_bytes("k_norm_dw_reduce", d) == 4096 * 4
    with pytest.raises(KeyError):
        roofline.norm_kernel_bytes("k_other", d)
