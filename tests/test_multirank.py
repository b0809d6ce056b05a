"""The N > 1 launch path of bench.py, on CPU ranks (gloo / torchrun on 127.0.0.1).

One GPU per box means the data-parallel path only ever runs as independent
replicas: every rank times its own batch and the job's throughput is the
tokens of all ranks over the slowest rank's time.  These tests check that
reduction on two gloo ranks and the reference arm's launch contract under
torchrun (rank 0 prints the one JSON line, the other rank exits 0 without work).
"""
import json
import os
import socket
import subprocess
import sys

import pytest

ROOT = os.path.dirname(os.path.dirname(os.path.abspath(__file__)))


def _free_port():
    with socket.socket(socket.AF_INET, socket.SOCK_STREAM) as s:
        s.bind(("127.0.0.1", 0))
        return s.getsockname()[1]


def _rank_main(rank, world, port, out_dir):
    sys.path.insert(0, ROOT)
    import torch.distributed as dist

    import bench
    os.environ["MASTER_ADDR"] = "127.0.0.1"
    os.environ["MASTER_PORT"] = str(port)
    dist.init_process_group("gloo", rank=rank, world_size=world)
    try:
        # rank r took 10 (r + 1) ms for 1000 tokens
        ms, value = bench.aggregate_over_ranks(10.0 * (rank + 1), 1000, world, None)
        with open(os.path.join(out_dir, f"rank{rank}.json"), "w") as f:
            json.dump({"ms": ms, "value": value}, f)
    finally:
        dist.destroy_process_group()


def test_aggregate_over_ranks_gloo(tmp_path):
    import torch.multiprocessing as mp
    world = 2
    mp.spawn(_rank_main, args=(world, _free_port(), str(tmp_path)), nprocs=world, join=True)
    for r in range(world):
        with open(tmp_path / f"rank{r}.json") as f:
            got = json.load(f)
        # every rank sees the slowest rank's time and the whole job's tokens
        assert got["ms"] == pytest.approx(20.0)
        assert got["value"] == pytest.approx(2 * 1000 / 0.020)


def test_aggregate_single_rank_needs_no_group():
    sys.path.insert(0, ROOT)
    import bench
    ms, value = bench.aggregate_over_ranks(4.0, 512, 1)
    assert ms == 4.0 and value == pytest.approx(512 / 0.004)


def test_reference_arm_under_torchrun():
    cmd = [sys.executable, "-m", "torch.distributed.run", "--nnodes=1", "--nproc-per-node", "2",
           "--master-addr", "127.0.0.1", "--master-port", str(_free_port()),
           os.path.join(ROOT, "bench.py"), "--gpus", "2", "--impl", "reference",
           "--workload", "tiny_f32", "--steps", "1", "--warmup", "1"]
    p = subprocess.run(cmd, cwd=ROOT, capture_output=True, text=True, timeout=600)
    assert p.returncode == 0, p.stderr[-2000:]
    lines = [ln for ln in p.stdout.splitlines() if ln.startswith("{")]
    assert len(lines) == 1, p.stdout
    d = json.loads(lines[0])
    assert d["impl"] == "reference" and d["n_gpus"] == 2 and d["value"] > 0
    assert d["e2e"]["h2d_bytes_per_step"] == 0 and d["cpu_baseline"]["kind"] == "oracle"
