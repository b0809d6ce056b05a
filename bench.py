#!/usr/bin/env python
"""SSD forward + backward throughput (tokens/s) on GB300.

One step = ssd_fwd + ssd_bwd over one batch of the Mamba-2 layer workload
(batch 4, seqlen 4096, 24 heads, headdim 64, d_state 128, 1 group, chunk 256,
bf16 inputs, fp32 outputs and gradients), i.e. every step of the chunked scan
and its backward.  Inputs are seeded synthetic data resident in HBM before the
timed region; L2 (129 MB) is flushed by writing a 512 MB buffer before every
timed step, outside the step's CUDA events.

  python bench.py [--gpus N] [--steps K] [--warmup W] [--impl ours|reference]

Under torchrun (N > 1) every rank runs its own batch (weak scaling, no
collective on the data path); the reported time is the max over ranks.
"""
from __future__ import annotations

import argparse
import json
import os
import subprocess
import sys
import threading
import time

ROOT = os.path.dirname(os.path.abspath(__file__))
sys.path.insert(0, ROOT)

WORKLOAD = "layer_fwdbwd_bf16"
METRIC = "SSD fwd+bwd tokens/sec on 1 GB300; % tensor-pipe peak and HBM GB/s per kernel"
UNIT = "tokens/s"
FP32_ALU_PEAK_TFLOPS = 152 * 128 * 2 * 2.07e9 / 1e12   # SMs x FP32 lanes x FMA x max clock


def parse():
    ap = argparse.ArgumentParser()
    ap.add_argument("--gpus", type=int, default=1)
    ap.add_argument("--steps", type=int, default=20)
    ap.add_argument("--warmup", type=int, default=5)
    ap.add_argument("--impl", choices=["ours", "reference"], default="ours")
    ap.add_argument("--workload", default=WORKLOAD)
    ap.add_argument("--no-cpu-baseline", action="store_true")
    ap.add_argument("--context-parallel", type=int, default=0, metavar="R",
                    help="time each rank's share of an R-way sequence split (one GPU)")
    ap.add_argument("--gated-norm", action="store_true",
                    help="time the gated RMSNorm forward + backward instead of the SSD")
    ap.add_argument("--norm-workload", default="norm_hybrid_bf16")
    return ap.parse_args()


def dist_setup(args):
    world = int(os.environ.get("WORLD_SIZE", "1"))
    rank = int(os.environ.get("RANK", "0"))
    local = int(os.environ.get("LOCAL_RANK", "0"))
    return world, rank, local


def aggregate_over_ranks(ms, tokens_per_rank, world, device=None):
    """Whole-job throughput of a timed region: the slowest rank's time (max
    over ranks) and the tokens every rank processed in it.  Returns
    (max_ms, tokens_per_second).  With world > 1 it takes part in one
    all-reduce on the default process group (device: where the reduced tensor
    lives, a CUDA device under NCCL, None for CPU under gloo)."""
    if world > 1:
        import torch
        import torch.distributed as dist
        t = torch.tensor([float(ms)], dtype=torch.float64, device=device)
        dist.all_reduce(t, op=dist.ReduceOp.MAX)
        ms = float(t.item())
    return ms, tokens_per_rank * world / (ms / 1e3)


def workload_config(name, scaling_note):
    from state_space_model_sm_gb300.inputs import WORKLOADS
    shape, dtype, init_std, seed, _ = WORKLOADS[name]
    return {"workload": f"{name}: SSD fwd+bwd batch={shape.batch} seqlen={shape.seqlen} "
                        f"nheads={shape.nheads} headdim={shape.headdim} dstate={shape.dstate} "
                        f"ngroups={shape.ngroups} chunk_size={shape.chunk_size}",
            "batch": shape.batch, "seqlen": shape.seqlen, "nheads": shape.nheads,
            "headdim": shape.headdim, "dstate": shape.dstate, "ngroups": shape.ngroups,
            "chunk_size": shape.chunk_size, "input_dtype": dtype, "grad_dtype": "f32",
            "seed": seed, "l2": scaling_note, "parallelism": "replicas (weak)"}


# ------------------------------------------------------------------ clocks
class ClockSampler:
    """Samples nvidia-smi clocks and throttle reasons while the timed region runs."""

    def __init__(self, index):
        self.index = index
        self.proc = None
        self.lines = []

    def __enter__(self):
        q = ("index,clocks.sm,clocks.max.sm,power.draw,clocks_event_reasons.active,"
             "clocks_event_reasons.hw_slowdown,clocks_event_reasons.hw_thermal_slowdown,"
             "clocks_event_reasons.sw_thermal_slowdown,clocks_event_reasons.sw_power_cap")
        try:
            self.proc = subprocess.Popen(
                ["nvidia-smi", f"--id={self.index}", f"--query-gpu={q}",
                 "--format=csv,noheader,nounits", "-lms", "200"],
                stdout=subprocess.PIPE, stderr=subprocess.DEVNULL, text=True)
            self.thread = threading.Thread(target=self._read, daemon=True)
            self.thread.start()
        except OSError:
            self.proc = None
        time.sleep(0.3)
        return self

    def _read(self):
        for line in self.proc.stdout:
            self.lines.append(line.strip())

    def __exit__(self, *exc):
        if self.proc is not None:
            time.sleep(0.25)
            self.proc.terminate()
            try:
                self.proc.wait(timeout=5)
            except subprocess.TimeoutExpired:
                self.proc.kill()

    def summary(self):
        sm, mx, reasons = [], [], set()
        names = ["hw_slowdown", "hw_thermal_slowdown", "sw_thermal_slowdown", "sw_power_cap"]
        for ln in self.lines:
            parts = [p.strip() for p in ln.split(",")]
            if len(parts) < 9:
                continue
            try:
                sm.append(float(parts[1]))
                mx.append(float(parts[2]))
            except ValueError:
                continue
            for nm, v in zip(names, parts[5:9]):
                if v.lower() == "active":
                    reasons.add(nm)
        if not sm:
            return None
        sm.sort()
        return {"sm_mhz": sm[len(sm) // 2], "sm_max_mhz": max(mx), "reasons": sorted(reasons),
                "samples": len(sm)}


# -------------------------------------------------------------- our arm
def run_ours(args, world, rank, local):
    import numpy as np
    import torch
    import torch.distributed as dist

    import state_space_model_sm_gb300 as ssd
    from state_space_model_sm_gb300 import roofline
    from state_space_model_sm_gb300.inputs import WORKLOADS, make_inputs, to_torch

    torch.cuda.set_device(local)
    dev = torch.device("cuda", local)
    ssd.build()
    ssd.load_library()
    shape, dtype, init_std, seed, _ = WORKLOADS[args.workload]
    inp = make_inputs(shape, seed=seed + 1000 * rank, dtype=dtype, init_std=init_std,
                      with_dy=True)
    t = to_torch(inp, dev)
    Bt, T, H, P, N, G, L = (shape.batch, shape.seqlen, shape.nheads, shape.headdim,
                            shape.dstate, shape.ngroups, shape.chunk_size)
    f32 = dict(dtype=torch.float32, device=dev)
    y = torch.empty((Bt, T, H, P), **f32)
    final = torch.empty((Bt, H, P, N), **f32)
    grads = dict(dx=torch.empty((Bt, T, H, P), **f32), ddt=torch.empty((Bt, T, H), **f32),
                 dA=torch.empty((H,), **f32), dB=torch.empty((Bt, T, G, N), **f32),
                 dC=torch.empty((Bt, T, G, N), **f32), dD=torch.empty((H,), **f32),
                 ddt_bias=torch.empty((H,), **f32))
    if t["init"] is not None:
        grads["dinit_states"] = torch.empty((Bt, H, P, N), **f32)
    sh = ssd.make_shape(Bt, T, H, P, N, G, L, ssd.SSD_BF16 if dtype == "bf16" else ssd.SSD_F32,
                        ssd.SSD_F32)
    ws = torch.empty(max(ssd.fwd_workspace_bytes(sh), ssd.bwd_workspace_bytes(sh)),
                     dtype=torch.uint8, device=dev)
    flush = torch.empty(512 * 1024 * 1024 // 4, dtype=torch.float32, device=dev)

    def step(tt):
        ssd.ssd_fwd(tt["x"], tt["dt"], tt["dt_bias"], tt["A"], tt["B"], tt["C"], tt["D"],
                    chunk_size=L, init_states=tt["init"], workspace=ws, y=y, final_states=final)
        ssd.ssd_bwd(tt["x"], tt["dt"], tt["dt_bias"], tt["A"], tt["B"], tt["C"], tt["D"], L,
                    tt["init"], tt["dy"], None, workspace=ws, out=grads)

    for _ in range(args.warmup):
        step(t)
    torch.cuda.synchronize()
    if ssd.device_status() != 0:
        raise RuntimeError("device status word set during warm-up")

    stream = torch.cuda.current_stream(dev)

    def timed_steps(profiled):
        """K steps, each after an L2 flush and bracketed by CUDA events on the
        launch stream; with profiled, the library also records an event pair
        around every kernel launch (per-kernel durations for the roofline)."""
        starts = [torch.cuda.Event(enable_timing=True) for _ in range(args.steps)]
        ends = [torch.cuda.Event(enable_timing=True) for _ in range(args.steps)]
        launches0 = ssd.launch_count()
        ssd.profile_enable(profiled)
        if world > 1:
            dist.barrier()
        torch.cuda.synchronize()
        for i in range(args.steps):
            flush.fill_(float(i))
            starts[i].record(stream)
            step(t)
            ends[i].record(stream)
        torch.cuda.synchronize()
        if world > 1:
            dist.barrier()
        prof_ = ssd.profile_read() if profiled else None
        ssd.profile_enable(False)
        if ssd.device_status() != 0:
            raise RuntimeError("device status word set during the timed region")
        return (float(sum(s.elapsed_time(e) for s, e in zip(starts, ends))),
                ssd.launch_count() - launches0, prof_)

    with ClockSampler(local) as clk:
        # the throughput: no per-kernel instrumentation inside the timed region
        plain_ms, launches, _ = timed_steps(False)
        # the same K steps again with per-kernel CUDA events (roofline inputs)
        prof_ms, _, prof = timed_steps(True)
    total_ms, value = aggregate_over_ranks(plain_ms, Bt * T * args.steps, world, dev)
    prof_ms, _ = aggregate_over_ranks(prof_ms, Bt * T * args.steps, world, dev)

    # dominant kernel and its roofline
    rd = roofline.Dims(Bt, T, H, P, N, G, L, ib=2 if dtype == "bf16" else 4, ob=4)
    per_kernel = {k: {"ms_total": v[0], "launches": v[1], "us_per_launch": 1e3 * v[0] / v[1]}
                  for k, v in prof.items() if v[1] > 0}
    dom = max(per_kernel, key=lambda k: per_kernel[k]["ms_total"])
    peaks = load_peaks()
    roof = kernel_roofline(dom, per_kernel[dom], rd, peaks, roofline)
    roof["traffic"] = measured_traffic(dom, args.workload)
    kernels_out = {}
    for k, v in per_kernel.items():
        r = kernel_roofline(k, v, rd, peaks, roofline)
        kernels_out[k] = {"us": round(v["us_per_launch"], 2), "launches_per_step":
                          v["launches"] / args.steps, "share": round(v["ms_total"] / sum(
                              x["ms_total"] for x in per_kernel.values()), 4),
                          "hbm_GBps": round(r["hbm_GBps"], 1) if r["hbm_GBps"] else None,
                          "bound": r["bound"],
                          "frac": round(r["frac"], 4) if r["frac"] is not None else None}
        if "tensor_frac" in r:
            kernels_out[k]["tensor_frac"] = round(r["tensor_frac"], 4)

    # end to end: host (pinned) buffers through the same C-ABI calls
    def step_into(tt, o):
        yb, fb, gl = o[0], o[1], o[2:]
        ssd.ssd_fwd(tt["x"], tt["dt"], tt["dt_bias"], tt["A"], tt["B"], tt["C"], tt["D"],
                    chunk_size=L, init_states=tt["init"], workspace=ws, y=yb, final_states=fb)
        ssd.ssd_bwd(tt["x"], tt["dt"], tt["dt_bias"], tt["A"], tt["B"], tt["C"], tt["D"], L,
                    tt["init"], tt["dy"], None, workspace=ws, out=dict(zip(grads.keys(), gl)))

    e2e = run_e2e(args, inp, t, step_into, [y, final] + list(grads.values()), dev, world)

    cpu = None
    if rank == 0 and world == 1 and not args.no_cpu_baseline:
        cpu = cpu_baseline_sample(args.workload)

    if rank == 0:
        out = {
            "metric": METRIC, "value": round(value, 1), "unit": UNIT, "n_gpus": world,
            "steps": args.steps, "warmup": args.warmup,
            "ms_per_step": round(total_ms / args.steps, 4), "higher_is_better": True,
            "scaling": "weak", "vs_baseline": None, "dtype": "bf16 in / f32 accum+grads",
            "data": "synthetic (seeded PCG64, workload distributions)",
            "config": workload_config(args.workload, "flushed (512 MB write) before every step"),
            "roofline": roof, "cpu_baseline": cpu, "e2e": e2e, "gpu_launches": launches,
            "clocks": clk.summary(), "kernels": kernels_out, "path": ssd.last_path(),
            "profiled_ms_per_step": round(prof_ms / args.steps, 4),
            "timing": "value: K steps without per-kernel events; kernels / roofline: the same "
                      "K steps again with an event pair around every launch",
            "gpu": torch.cuda.get_device_name(dev),
            "step_flops_algorithmic": roofline.step_flops(rd),
        }
        print(json.dumps(out))


def load_peaks():
    path = os.path.join(ROOT, "MEASURED_PEAKS.json")
    if os.path.exists(path):
        with open(path) as f:
            p = json.load(f)
        return {"hbm": float(p.get("hbm_gbs")), "bf16": float(p.get("bf16_tflops")),
                "bf16_sustained": float(p.get("bf16_tflops_sustained", p.get("bf16_tflops"))),
                "source": "measured"}
    return {"hbm": 6800.0, "bf16": 1900.0, "bf16_sustained": 1700.0, "source": "fallback"}


def measured_traffic(name, workload):
    """DRAM bytes per launch (dram__bytes_read.sum + dram__bytes_write.sum) of
    one ncu capture of this kernel on this workload, from profiles/; None when
    no capture exists or the kernel sources changed since it was taken."""
    import hashlib
    path = os.path.join(ROOT, "profiles", "dram_traffic.json")
    if not os.path.exists(path):
        return None
    with open(path) as f:
        entry = json.load(f).get(name)
    if not entry or entry.get("workload") != workload:
        return None
    h = hashlib.sha256()
    for src in entry["sources"]:
        with open(os.path.join(ROOT, src), "rb") as f:
            h.update(f.read())
    return int(entry["bytes_per_launch"]) if h.hexdigest() == entry["sources_sha256"] else None


def kernel_roofline(name, v, rd, peaks, roofline):
    """Roofline entry of one kernel from its live CUDA-event time per launch."""
    sec = v["us_per_launch"] / 1e6
    try:
        nbytes = roofline.kernel_bytes(name, rd)
    except KeyError:
        nbytes = None
    try:
        flops = roofline.kernel_flops(name, rd)
    except KeyError:
        flops = None
    gbs = nbytes / sec / 1e9 if nbytes is not None else None
    if flops is not None and not name.endswith("_tc") and not name.endswith("_tc_dx"):
        # generic SIMT contraction: bounded by the fp32 FMA pipes
        ach = flops / sec / 1e12
        return {"kernel": name, "bound": "alu", "achieved": round(ach, 3),
                "peak": round(FP32_ALU_PEAK_TFLOPS, 1), "unit": "TFLOP/s",
                "frac": ach / FP32_ALU_PEAK_TFLOPS, "traffic": None, "hbm_GBps": gbs,
                "algorithmic_bytes": nbytes, "algorithmic_flops": flops,
                "peak_source": "derived: 152 SMs x 128 FP32 lanes x 2 x 2070 MHz"}
    out = {"kernel": name, "bound": "hbm", "achieved": round(gbs, 1) if gbs else None,
           "peak": peaks["hbm"], "unit": "GB/s", "frac": (gbs / peaks["hbm"]) if gbs else None,
           "traffic": None, "hbm_GBps": gbs, "algorithmic_bytes": nbytes,
           "algorithmic_flops": flops, "peak_source": peaks["source"]}
    if flops is not None:
        # tensor-core contraction; at these shapes its arithmetic intensity is
        # below the ridge point, so HBM is the binding roof; the tensor-pipe
        # fraction is reported beside it
        tf = flops / sec / 1e12
        out["tensor_tflops"] = round(tf, 2)
        out["tensor_frac"] = tf / peaks["bf16"]
    return out


def run_e2e(args, inp, t, step_into, outs0, dev, world):
    """The same step through the public API with pinned host buffers: every
    step copies its inputs host->device and reads y, final and every gradient
    back to the host, all inside the timed region.  Like an input pipeline,
    step i+1's inputs go up on one copy stream and step i-1's results come
    down on another while step i computes (inputs and outputs double
    buffered, ordered by events).  Every rank runs it; the value is whole-job
    tokens/s (max time over ranks)."""
    import torch
    names_in = [k for k in ("x", "dt", "dt_bias", "A", "B", "C", "D", "init", "dy")
                if t[k] is not None]
    host_in = {k: t[k].cpu().pin_memory() for k in names_in}
    dev_in = [{k: torch.empty_like(t[k]) for k in names_in} for _ in range(2)]
    outs = [outs0, [torch.empty_like(o) for o in outs0]]
    host_out = [[torch.empty(o.shape, dtype=o.dtype, pin_memory=True) for o in outs0]
                for _ in range(2)]
    h2d = sum(v.numel() * v.element_size() for v in host_in.values())
    d2h = sum(o.numel() * o.element_size() for o in outs0)
    comp = torch.cuda.current_stream(dev)
    s_in, s_out = torch.cuda.Stream(dev), torch.cuda.Stream(dev)
    ev = lambda: torch.cuda.Event(enable_timing=False)
    done = [None, None]      # compute of the last step that used buffer set k
    read_back = [None, None]  # read-back of the last step that used buffer set k
    n = max(3, min(args.steps, 10))
    warm = 2
    for i in range(warm + n):
        k = i % 2
        if i == warm:
            torch.cuda.synchronize()
            start = torch.cuda.Event(enable_timing=True)
            start.record(comp)
            s_in.wait_event(start)
            s_out.wait_event(start)
        with torch.cuda.stream(s_in):
            if done[k] is not None:
                s_in.wait_event(done[k])        # step i-2 is done reading these inputs
            for name in names_in:
                dev_in[k][name].copy_(host_in[name], non_blocking=True)
            ready = ev()
            ready.record(s_in)
        comp.wait_event(ready)
        if read_back[k] is not None:
            comp.wait_event(read_back[k])       # step i-2's results are on the host
        tt = {name: None for name in t}
        tt.update(dev_in[k])
        step_into(tt, outs[k])
        done[k] = ev()
        done[k].record(comp)
        with torch.cuda.stream(s_out):
            s_out.wait_event(done[k])
            for o, h in zip(outs[k], host_out[k]):
                h.copy_(o, non_blocking=True)
            read_back[k] = ev()
            read_back[k].record(s_out)
    for k in range(2):
        comp.wait_event(read_back[k])
    end = torch.cuda.Event(enable_timing=True)
    end.record(comp)
    torch.cuda.synchronize()
    ms, value = aggregate_over_ranks(start.elapsed_time(end) / n,
                                     inp.shape.batch * inp.shape.seqlen, world, dev)
    return {"value": round(value, 1), "unit": UNIT, "ms_per_step": round(ms, 4),
            "h2d_bytes_per_step": int(h2d), "d2h_bytes_per_step": int(d2h),
            "overlap": "copies of steps i+1 / i-1 overlap step i (separate streams)"}


# ------------------------------------------------------------ CPU oracle
def cpu_baseline_sample(workload, min_seconds=10.0):
    """The CPU oracle (fp64 recurrence, forward + reverse sweep, as it stands)
    on batch rows of the same workload, repeated until >= min_seconds."""
    import numpy as np

    import oracle
    from state_space_model_sm_gb300.inputs import WORKLOADS, SSDShape, make_inputs
    shape, dtype, init_std, seed, _ = WORKLOADS[workload]
    one = SSDShape(1, shape.seqlen, shape.nheads, shape.headdim, shape.dstate, shape.ngroups,
                   shape.chunk_size)
    inp = make_inputs(one, seed=seed, dtype=dtype, init_std=init_std, with_dy=True)
    args = oracle.from_inputs(inp)
    dy = inp.dy.astype(np.float64)
    cores = oracle.hardware_threads()
    t0 = time.perf_counter()
    reps = 0
    while True:
        oracle.ssd_fwd(*args, nthreads=cores)
        oracle.ssd_bwd(*args, dy, None, nthreads=cores)
        reps += 1
        el = time.perf_counter() - t0
        if el >= min_seconds or reps >= 50:
            break
    tokens = reps * one.seqlen
    # the same oracle on one host thread, one repetition
    t1 = time.perf_counter()
    oracle.ssd_fwd(*args, nthreads=1)
    oracle.ssd_bwd(*args, dy, None, nthreads=1)
    el1 = time.perf_counter() - t1
    return {"value": round(tokens / el, 1), "unit": UNIT, "cores": cores, "kind": "oracle",
            "sample": f"{reps} x (batch row 0 of {workload}: seqlen {one.seqlen}, "
                      f"{one.nheads} heads), fp64 forward + backward, {el:.1f} s; tokens/s "
                      f"of the whole {shape.batch}-row workload extrapolated from these rows "
                      f"(rows are independent and cost the same)",
            "value_1core": round(one.seqlen / el1, 1),
            "sample_1core": f"1 x the same batch row on 1 thread, {el1:.1f} s"}


def run_reference(args, world, rank):
    """Reference arm: the CPU oracle as it stands on the host cores, on a
    bounded sample (one batch row) of the same workload per step."""
    if rank != 0:
        return
    import numpy as np

    import oracle
    from state_space_model_sm_gb300.inputs import WORKLOADS, SSDShape, make_inputs
    shape, dtype, init_std, seed, _ = WORKLOADS[args.workload]
    one = SSDShape(1, shape.seqlen, shape.nheads, shape.headdim, shape.dstate, shape.ngroups,
                   shape.chunk_size)
    inp = make_inputs(one, seed=seed, dtype=dtype, init_std=init_std, with_dy=True)
    a = oracle.from_inputs(inp)
    dy = inp.dy.astype(np.float64)
    cores = oracle.hardware_threads()

    def step():
        oracle.ssd_fwd(*a, nthreads=cores)
        oracle.ssd_bwd(*a, dy, None, nthreads=cores)
    for _ in range(args.warmup):
        step()
    t0 = time.perf_counter()
    for _ in range(args.steps):
        step()
    el = time.perf_counter() - t0
    value = args.steps * one.seqlen / el
    sample = (f"per step: batch row 0 of {args.workload} (seqlen {one.seqlen}, "
              f"{one.nheads} heads), fp64 forward + backward; tokens/s extrapolated from "
              f"1 of {shape.batch} batch rows (rows are independent and cost the same)")
    print(json.dumps({
        "impl": "reference", "metric": METRIC, "value": round(value, 1), "unit": UNIT,
        "n_gpus": world, "steps": args.steps, "warmup": args.warmup,
        "ms_per_step": round(1e3 * el / args.steps, 3), "higher_is_better": True,
        "scaling": "weak", "vs_baseline": None, "dtype": "f64", "data": "synthetic",
        "config": workload_config(args.workload, "n/a (host)"),
        "cpu_baseline": {"value": round(value, 1), "unit": UNIT, "cores": cores,
                         "kind": "oracle", "sample": sample},
        "e2e": {"value": round(value, 1), "unit": UNIT, "h2d_bytes_per_step": 0,
                "d2h_bytes_per_step": 0}}))


class _StandInComm:
    """The exchange of one rank of an R-way split, stood in for on one GPU:
    the all-gather stacks R copies of the rank's own tensor and the
    all-reduce scales by R (same shapes and device copies, no transfer)."""

    def __init__(self, rank, world):
        self.rank, self.world = rank, world

    def allgather(self, t):
        import torch
        return torch.stack([t] * self.world)

    def allreduce_sum(self, t):
        return t.mul_(self.world)


def run_context_parallel(args):
    """Per-rank step time of the context-parallel path (forward + backward
    over one segment of an R-way split of the workload's sequence), each rank
    role timed in turn on this GPU; the job's step time is the slowest
    rank's.  The exchange (two all-gathers of b*h*p*n floats and one of b*h,
    plus three (h,) all-reduces per step) is stood in for by local copies."""
    import torch

    import state_space_model_sm_gb300 as ssd
    from state_space_model_sm_gb300 import context
    from state_space_model_sm_gb300.inputs import WORKLOADS, make_inputs, to_torch

    R = args.context_parallel
    dev = torch.device("cuda", 0)
    ssd.build()
    ssd.load_library()
    shape, dtype, init_std, seed, _ = WORKLOADS[args.workload]
    inp = make_inputs(shape, seed=seed, dtype=dtype, init_std=init_std, with_dy=True)
    t = to_torch(inp, dev)
    Bt, T, L = shape.batch, shape.seqlen, shape.chunk_size
    sizes = context.split_sizes(T, R, L)
    bounds = [0]
    for n in sizes:
        bounds.append(bounds[-1] + n)
    eng = context.LibraryEngine(L)
    flush = torch.empty(512 * 1024 * 1024 // 4, dtype=torch.float32, device=dev)
    stream = torch.cuda.current_stream(dev)
    per_rank = []
    launches0 = ssd.launch_count()
    with ClockSampler(0) as clk:
        for r in range(R):
            lo, hi = bounds[r], bounds[r + 1]
            seg = {k: (t[k][:, lo:hi].contiguous() if k in ("x", "dt", "B", "C") else t[k])
                   for k in ("x", "dt", "dt_bias", "A", "B", "C", "D")}
            dy = t["dy"][:, lo:hi].contiguous()
            comm = _StandInComm(r, R)

            def step():
                _, _, h_in = context.cp_forward(eng, comm, seg, t["init"] if r == 0 else None)
                context.cp_backward(eng, comm, seg, h_in, dy, None)

            for _ in range(args.warmup):
                step()
            torch.cuda.synchronize()
            ev = [(torch.cuda.Event(enable_timing=True), torch.cuda.Event(enable_timing=True))
                  for _ in range(args.steps)]
            for s0, s1 in ev:
                flush.fill_(1.0)
                s0.record(stream)
                step()
                s1.record(stream)
            torch.cuda.synchronize()
            per_rank.append(sum(a.elapsed_time(b) for a, b in ev) / args.steps)
    if ssd.device_status() != 0:
        raise RuntimeError("device status word set during the timed region")
    launches = ssd.launch_count() - launches0
    ms = max(per_rank)
    out = {
        "metric": METRIC, "impl": "ours", "context_parallel": R,
        "value": round(Bt * T / (ms / 1e3), 1), "unit": UNIT, "n_gpus": 1, "steps": args.steps,
        "warmup": args.warmup, "ms_per_step": round(ms, 4), "higher_is_better": True,
        "scaling": "strong", "vs_baseline": None, "dtype": "bf16 in / f32 accum+grads",
        "data": "synthetic (seeded PCG64, workload distributions)",
        "config": dict(workload_config(args.workload, "flushed (512 MB write) before every step"),
                       segments=sizes),
        "per_rank_ms": [round(v, 4) for v in per_rank],
        "projection": f"value = tokens of the whole sequence over the slowest of the {R} rank "
                      "roles, each timed alone on this GPU; the exchange is stood in for by "
                      "local stacks of the same size (no inter-GPU transfer timed)",
        "gpu_launches": launches, "clocks": clk.summary(),
        "gpu": torch.cuda.get_device_name(dev),
    }
    print(json.dumps(out))


def run_gated_norm(args):
    """Gated RMSNorm forward + backward (the step after the SSD output; its
    backward is the pages' _layer_norm_bwd) on one GPU: tokens (rows) per
    second, per-kernel times and the HBM roofline of the backward."""
    import numpy as np
    import torch

    import state_space_model_sm_gb300 as ssd
    from state_space_model_sm_gb300 import roofline
    from state_space_model_sm_gb300.inputs import NORM_WORKLOADS, make_norm_workload

    dev = torch.device("cuda", 0)
    ssd.build()
    ssd.load_library()
    shape, dtype, seed = NORM_WORKLOADS[args.norm_workload]
    inp = make_norm_workload(args.norm_workload)
    tdt = torch.bfloat16 if dtype == "bf16" else torch.float32

    def cv(a, dt=tdt):
        return torch.from_numpy(np.ascontiguousarray(a)).to(dev, dt)
    y, z, dout, w = cv(inp.y), cv(inp.z), cv(inp.dout), cv(inp.w, torch.float32)
    gs, eps = shape.group_size, shape.eps
    out, rstd = ssd.gated_norm_fwd(y, z, w, gs, eps=eps)
    ws = torch.empty(ssd.gated_norm_workspace_bytes(y, gs, eps), dtype=torch.uint8, device=dev)
    grads = ssd.gated_norm_bwd(y, z, w, dout, gs, eps=eps, rstd=rstd, workspace=ws)
    flush = torch.empty(512 * 1024 * 1024 // 4, dtype=torch.float32, device=dev)
    stream = torch.cuda.current_stream(dev)

    def step():
        ssd.gated_norm_fwd(y, z, w, gs, eps=eps, out=out, rstd=rstd)
        ssd.gated_norm_bwd(y, z, w, dout, gs, eps=eps, rstd=rstd, workspace=ws, out=grads)

    for _ in range(args.warmup):
        step()
    torch.cuda.synchronize()

    def timed(profiled):
        ev = [(torch.cuda.Event(enable_timing=True), torch.cuda.Event(enable_timing=True))
              for _ in range(args.steps)]
        l0 = ssd.launch_count()
        ssd.profile_enable(profiled)
        torch.cuda.synchronize()
        for a, b in ev:
            flush.fill_(1.0)
            a.record(stream)
            step()
            b.record(stream)
        torch.cuda.synchronize()
        prof = ssd.profile_read() if profiled else None
        ssd.profile_enable(False)
        return sum(a.elapsed_time(b) for a, b in ev), ssd.launch_count() - l0, prof

    with ClockSampler(0) as clk:
        ms, launches, _ = timed(False)
        _, _, prof = timed(True)
    if ssd.device_status() != 0:
        raise RuntimeError("device status word set during the timed region")
    rd = roofline.NormDims(shape.rows, shape.features, gs, 2 if dtype == "bf16" else 4,
                           2 if dtype == "bf16" else 4)
    peaks = load_peaks()
    kernels = {}
    for k, (tot, n) in prof.items():
        if n == 0:
            continue
        us = 1e3 * tot / n
        nb = roofline.norm_kernel_bytes(k, rd)
        gbs = nb / (us / 1e6) / 1e9
        kernels[k] = {"us": round(us, 2), "launches_per_step": n / args.steps,
                      "algorithmic_bytes": nb, "hbm_GBps": round(gbs, 1),
                      "frac": round(gbs / peaks["hbm"], 4)}
    dom = "k_gated_norm_bwd"
    roof = {"kernel": dom, "bound": "hbm", "achieved": kernels[dom]["hbm_GBps"],
            "peak": peaks["hbm"], "unit": "GB/s", "frac": kernels[dom]["frac"],
            "traffic": measured_traffic(dom, args.norm_workload),
            "algorithmic_bytes": kernels[dom]["algorithmic_bytes"],
            "peak_source": peaks["source"]}
    cpu = None
    if not args.no_cpu_baseline:
        from oracle import gated_norm as gn
        n = 256
        t0 = time.perf_counter()
        reps = 0
        while time.perf_counter() - t0 < 10.0:
            gn.gated_rmsnorm_fwd(inp.y[:n], inp.z[:n], inp.w, gs, eps=eps)
            gn.gated_rmsnorm_bwd(inp.y[:n], inp.z[:n], inp.w, inp.dout[:n], gs, eps=eps)
            reps += 1
        sec = time.perf_counter() - t0
        cpu = {"value": round(n * reps / sec, 1), "unit": "tokens/s", "cores": 1,
               "kind": "oracle",
               "sample": f"rows 0..{n - 1} of {args.norm_workload}, forward + backward, "
                         f"{reps} repetitions in {sec:.1f} s (numpy fp64, one thread)"}
    from state_space_model_sm_gb300 import tuning
    launch_cfg, from_table = tuning.get_norm_config(shape.features, gs, dtype)
    rows = shape.rows
    out_line = {
        "metric": "gated RMSNorm fwd+bwd tokens/sec on 1 GB300 (the step after the SSD output)",
        "impl": "ours", "value": round(rows * args.steps / (ms / 1e3), 1), "unit": "tokens/s",
        "n_gpus": 1, "steps": args.steps, "warmup": args.warmup,
        "ms_per_step": round(ms / args.steps, 4), "higher_is_better": True, "scaling": "weak",
        "vs_baseline": None, "dtype": f"{dtype} in/out, f32 statistics and dw",
        "data": "synthetic (seeded PCG64: y, z, dout ~ N(0,1), w = 1 + 0.1 N(0,1))",
        "config": {"workload": args.norm_workload, "rows": rows, "features": shape.features,
                   "group_size": gs, "eps": eps, "l2": "flushed (512 MB write) before every step"},
        "roofline": roof, "kernels": kernels, "cpu_baseline": cpu, "gpu_launches": launches,
        "clocks": clk.summary(), "gpu": torch.cuda.get_device_name(dev),
        "launch_config": dict(launch_cfg, source="table" if from_table else "built-in",
                              table=os.environ.get("SSD_TUNING_TABLE", tuning.DEFAULT_TABLE)
                              if from_table else None),
    }
    print(json.dumps(out_line))


def main():
    args = parse()
    world, rank, local = dist_setup(args)
    if args.impl == "reference":
        run_reference(args, world, rank)
        return
    if args.gated_norm:
        if world > 1:
            raise SystemExit("--gated-norm runs on one GPU; run it without torchrun")
        run_gated_norm(args)
        return
    if args.context_parallel:
        if world > 1:
            raise SystemExit("--context-parallel times rank roles on one GPU; run it without torchrun")
        run_context_parallel(args)
        return
    if world > 1:
        import torch
        import torch.distributed as dist
        torch.cuda.set_device(local)
        dist.init_process_group("nccl")
    try:
        run_ours(args, world, rank, local)
    finally:
        if world > 1:
            import torch.distributed as dist
            dist.destroy_process_group()


if __name__ == "__main__":
    main()
