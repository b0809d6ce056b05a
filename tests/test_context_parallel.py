"""Context (sequence) parallel SSD against the unsplit sequence.

CPU: the orchestration (``context.cp_forward`` / ``cp_backward``) runs on two
and three gloo ranks, with the fp64 oracle as each rank's engine, and its
concatenated outputs and gradients must equal the oracle's over the whole
sequence to fp64 rounding.  The same check runs on four in-process ranks
(threads) with uneven segments.

GPU: the library's own building blocks (``segment_decay``, ``state_scan``)
against their definitions, and the whole path with the library as engine on
ranks emulated by threads in one process (host-side exchange, no kernel waits
on another), against the oracle over the whole sequence at the parity
tolerances.
"""
import os
import socket
import sys
import threading

import numpy as np
import pytest

ROOT = os.path.dirname(os.path.dirname(os.path.abspath(__file__)))

SHAPE_ARGS = (2, 150, 3, 8, 6, 1, 32)   # batch, seqlen, nheads, headdim, dstate, ngroups, chunk
GRADS = ("dx", "ddt", "dB", "dC")       # cut along the sequence
SHARED = ("dA", "dD", "ddt_bias")       # summed over ranks


def _free_port():
    with socket.socket(socket.AF_INET, socket.SOCK_STREAM) as s:
        s.bind(("127.0.0.1", 0))
        return s.getsockname()[1]


def _inputs(shape_args=SHAPE_ARGS, seed=11, dtype="f32"):
    from state_space_model_sm_gb300.inputs import SSDShape, make_inputs
    return make_inputs(SSDShape(*shape_args), seed=seed, dtype=dtype, init_std=0.3,
                       with_dy=True, dfinal_std=0.5)


def _segment(inp, lo, hi, conv):
    """This rank's slice of the inputs; conv = (storage-dtype, float32) converters."""
    cin, cf = conv
    return dict(x=cin(inp.x[:, lo:hi]), dt=cin(inp.dt[:, lo:hi]), dt_bias=cf(inp.dt_bias),
                A=cf(inp.A), B=cin(inp.B[:, lo:hi]), C=cin(inp.C[:, lo:hi]), D=cf(inp.D))


class OracleEngine:
    """Each rank's steps on the fp64 CPU oracle; decay and scan written out
    from their definitions (product of per-step decays; the affine maps
    composed rank by rank)."""

    def fwd(self, seg, init):
        import oracle
        import torch
        n = {k: v.numpy() for k, v in seg.items()}
        y, f = oracle.ssd_fwd(n["x"], n["dt"], n["dt_bias"], n["A"], n["B"], n["C"], n["D"],
                              None if init is None else init.numpy())
        return torch.from_numpy(y), torch.from_numpy(f)

    def bwd(self, seg, init, dy, dfinal):
        import oracle
        import torch
        n = {k: v.numpy() for k, v in seg.items()}
        g = oracle.ssd_bwd(n["x"], n["dt"], n["dt_bias"], n["A"], n["B"], n["C"], n["D"],
                           None if init is None else init.numpy(), dy.numpy(),
                           None if dfinal is None else dfinal.numpy())
        return {k: torch.from_numpy(v) for k, v in g.items()}

    def final_state(self, seg):
        return self.fwd(seg, None)[1]

    def dinit(self, seg, dy, dfinal):
        return self.bwd(seg, None, dy, dfinal)["dinit"]

    def zeros_state(self, seg):
        import torch
        Bt, _, H, P = seg["x"].shape
        return torch.zeros((Bt, H, P, seg["B"].shape[-1]), dtype=torch.float64)

    def decay(self, seg):
        import torch
        dt, bias, A = (seg[k].numpy() for k in ("dt", "dt_bias", "A"))
        d = np.ones(dt.shape[::2])                      # (b, h)
        for t in range(dt.shape[1]):
            v = dt[:, t, :] + bias[None, :]
            d = d * np.exp(A[None, :] * np.logaddexp(0.0, v))
        return torch.from_numpy(d)

    def scan(self, decays, states, rank, direction):
        import torch
        R = decays.shape[0]
        order = range(rank) if direction == 0 else range(R - 1, rank, -1)
        acc = torch.zeros_like(states[0])
        for k in order:
            acc = decays[k][:, :, None, None] * acc + states[k]
        return acc


class _Hub:
    def __init__(self, world):
        self.world = world
        self.barrier = threading.Barrier(world, timeout=300)
        self.slots = [None] * world


class ThreadComm:
    """In-process exchange between ranks that run as threads."""

    def __init__(self, hub, rank):
        self.hub, self.rank, self.world = hub, rank, hub.world

    def allgather(self, t):
        import torch
        if t.is_cuda:
            torch.cuda.current_stream(t.device).synchronize()
        self.hub.slots[self.rank] = t
        self.hub.barrier.wait()
        out = torch.stack(list(self.hub.slots))
        self.hub.barrier.wait()
        return out

    def allreduce_sum(self, t):
        t.copy_(self.allgather(t).sum(0))
        return t


def _run_rank(engine, comm, inp, bounds, conv):
    from state_space_model_sm_gb300 import context
    lo, hi = bounds[comm.rank], bounds[comm.rank + 1]
    seg = _segment(inp, lo, hi, conv)
    cin, cf = conv
    init = cf(inp.init) if comm.rank == 0 else None
    y, h_out, h_in = context.cp_forward(engine, comm, seg, init)
    last = comm.rank == comm.world - 1
    g = context.cp_backward(engine, comm, seg, h_in, cin(inp.dy[:, lo:hi]),
                            cf(inp.dfinal) if last else None)
    out = dict(y=y, final=h_out)
    out.update(g)
    return {k: v.detach().double().cpu().numpy() for k, v in out.items() if v is not None}


def _run_threads(engine_for, inp, sizes, conv):
    world = len(sizes)
    bounds = np.concatenate([[0], np.cumsum(sizes)]).tolist()
    hub = _Hub(world)
    results, errors = [None] * world, []

    def body(r):
        try:
            results[r] = _run_rank(engine_for(r), ThreadComm(hub, r), inp, bounds, conv)
        except BaseException as e:  # noqa: BLE001 -- reported below
            errors.append(e)
            hub.barrier.abort()

    ths = [threading.Thread(target=body, args=(r,)) for r in range(world)]
    for t in ths:
        t.start()
    for t in ths:
        t.join()
    if errors:
        raise errors[0]
    return results


def _full_oracle(inp):
    import oracle
    y, final = oracle.ssd_fwd(inp.x, inp.dt, inp.dt_bias, inp.A, inp.B, inp.C, inp.D, inp.init)
    g = oracle.ssd_bwd(inp.x, inp.dt, inp.dt_bias, inp.A, inp.B, inp.C, inp.D, inp.init, inp.dy,
                       inp.dfinal)
    return y, final, g


def _assemble(results):
    got = {k: np.concatenate([r[k] for r in results], axis=1) for k in ("y",) + GRADS}
    got["final"] = results[-1]["final"]
    for k in SHARED:
        got[k] = results[0][k]
        for r in results[1:]:  # every rank holds the same sum
            np.testing.assert_array_equal(r[k], got[k])
    got["dinit"] = results[0]["dinit"]
    assert all("dinit" not in r for r in results[1:])
    return got


def _check_fp64(got, inp):
    y, final, g = _full_oracle(inp)
    ref = dict(y=y, final=final, **{k: g[k] for k in GRADS + SHARED + ("dinit",)})
    for k, r in ref.items():
        np.testing.assert_allclose(got[k], r, rtol=1e-9, atol=1e-11, err_msg=k)


def _torch_f64(a):
    import torch
    return None if a is None else torch.from_numpy(np.ascontiguousarray(a, dtype=np.float64))


F64 = (_torch_f64, _torch_f64)


# ---------------------------------------------------------------- CPU ----

def test_split_sizes():
    from state_space_model_sm_gb300.context import split_sizes
    assert split_sizes(8192, 4, 256) == [2048] * 4
    assert split_sizes(300, 2, 128) == [256, 44]
    assert split_sizes(300, 3, 128) == [128, 128, 44]
    assert split_sizes(7, 7) == [1] * 7
    assert split_sizes(100, 2, 64) == [64, 36]
    with pytest.raises(ValueError):
        split_sizes(100, 3, 64)      # two chunks of 64 for three ranks


def test_threads_oracle_four_ranks_uneven():
    inp = _inputs()
    res = _run_threads(lambda r: OracleEngine(), inp, [40, 7, 64, 39], F64)
    _check_fp64(_assemble(res), inp)


def test_single_rank_is_the_plain_path():
    inp = _inputs()
    res = _run_threads(lambda r: OracleEngine(), inp, [inp.shape.seqlen], F64)
    _check_fp64(_assemble(res), inp)


def _gloo_rank(rank, world, port, out_dir, sizes):
    sys.path.insert(0, ROOT)
    import torch.distributed as dist

    from state_space_model_sm_gb300.context import DistComm
    os.environ["MASTER_ADDR"] = "127.0.0.1"
    os.environ["MASTER_PORT"] = str(port)
    dist.init_process_group("gloo", rank=rank, world_size=world)
    try:
        inp = _inputs()
        bounds = np.concatenate([[0], np.cumsum(sizes)]).tolist()
        res = _run_rank(OracleEngine(), DistComm(), inp, bounds, F64)
        np.savez(os.path.join(out_dir, f"rank{rank}.npz"), **res)
    finally:
        dist.destroy_process_group()


@pytest.mark.parametrize("sizes", [[96, 54], [32, 64, 54]])
def test_gloo_ranks_match_unsplit_oracle(tmp_path, sizes):
    import torch.multiprocessing as mp
    world = len(sizes)
    mp.spawn(_gloo_rank, args=(world, _free_port(), str(tmp_path), sizes), nprocs=world,
             join=True)
    res = []
    for r in range(world):
        with np.load(tmp_path / f"rank{r}.npz") as z:
            res.append({k: z[k] for k in z.files})
    _check_fp64(_assemble(res), _inputs())


def test_planted_scan_mistake_is_caught():
    """A scan that forgets the decay of the ranks in between must fail the
    check against the unsplit sequence (the test can see such a mistake)."""
    import torch

    class Broken(OracleEngine):
        def scan(self, decays, states, rank, direction):
            return super().scan(torch.ones_like(decays), states, rank, direction)
    inp = _inputs()
    res = _run_threads(lambda r: Broken(), inp, [50, 50, 50], F64)
    with pytest.raises(AssertionError):
        _check_fp64(_assemble(res), inp)


# ---------------------------------------------------------------- GPU ----

@pytest.mark.gpu
@pytest.mark.parametrize("dtype,B,T,H", [("f32", 3, 1000, 5), ("bf16", 3, 1000, 5),
                                          ("bf16", 1, 70001, 37), ("f32", 2, 1, 33)])
def test_segment_decay_matches_definition(cuda_lib, dtype, B, T, H):
    """Many sequence splits with a ragged last one, heads beyond one warp's
    32 lanes, and a single position."""
    import torch

    from state_space_model_sm_gb300.inputs import SSDShape, make_inputs
    inp = make_inputs(SSDShape(B, T, H, 8, 8, 1, 64), seed=21, dtype=dtype)
    tdt = torch.bfloat16 if dtype == "bf16" else torch.float32
    dt = torch.from_numpy(inp.dt).to("cuda", tdt)
    # A scaled down with the length, so that the decay over the whole segment
    # stays well inside float range and the summed steps are really compared
    A = (inp.A * np.float32(min(1.0, 100.0 / T))).astype(np.float32)
    got = cuda_lib.segment_decay(dt, torch.from_numpy(inp.dt_bias).cuda(),
                                 torch.from_numpy(A).cuda()).double().cpu().numpy()
    s = np.logaddexp(0.0, inp.dt.astype(np.float64) + inp.dt_bias[None, None, :]).sum(1)
    ref = np.exp(A[None, :].astype(np.float64) * s)
    assert ref.min() > 1e-30
    np.testing.assert_allclose(got, ref, rtol=2e-5, atol=0)


@pytest.mark.gpu
@pytest.mark.parametrize("dtype,shape_args", [
    ("f32", (2, 300, 4, 16, 32, 2, 64)),          # generic kernels, ragged last chunk
    ("bf16", (2, 1000, 8, 64, 128, 2, 256)),      # tensor-core kernels, ragged last chunk
    ("bf16", (1, 640, 4, 64, 64, 1, 128)),
    ("bf16", (1, 640, 3, 128, 64, 3, 128)),       # headdim 128 on the tensor cores
])
def test_first_passes_match_oracle(cuda_lib, dtype, shape_args):
    """ssd_final_state = the oracle forward's final state; ssd_dinit = the
    oracle backward's initial-state gradient (with and without dfinal)."""
    import torch

    import oracle
    from parity_util import assert_close, to_np
    inp = _inputs(shape_args, seed=41, dtype=dtype)
    tdt = torch.bfloat16 if dtype == "bf16" else torch.float32

    def cv(a, dt=tdt):
        return torch.from_numpy(np.ascontiguousarray(a)).to("cuda", dt)
    f32 = torch.float32
    x, dt, B, C, dy = (cv(a) for a in (inp.x, inp.dt, inp.B, inp.C, inp.dy))
    dtb, A, init, dfin = (cv(a, f32) for a in (inp.dt_bias, inp.A, inp.init, inp.dfinal))
    L = shape_args[-1]
    _, f_ref = oracle.ssd_fwd(inp.x, inp.dt, inp.dt_bias, inp.A, inp.B, inp.C, inp.D, inp.init)
    f = cuda_lib.ssd_final_state(x, dt, dtb, A, B, chunk_size=L, init_states=init)
    assert_close("final", to_np(f), f_ref, dtype)
    for with_dfinal in (False, True):
        g_ref = oracle.ssd_bwd(inp.x, inp.dt, inp.dt_bias, inp.A, inp.B, inp.C, inp.D, None,
                               inp.dy, inp.dfinal if with_dfinal else None)["dinit"]
        g = cuda_lib.ssd_dinit(x, dt, dtb, A, C, dy, chunk_size=L,
                               dfinal_states=dfin if with_dfinal else None)
        assert_close(f"dinit(dfinal={with_dfinal})", to_np(g), g_ref, dtype)
    assert cuda_lib.device_status() == 0


@pytest.mark.gpu
@pytest.mark.parametrize("R", [1, 2, 5])
def test_state_scan_matches_definition(cuda_lib, R):
    import torch
    rng = np.random.default_rng(R)
    dec = rng.uniform(0.2, 1.0, size=(R, 2, 3)).astype(np.float32)
    st = rng.standard_normal((R, 2, 3, 4, 5)).astype(np.float32)
    eng = OracleEngine()
    for rank in range(R):
        for direction in (0, 1):
            got = cuda_lib.state_scan(torch.from_numpy(dec).cuda(), torch.from_numpy(st).cuda(),
                                      rank, direction).double().cpu().numpy()
            ref = eng.scan(_torch_f64(dec), _torch_f64(st), rank, direction).numpy()
            np.testing.assert_allclose(got, ref, rtol=1e-5, atol=1e-6)


@pytest.mark.gpu
@pytest.mark.parametrize("dtype,shape_args,sizes", [
    ("f32", (2, 700, 4, 16, 32, 2, 64), [256, 192, 252]),
    ("bf16", (2, 2048, 8, 64, 128, 2, 256), [1024, 512, 512]),
    ("bf16", (1, 1024, 4, 128, 128, 1, 256), [512, 256, 256]),
])
def test_library_context_parallel_matches_unsplit_oracle(cuda_lib, dtype, shape_args, sizes):
    import torch

    from parity_util import assert_close
    from state_space_model_sm_gb300.context import LibraryEngine
    inp = _inputs(shape_args, seed=31, dtype=dtype)
    tdt = torch.bfloat16 if dtype == "bf16" else torch.float32

    def to(dt):
        return lambda a: None if a is None else torch.from_numpy(np.ascontiguousarray(a)).to(
            "cuda", dt)

    lock = threading.Lock()

    class Locked(LibraryEngine):
        def fwd(self, *a):
            with lock:
                return super().fwd(*a)

        def bwd(self, *a):
            with lock:
                return super().bwd(*a)

    L = shape_args[-1]
    res = _run_threads(lambda r: Locked(L), inp, sizes, (to(tdt), to(torch.float32)))
    got = _assemble(res)
    y, final, g = _full_oracle(inp)
    ref = dict(y=y, final=final, **{k: g[k] for k in GRADS + SHARED + ("dinit",)})
    for k, r in ref.items():
        assert_close(k, got[k], r, dtype)


def test_random_splits_match_unsplit_oracle():
    """Property check of the orchestration: any split of the sequence into 1..5
    contiguous non-empty segments gives the unsplit outputs and gradients."""
    hyp = pytest.importorskip("hypothesis")
    st = pytest.importorskip("hypothesis.strategies")
    inp = _inputs((1, 60, 2, 4, 3, 1, 16), seed=5)

    @hyp.settings(max_examples=15, deadline=None, derandomize=True)
    @hyp.given(cuts=st.lists(st.integers(1, 59), min_size=0, max_size=4, unique=True))
    def check(cuts):
        bounds = [0] + sorted(cuts) + [60]
        sizes = [b - a for a, b in zip(bounds, bounds[1:])]
        res = _run_threads(lambda r: OracleEngine(), inp, sizes, F64)
        _check_fp64(_assemble(res), inp)
    check()
