"""Context (sequence) parallel SSD: the sequence cut into contiguous segments,
one per rank, joined by one exchange of per-segment states.

Over a segment r the SSD recurrence (h_t = exp(delta_t A) h_{t-1} +
delta_t x_t B_t, "Mamba-2 offers a different scaling path") maps the state
that enters it affinely to the state that leaves it:

    H_out(r) = D_r * H_in(r) + F_r,   D_r = exp(A * sum_{t in r} delta_t)

with F_r the segment's final state from a zero start.  So:

forward
  1. rank 0 runs the whole forward from the caller's initial state (its
     final state is F_0); ranks 0 < r < R-1 compute only F_r, the final
     state from a zero start (chunk_cumsum, chunk_state, state_passing: no
     chunk_scan); every rank computes D_r;
  2. one all-gather of (D_r, F_r) (the last rank's map is applied by no
     one: it sends zeros);
  3. rank r > 0 scans ranks 0 .. r-1 to its incoming state H_in(r) and runs
     the whole forward from it.

backward (loss <dy, y> + <dfinal, H_out(R-1)>)
  1. ranks r > 0 compute only G_r, the gradient of their incoming state
     with dfinal = 0 (the last rank: the caller's dfinal), from dy, C and the
     decays (chunk_cumsum, dstates, the reverse chunk recurrence); it does
     not depend on the incoming state;
  2. one all-gather of G_r (rank 0's is read by no one: it sends zeros);
  3. rank r < R-1 scans ranks R-1 .. r+1 backwards to dL/dH_out(r), and
     every rank runs the whole backward once with it as dfinal;
  4. dA, dD and ddt_bias (shared over the sequence) are summed over ranks.

So each rank runs one forward and one backward over its segment, plus the
two cheap first passes and the exchange.

The step on the device is the engine's (``LibraryEngine``: the CUDA library);
the exchange is the communicator's (``DistComm``: ``torch.distributed``).
Both are duck-typed, so another engine or communicator can stand in.
"""
from __future__ import annotations

__all__ = ["LibraryEngine", "DistComm", "cp_forward", "cp_backward", "split_sizes"]

_SHARED = ("dA", "dD", "ddt_bias")


def split_sizes(seqlen: int, nranks: int, multiple: int = 1):
    """Segment lengths for ``nranks`` ranks: as even as possible, each a
    multiple of ``multiple`` except the last, which takes the remainder."""
    if nranks < 1 or seqlen < nranks:
        raise ValueError("need 1 <= nranks <= seqlen")
    units = -(-seqlen // multiple)
    base, extra = divmod(units, nranks)
    if base == 0:
        raise ValueError("fewer chunks than ranks")
    sizes = [(base + (1 if r < extra else 0)) * multiple for r in range(nranks)]
    sizes[-1] -= sum(sizes) - seqlen
    return sizes


class LibraryEngine:
    """Per-segment steps on the CUDA library: ``ssd_fwd``, ``ssd_bwd``, the
    first passes ``ssd_fwd_final_state`` / ``ssd_bwd_dinit``, and the
    exchange's arithmetic ``ssd_segment_decay`` / ``ssd_state_scan``."""

    def __init__(self, chunk_size: int = 256):
        from . import segment_decay, ssd_bwd, ssd_dinit, ssd_final_state, ssd_fwd, state_scan
        self.chunk_size = chunk_size
        self._fwd, self._bwd = ssd_fwd, ssd_bwd
        self._final, self._dinit = ssd_final_state, ssd_dinit
        self._decay, self._scan = segment_decay, state_scan

    def fwd(self, seg, init):
        return self._fwd(seg["x"], seg["dt"], seg["dt_bias"], seg["A"], seg["B"], seg["C"],
                         seg.get("D"), chunk_size=self.chunk_size, init_states=init)

    def bwd(self, seg, init, dy, dfinal):
        x = seg["x"]
        if init is None:  # the gradient of the incoming state is always returned
            init = self.zeros_state(seg)
        g = self._bwd(x, seg["dt"], seg["dt_bias"], seg["A"], seg["B"], seg["C"], seg.get("D"),
                      self.chunk_size, init, dy, dfinal)
        g["dinit"] = g.pop("dinit_states")
        return g

    def final_state(self, seg):
        return self._final(seg["x"], seg["dt"], seg["dt_bias"], seg["A"], seg["B"],
                           chunk_size=self.chunk_size)

    def dinit(self, seg, dy, dfinal):
        return self._dinit(seg["x"], seg["dt"], seg["dt_bias"], seg["A"], seg["C"], dy,
                           chunk_size=self.chunk_size, dfinal_states=dfinal)

    def zeros_state(self, seg):
        import torch
        x = seg["x"]
        Bt, _, H, P = x.shape
        return torch.zeros((Bt, H, P, seg["B"].shape[-1]), dtype=torch.float32, device=x.device)

    def decay(self, seg):
        return self._decay(seg["dt"], seg["dt_bias"], seg["A"])

    def scan(self, decays, states, rank, direction):
        return self._scan(decays, states, rank, direction)


class DistComm:
    """The exchange over the default ``torch.distributed`` process group."""

    def __init__(self, group=None):
        import torch.distributed as dist
        self._dist, self.group = dist, group
        self.rank = dist.get_rank(group)
        self.world = dist.get_world_size(group)

    def allgather(self, t):
        import torch
        t = t.contiguous()
        parts = [torch.empty_like(t) for _ in range(self.world)]
        self._dist.all_gather(parts, t, group=self.group)
        return torch.stack(parts)

    def allreduce_sum(self, t):
        self._dist.all_reduce(t, group=self.group)
        return t


def cp_forward(engine, comm, seg, init=None):
    """Forward over this rank's segment ``seg`` (dict of x, dt, dt_bias, A,
    B, C, D; x/dt/B/C cut along the sequence).  ``init`` is the sequence's
    initial state and is read on rank 0 only.

    Returns (y, H_out, H_in): this segment's output, the state leaving it
    (the sequence's final state on the last rank) and the state entering it
    (None on rank 0 without ``init``), which ``cp_backward`` takes back."""
    R, r = comm.world, comm.rank
    if r == 0:
        y, final = engine.fwd(seg, init)
        if R == 1:
            return y, final, init
        send = final
    elif r < R - 1:
        send = engine.final_state(seg)
    else:
        send = engine.zeros_state(seg)
    decays = comm.allgather(engine.decay(seg))
    finals = comm.allgather(send)
    if r == 0:
        return y, final, init
    h_in = engine.scan(decays, finals, r, 0)
    y, final = engine.fwd(seg, h_in)
    return y, final, h_in


def cp_backward(engine, comm, seg, h_in, dy, dfinal=None):
    """Gradients of <dy, y> + <dfinal, H_out(last rank)> for this rank's
    segment, ``h_in`` as ``cp_forward`` returned it and ``dfinal`` read on the
    last rank only.  dx, ddt, dB, dC are this segment's; dA, dD, ddt_bias
    are summed over ranks; "dinit" (the gradient of the sequence's initial
    state) is returned on rank 0 only."""
    R, r = comm.world, comm.rank
    last = r == R - 1
    if R == 1:
        return engine.bwd(seg, h_in, dy, dfinal)
    send = engine.dinit(seg, dy, dfinal if last else None) if r > 0 else engine.zeros_state(seg)
    decays = comm.allgather(engine.decay(seg))
    gin = comm.allgather(send)
    g = engine.bwd(seg, h_in, dy, dfinal if last else engine.scan(decays, gin, r, 1))
    for k in _SHARED:
        if g.get(k) is not None:
            g[k] = comm.allreduce_sum(g[k])
    if r != 0:
        g.pop("dinit", None)
    return g
