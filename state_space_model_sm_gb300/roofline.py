"""Algorithmic bytes and FLOPs per kernel launch of the SSD scan.

"Algorithmic" means what the chunked method has to move or compute, counted
once: every tensor a kernel consumes is read once and every tensor it produces
is written once, whatever the kernel re-reads through L2; FLOPs count the
multiply-adds of the contractions (2 per MAC) on the causal half where the
method only needs that half.  These are the numerators of the roofline
fractions; the denominators are measured peaks.

Sizes: B batch, T seqlen, H heads, P headdim, N dstate, G groups, L chunk,
nc = ceil(T / L); `ib` = bytes of an input element (2 for bf16, 4 for fp32),
`ob` = bytes of a y element.
"""
from __future__ import annotations

import dataclasses


@dataclasses.dataclass
class Dims:
    B: int
    T: int
    H: int
    P: int
    N: int
    G: int
    L: int
    ib: int = 2
    ob: int = 4

    @property
    def nc(self):
        return -(-self.T // self.L)


def _terms(d: Dims):
    f = 4
    tok = d.B * d.T
    x = tok * d.H * d.P * d.ib          # x, dy (input dtype)
    xf = tok * d.H * d.P * f            # dx (fp32)
    bc = tok * d.G * d.N * d.ib         # one of B, C
    bcf = tok * d.G * d.N * f           # one of dB, dC
    dtb = tok * d.H * d.ib              # dt
    vec = d.B * d.H * d.nc * d.L * f    # delta or dA_cumsum
    st = d.B * d.nc * d.H * d.P * d.N * f   # chunk states (S, Hprev, dHs, dS)
    fin = d.B * d.H * d.P * d.N * f
    cb = d.B * d.nc * d.G * d.L * (d.L + 1) // 2 * f   # causal half of C.B^T
    y = tok * d.H * d.P * d.ob
    return dict(x=x, xf=xf, bc=bc, bcf=bcf, dtb=dtb, vec=vec, st=st, fin=fin, cb=cb, y=y)


def kernel_bytes(name: str, d: Dims) -> int:
    """Algorithmic DRAM bytes of one launch of the kernel `name`."""
    t = _terms(d)
    table = {
        # tensor-core path
        # chunk_state with chunk_cumsum inside: reads dt, writes delta and dA_cumsum
        "k_state_tc": t["x"] + t["bc"] + t["dtb"] + 2 * t["vec"] + t["st"],
        "k_dstates_tc": t["x"] + t["bc"] + t["vec"] + t["st"],
        "k_scan_tc": t["x"] + 2 * t["bc"] + 2 * t["vec"] + t["st"] + t["y"],
        "k_scan_tc_dx": 2 * t["x"] + 2 * t["bc"] + 5 * t["vec"] + t["st"] + t["xf"],
        # dC / dB: the method writes each gradient once; the head-block
        # partials the kernels write instead when nb > 1 (and the tail sums)
        # are the implementation's choice, not counted
        "k_bwd_dc_tc": 2 * t["x"] + 2 * t["bc"] + 4 * t["vec"] + t["st"] + t["bcf"],
        "k_bwd_db_tc": 2 * t["x"] + 2 * t["bc"] + 3 * t["vec"] + t["st"] + t["bcf"],
        # ddA / ddt finalize (with the dC / dB head-block sums in the same launch)
        "k_bwd_tail_tc": t["dtb"] + 7 * t["vec"] + d.B * d.T * d.H * 4,
        # forward
        "k_chunk_cumsum": t["dtb"] + 2 * t["vec"],
        "k_bmm_cb": 2 * t["bc"] + t["cb"],
        "k_chunk_state": t["x"] + t["bc"] + 2 * t["vec"] + t["st"],
        "k_state_passing": 2 * t["st"] + t["vec"] // d.L + t["fin"],
        "k_chunk_scan": t["x"] + t["bc"] + t["cb"] + 2 * t["vec"] + t["st"] + t["y"],
        # backward
        "k_state_passing_bwd": 3 * t["st"] + t["vec"] // d.L + t["fin"],
        "k_dyx": 2 * t["x"],
        "k_bwd_dx": 2 * t["x"] + t["bc"] + t["cb"] + 2 * t["vec"] + t["st"] + t["xf"],
        "k_bwd_dC": t["x"] + 2 * t["bc"] + 2 * t["vec"] + t["st"] + t["bcf"] * d.H // d.G,
        "k_bwd_dB": t["x"] + t["bc"] + 2 * t["vec"] + t["st"] + t["bcf"] * d.H // d.G,
        "k_bwd_ddA": t["dtb"] + t["cb"] + 2 * t["vec"] + d.B * d.T * d.H * 4,
        "k_group_reduce": t["bcf"] * d.H // d.G + t["bcf"],
        "k_param_grads": d.B * d.H * d.nc * 12,
    }
    if name not in table:
        raise KeyError(name)
    return int(table[name])


def kernel_flops(name: str, d: Dims) -> int:
    """Algorithmic FLOPs (2 per multiply-add) of one launch of `name`."""
    tri = d.L * (d.L + 1)               # 2 x the causal (s <= l) pairs of a chunk
    if name in ("k_scan_tc", "k_scan_tc_dx"):
        return int(d.B * d.nc * d.G * tri * d.N + d.B * d.nc * d.H * (tri * d.P + 2 * d.L * d.N * d.P))
    if name in ("k_bwd_dc_tc", "k_bwd_db_tc"):
        return int(d.B * d.nc * d.G * tri * d.N
                   + d.B * d.nc * d.H * (tri * d.P + tri * d.N + 2 * d.L * d.P * d.N))
    per_chunk_head = {
        "k_state_tc": 2 * d.L * d.P * d.N,
        "k_dstates_tc": 2 * d.L * d.P * d.N,
        "k_chunk_state": 2 * d.L * d.P * d.N,
        "k_chunk_scan": tri * d.P + 2 * d.L * d.N * d.P,
        "k_dyx": tri * d.P,
        "k_bwd_dx": tri * d.P + 2 * d.L * d.N * d.P,
        "k_bwd_dC": tri * d.N + 2 * d.L * d.P * d.N,
        "k_bwd_dB": tri * d.N + 2 * d.L * d.P * d.N,
    }
    if name == "k_bmm_cb":
        return int(d.B * d.nc * d.G * tri * d.N)
    if name in per_chunk_head:
        return int(d.B * d.nc * d.H * per_chunk_head[name])
    raise KeyError(name)


def step_flops(d: Dims) -> int:
    """MMA FLOPs of one forward + backward of the chunked method (causal halves)."""
    bch = d.B * d.nc * d.H
    tri = d.L * (d.L + 1)               # 2 * (causal MACs per unit inner dim)
    fwd = d.B * d.nc * d.G * tri * d.N + bch * (2 * d.L * d.P * d.N + tri * d.P + 2 * d.L * d.N * d.P)
    # backward: recompute CB and S; dstates; dyx; dx (intra + state); dC, dB (intra + state)
    bwd = d.B * d.nc * d.G * tri * d.N + bch * (2 * d.L * d.P * d.N) * 2 + bch * tri * d.P
    bwd += bch * (tri * d.P + 2 * d.L * d.N * d.P)            # dx
    bwd += 2 * bch * (tri * d.N + 2 * d.L * d.P * d.N)        # dC, dB
    return int(fwd + bwd)


# ------------------------------------------------------------ gated norm
@dataclasses.dataclass
class NormDims:
    """rows = batch * seqlen, features = nheads * headdim; ib / ob bytes of an
    element of y, z, dout / of out, dy, dz."""
    rows: int
    features: int
    group_size: int
    ib: int = 2
    ob: int = 2


def norm_kernel_bytes(name: str, d: NormDims) -> int:
    """Algorithmic bytes of one launch: the forward reads y, z and writes out
    and rstd; the backward reads y, z, dout and the saved rstd and writes dy,
    dz (dw, one row of fp32, is counted where it is written)."""
    md = d.rows * d.features
    rs = d.rows * (d.features // d.group_size) * 4
    if name == "k_gated_norm_fwd":
        return md * (2 * d.ib + d.ob) + rs
    if name == "k_gated_norm_bwd":
        return md * (3 * d.ib + 2 * d.ob) + rs
    if name == "k_norm_dw_reduce":
        return d.features * 4
    raise KeyError(name)
