"""Chunked SSD algorithm in fp64 numpy -- TEST INFRASTRUCTURE (see ``oracle``).

The four steps of the chunked Mamba-2 scan as the pages name them
("Optimizing Mamba-2 kernels for the B200", Stage 1 kernel table:
_chunk_state_fwd, _state_passing_fwd, _chunk_scan_fwd; "Mamba-2 offers a
different scaling path": chunk_cumsum, fwd_pass_state, compute_out), each
written out plainly with numpy einsum as the only library step:

  chunk_cumsum   delta = softplus(dt + dt_bias) (0 on the padded tail),
                 a[l]  = sum_{r<=l} delta[r] * A[h]   inside each chunk
  chunk_state    S_c   = sum_l exp(a[L-1] - a[l]) delta[l] x_l (outer) B_l
  state_passing  H_0 = init, H_{c+1} = exp(a_c[L-1]) H_c + S_c
  chunk_scan     y_l   = sum_{s<=l} (C_l . B_s) exp(a_l - a_s) delta_s x_s
                         + exp(a_l) H_c C_l + D x_l

It also gives the chunked backward with the same decomposition (dstates,
state_passing backward, dx / dB / dC / ddA in the overflow-safe form that
only ever exponentiates a_l - a_s with s <= l).

Intermediate layouts match the CUDA library's workspace:
  delta, a : (B, H, nc, L);  S, Hprev : (B, nc, H, P, N)
"""
from __future__ import annotations

import numpy as np


def softplus(v):
    v = np.asarray(v, dtype=np.float64)
    return np.where(v > 20.0, v, np.log1p(np.exp(np.minimum(v, 20.0))))


def softplus_grad(v):
    v = np.asarray(v, dtype=np.float64)
    return np.where(v > 20.0, 1.0, 1.0 / (1.0 + np.exp(-np.minimum(v, 20.0))))


def _heads_to_groups(H, G):
    return np.arange(H) // (H // G)


def chunk_cumsum(dt, dt_bias, A, L):
    """Returns delta, a with shape (B, H, nc, L); padded positions get delta = 0."""
    Bt, T, H = dt.shape
    nc = -(-T // L)
    v = dt + (0.0 if dt_bias is None else dt_bias[None, None, :])
    delta = np.zeros((Bt, nc * L, H))
    delta[:, :T] = softplus(v)
    delta = delta.reshape(Bt, nc, L, H).transpose(0, 3, 1, 2)
    a = np.cumsum(delta * A[None, :, None, None], axis=-1)
    return delta, a


def _pad_chunks(arr, L):
    """(B, T, ...) -> (B, nc, L, ...) with zero padding of the tail."""
    Bt, T = arr.shape[:2]
    nc = -(-T // L)
    out = np.zeros((Bt, nc * L) + arr.shape[2:])
    out[:, :T] = arr
    return out.reshape((Bt, nc, L) + arr.shape[2:])


def chunk_state(x, B, delta, a, L):
    """S[b,c,h,p,n] = sum_l exp(a[L-1]-a[l]) delta[l] x[l,p] B[l,n]."""
    H = x.shape[2]
    G = B.shape[2]
    gh = _heads_to_groups(H, G)
    xc = _pad_chunks(x, L)                       # (B, nc, L, H, P)
    Bc = _pad_chunks(B, L)[:, :, :, gh, :]       # (B, nc, L, H, N)
    w = np.exp(a[..., -1:] - a) * delta          # (B, H, nc, L)
    return np.einsum("bhcl,bclhp,bclhn->bchpn", w, xc, Bc)


def state_passing(S, a, init=None):
    """Returns (Hprev, final): Hprev[:, c] is the state entering chunk c."""
    Bt, nc, H, P, N = S.shape
    Hprev = np.empty_like(S)
    cur = np.zeros((Bt, H, P, N)) if init is None else np.array(init, dtype=np.float64)
    decay = np.exp(a[..., -1])                    # (B, H, nc)
    for c in range(nc):
        Hprev[:, c] = cur
        cur = decay[:, :, c, None, None] * cur + S[:, c]
    return Hprev, cur


def chunk_scan(x, B, C, D, delta, a, Hprev, L):
    """y for every padded position, shape (B, nc*L, H, P)."""
    Bt, T, H, P = x.shape
    G = B.shape[2]
    gh = _heads_to_groups(H, G)
    xc = _pad_chunks(x, L)
    Bc = _pad_chunks(B, L)[:, :, :, gh, :]
    Cc = _pad_chunks(C, L)[:, :, :, gh, :]
    CB = np.einsum("bclhn,bcshn->bchls", Cc, Bc)
    seg = a[..., :, None] - a[..., None, :]      # (B, H, nc, L, L): a_l - a_s
    causal = np.tril(np.ones((L, L), dtype=bool))
    decay = np.where(causal, np.exp(np.where(causal, seg, 0.0)), 0.0)
    Wm = decay.transpose(0, 2, 1, 3, 4) * CB * delta.transpose(0, 2, 1, 3)[:, :, :, None, :]
    y = np.einsum("bchls,bcshp->bclhp", Wm, xc)
    y += np.exp(a).transpose(0, 2, 3, 1)[..., None] * np.einsum("bclhn,bchpn->bclhp", Cc, Hprev)
    if D is not None:
        y += D[None, None, None, :, None] * xc
    return y.reshape(Bt, -1, H, P)


def ssd_chunked_fwd(x, dt, dt_bias, A, B, C, D, init, L):
    """Chunked forward.  Returns y (B,T,H,P), final and the intermediates."""
    T = x.shape[1]
    delta, a = chunk_cumsum(dt, dt_bias, A, L)
    S = chunk_state(x, B, delta, a, L)
    Hprev, final = state_passing(S, a, init)
    y = chunk_scan(x, B, C, D, delta, a, Hprev, L)[:, :T]
    return dict(y=y, final=final, delta=delta, a=a, S=S, Hprev=Hprev)


def ssd_chunked_bwd(x, dt, dt_bias, A, B, C, D, init, dy, dfinal, L):
    """Chunked backward.  Returns the gradients plus the backward intermediates
    dHs (dstates), dS, dlast and ddA (gradient w.r.t. delta*A per position)."""
    Bt, T, H, P = x.shape
    G, N = B.shape[2], B.shape[3]
    gh = _heads_to_groups(H, G)
    f = ssd_chunked_fwd(x, dt, dt_bias, A, B, C, D, init, L)
    delta, a, Hprev = f["delta"], f["a"], f["Hprev"]
    nc = delta.shape[2]
    xc = _pad_chunks(x, L)                        # (B, nc, L, H, P)
    dyc = _pad_chunks(dy, L)
    Bc = _pad_chunks(B, L)[:, :, :, gh, :]        # (B, nc, L, H, N)
    Cc = _pad_chunks(C, L)[:, :, :, gh, :]
    aT = a.transpose(0, 2, 3, 1)                  # (B, nc, L, H)
    dT = delta.transpose(0, 2, 3, 1)
    ea = np.exp(aT)
    elast = np.exp(aT[:, :, -1:, :] - aT)         # exp(a[L-1] - a[l])

    # dstates: dHs_c = sum_l exp(a_l) dy_l (outer) C_l
    dHs = np.einsum("bclh,bclhp,bclhn->bchpn", ea, dyc, Cc)
    # state passing backward
    decay = np.exp(a[..., -1])                    # (B, H, nc)
    Gn = np.zeros((Bt, H, P, N)) if dfinal is None else np.array(dfinal, dtype=np.float64)
    dS = np.empty_like(dHs)
    dlast = np.empty((Bt, H, nc))
    for c in range(nc - 1, -1, -1):
        dS[:, c] = Gn
        dlast[:, :, c] = decay[:, :, c] * np.einsum("bhpn,bhpn->bh", Hprev[:, c], Gn)
        Gn = dHs[:, c] + decay[:, :, c, None, None] * Gn
    dinit = Gn

    causal = np.tril(np.ones((L, L), dtype=bool))
    seg = aT[:, :, :, None, :] - aT[:, :, None, :, :]          # (B,nc,L(l),L(s),H)
    W = np.where(causal[None, None, :, :, None], np.exp(np.where(causal[None, None, :, :, None], seg, 0.0)), 0.0)
    CB = np.einsum("bclhn,bcshn->bclsh", Cc, Bc)
    dyx = np.einsum("bclhp,bcshp->bclsh", dyc, xc)
    P2 = W * dT[:, :, None, :, :] * dyx                          # W delta_s <dy_l, x_s>
    M = CB * P2
    # dx
    u = np.einsum("bclsh,bclhp->bcshp", CB * W, dyc)             # intra part
    ustate = elast[..., None] * np.einsum("bcshn,bchpn->bcshp", Bc, dS)
    u = u + ustate
    dx = dT[..., None] * u + (0.0 if D is None else D[None, None, None, :, None]) * dyc
    ddelta = np.einsum("bcshp,bcshp->bcsh", xc, u)
    # dB, dC (per head, then summed over the heads of a group)
    dBh = np.einsum("bclsh,bclhn->bcshn", P2, Cc)
    dBh += (elast * dT)[..., None] * np.einsum("bcshp,bchpn->bcshn", xc, dS)
    dCh = np.einsum("bclsh,bcshn->bclhn", P2, Bc)
    dCstate = ea[..., None] * np.einsum("bclhp,bchpn->bclhn", dyc, Hprev)
    dCh += dCstate
    # ddA_r = sum_{l>=r, s<r} M[l,s] + sum_{l>=r} exp(a_l)<dy_l, H C_l>
    #         + sum_{s<r} Q_s + dlast,  Q_s = delta_s <x_s, ustate_s>
    Rex = np.cumsum(M, axis=3) - M                              # sum_{s<r} M[l, s], r = s index
    ddA = np.cumsum(Rex[:, :, ::-1], axis=2)[:, :, ::-1]        # sum over l >= r
    ddA = np.einsum("bclrh->bcrh", np.where(np.eye(L, dtype=bool)[None, None, :, :, None], ddA, 0.0))
    ycs = np.einsum("bclhn,bclhn->bclh", Cc, dCstate)           # exp(a_l)<dy_l, H C_l>
    ddA += np.cumsum(ycs[:, :, ::-1], axis=2)[:, :, ::-1]
    Q = dT * np.einsum("bcshp,bcshp->bcsh", xc, ustate)
    ddA += np.cumsum(Q, axis=2) - Q
    ddA += dlast.transpose(0, 2, 1)[:, :, None, :]
    ddelta += A[None, None, None, :] * ddA
    ddelta_t = ddelta.reshape(Bt, nc * L, H)[:, :T]
    v = dt + (0.0 if dt_bias is None else dt_bias[None, None, :])
    ddt = ddelta_t * softplus_grad(v)
    dA = np.einsum("bclh,bclh->h", dT, ddA)
    dB = np.zeros((Bt, nc * L, G, N))
    dC = np.zeros((Bt, nc * L, G, N))
    dBt = dBh.reshape(Bt, nc * L, H, N)
    dCt = dCh.reshape(Bt, nc * L, H, N)
    for g in range(G):
        dB[:, :, g] = dBt[:, :, gh == g].sum(axis=2)
        dC[:, :, g] = dCt[:, :, gh == g].sum(axis=2)
    dD = np.einsum("bthp,bthp->h", dy, x)
    return dict(dx=dx.reshape(Bt, nc * L, H, P)[:, :T], ddt=ddt, dA=dA, dB=dB[:, :T],
                dC=dC[:, :T], dD=dD, ddt_bias=ddt.sum(axis=(0, 1)), dinit=dinit,
                dHs=dHs, dS=dS, dlast=dlast, ddA=ddA.transpose(0, 3, 1, 2), fwd=f)
