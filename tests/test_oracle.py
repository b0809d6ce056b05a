"""Pins for the CPU oracle (no GPU).

Each test checks the oracle against something other than itself: the
quadratic (masked-attention) dual form of the SSD, closed forms, invariants,
brute-force finite differences and torch autograd of the dual form.  The
pages print no worked example, so no pin comes from printed values.
"""
import numpy as np
import pytest

import oracle
from oracle import chunked
from state_space_model_sm_gb300.inputs import SSDShape, make_inputs


def rand_problem(Bt=2, T=37, H=4, P=3, N=5, G=2, seed=0, init=True, D=True):
    rng = np.random.default_rng(seed)
    x = rng.standard_normal((Bt, T, H, P))
    # steps of size ~0.3 with a strongly negative A so the decay matters
    dt = rng.normal(-1.0, 0.5, size=(Bt, T, H))
    dt_bias = rng.normal(0.0, 0.3, size=H)
    A = -np.exp(rng.uniform(0, np.log(4.0), size=H))
    Bm = rng.standard_normal((Bt, T, G, N))
    Cm = rng.standard_normal((Bt, T, G, N))
    Dv = rng.uniform(0, 1, size=H) if D else None
    init_s = rng.standard_normal((Bt, H, P, N)) * 0.5 if init else None
    return x, dt, dt_bias, A, Bm, Cm, Dv, init_s


def quadratic_form(x, dt, dt_bias, A, Bm, Cm, D, init):
    """Masked-attention (dual) form of the SSD, independent of the recurrence:
    y_t = sum_{s<=t} (C_t.B_s) exp(A sum_{r=s+1..t} delta_r) delta_s x_s
          + exp(A sum_{r<=t} delta_r) (init C_t) + D x_t."""
    Bt, T, H, P = x.shape
    G, N = Bm.shape[2], Bm.shape[3]
    gh = np.arange(H) // (H // G)
    v = dt + dt_bias[None, None, :]
    delta = np.log1p(np.exp(v))
    cs = np.cumsum(delta * A[None, None, :], axis=1)          # (B, T, H)
    Bh, Ch = Bm[:, :, gh, :], Cm[:, :, gh, :]                  # (B, T, H, N)
    y = np.zeros_like(x)
    final = np.zeros((Bt, H, P, N))
    for b in range(Bt):
        for h in range(H):
            CB = Ch[b, :, h, :] @ Bh[b, :, h, :].T              # (T, T)
            seg = cs[b, :, h][:, None] - cs[b, :, h][None, :]
            mask = np.tril(np.ones((T, T), dtype=bool))
            Lm = np.where(mask, np.exp(np.where(mask, seg, 0.0)), 0.0)
            y[b, :, h, :] = (CB * Lm * delta[b, :, h][None, :]) @ x[b, :, h, :]
            w_end = np.exp(cs[b, -1, h] - cs[b, :, h]) * delta[b, :, h]
            final[b, h] = (x[b, :, h, :] * w_end[:, None]).T @ Bh[b, :, h, :]
            if init is not None:
                y[b, :, h, :] += np.exp(cs[b, :, h])[:, None] * (Ch[b, :, h, :] @ init[b, h].T)
                final[b, h] += np.exp(cs[b, -1, h]) * init[b, h]
            if D is not None:
                y[b, :, h, :] += D[h] * x[b, :, h, :]
    return y, final


def close(a, b, rtol=1e-11):
    a, b = np.asarray(a), np.asarray(b)
    scale = max(np.abs(b).max(), 1e-300)
    return np.abs(a - b).max() <= rtol * scale


# ---------------------------------------------------------------- forward pins

@pytest.mark.parametrize("G,init,D", [(1, True, True), (2, True, False), (4, False, True)])
def test_forward_matches_quadratic_dual_form(G, init, D):
    args = rand_problem(G=G, init=init, D=D)
    y, final = oracle.ssd_fwd(*args)
    yq, fq = quadratic_form(*args)
    assert close(y, yq) and close(final, fq)


def test_forward_A_zero_is_prefix_sum():
    x, dt, dt_bias, A, Bm, Cm, D, init = rand_problem(G=1)
    A = np.zeros_like(A)
    y, final = oracle.ssd_fwd(x, dt, dt_bias, A, Bm, Cm, D, init)
    delta = np.log1p(np.exp(dt + dt_bias))
    upd = np.einsum("bth,bthp,btn->bthpn", delta, x, Bm[:, :, 0, :])
    h = init[:, None] + np.cumsum(upd, axis=1)                   # (B, T, H, P, N)
    y_ref = np.einsum("bthpn,btn->bthp", h, Cm[:, :, 0, :]) + D[None, None, :, None] * x
    assert close(y, y_ref) and close(final, h[:, -1])


@pytest.mark.parametrize("dt_raw,Aval", [(-1.0, -2.0), (0.5, -0.3), (-3.0, -16.0)])
def test_forward_constant_input_geometric_series(dt_raw, Aval):
    T = 50
    x = np.ones((1, T, 1, 1))
    Bm = np.ones((1, T, 1, 1))
    Cm = np.ones((1, T, 1, 1))
    dt = np.full((1, T, 1), dt_raw)
    D = np.array([0.25])
    y, final = oracle.ssd_fwd(x, dt, np.zeros(1), np.array([Aval]), Bm, Cm, D, None)
    delta = np.log(1.0 + np.exp(dt_raw))
    r = np.exp(delta * Aval)
    t = np.arange(T)
    h = delta * (1.0 - r ** (t + 1)) / (1.0 - r)
    assert close(y[0, :, 0, 0], h + 0.25) and close(final.ravel(), h[-1:])


def test_forward_single_token_by_hand():
    x, dt, dt_bias, A, Bm, Cm, D, init = rand_problem(Bt=1, T=1, H=2, P=3, N=4, G=1)
    y, final = oracle.ssd_fwd(x, dt, dt_bias, A, Bm, Cm, D, init)
    for h in range(2):
        delta = np.log1p(np.exp(dt[0, 0, h] + dt_bias[h]))
        alpha = np.exp(delta * A[h])
        B0, C0 = Bm[0, 0, 0], Cm[0, 0, 0]
        hs = alpha * init[0, h] + delta * np.outer(x[0, 0, h], B0)
        assert close(final[0, h], hs)
        yh = delta * (C0 @ B0) * x[0, 0, h] + D[h] * x[0, 0, h] + alpha * (init[0, h] @ C0)
        assert close(y[0, 0, h], yh)


def test_softplus_linear_branch_above_20():
    """softplus(v) = v exactly for v > 20, log1p(exp(v)) at and below (the
    convention both sides share).  One token with N = P = 1, x = B = C = 1,
    D = 0 and no initial state gives y = final = delta, and with dy = 1 the
    gradient ddt = softplus'(v): exactly 1 above 20, sigmoid(v) below.  At
    v = 25 the two branches differ by 1.4e-11 (delta) and 1.4e-11 (slope), at
    v = 19 by 5.6e-9, so a threshold on the wrong side of either value fails."""
    v = np.array([25.0, 19.0, 20.0])
    x = np.ones((1, 1, 3, 1))
    dt = v.reshape(1, 1, 3)
    dt_bias = np.zeros(3)
    A = -np.ones(3)
    Bm = np.ones((1, 1, 1, 1))
    Cm = np.ones((1, 1, 1, 1))
    y, final = oracle.ssd_fwd(x, dt, dt_bias, A, Bm, Cm, np.zeros(3), None)
    expect = np.array([25.0, np.log1p(np.exp(19.0)), np.log1p(np.exp(20.0))])
    assert y[0, 0, 0, 0] == 25.0                       # linear branch, exactly
    assert abs(y[0, 0, 1, 0] - expect[1]) < 1e-15 * expect[1] and y[0, 0, 1, 0] != 19.0
    assert abs(y[0, 0, 2, 0] - expect[2]) < 1e-15 * expect[2]
    assert np.array_equal(final.reshape(3), y.reshape(3))
    g = oracle.ssd_bwd(x, dt, dt_bias, A, Bm, Cm, np.zeros(3), None, np.ones((1, 1, 3, 1)))
    assert g["ddt"][0, 0, 0] == 1.0                    # slope of the linear branch
    sig = 1.0 / (1.0 + np.exp(-np.array([19.0, 20.0])))
    assert np.allclose(g["ddt"][0, 0, 1:], sig, rtol=1e-15, atol=0)
    assert g["ddt"][0, 0, 1] != 1.0
    # the chunked numpy oracle uses the same convention
    assert chunked.softplus(25.0) == 25.0 and chunked.softplus_grad(25.0) == 1.0
    assert chunked.softplus(19.0) == np.log1p(np.exp(19.0))
    assert chunked.softplus_grad(19.0) == sig[0]


def test_forward_initial_state_only():
    x, dt, dt_bias, A, Bm, Cm, D, init = rand_problem(G=2)
    x = np.zeros_like(x)
    y, final = oracle.ssd_fwd(x, dt, dt_bias, A, Bm, Cm, D, init)
    delta = np.log1p(np.exp(dt + dt_bias))
    cs = np.cumsum(delta * A, axis=1)                            # (B, T, H)
    gh = np.arange(4) // 2
    y_ref = np.exp(cs)[..., None] * np.einsum("bhpn,bthn->bthp", init, Cm[:, :, gh, :])
    assert close(y, y_ref)
    assert close(final, np.exp(cs[:, -1])[:, :, None, None] * init)


def test_forward_split_and_resume():
    args = rand_problem(T=41)
    x, dt, dt_bias, A, Bm, Cm, D, init = args
    y, final = oracle.ssd_fwd(*args)
    T1 = 17
    y1, f1 = oracle.ssd_fwd(x[:, :T1], dt[:, :T1], dt_bias, A, Bm[:, :T1], Cm[:, :T1], D, init)
    y2, f2 = oracle.ssd_fwd(x[:, T1:], dt[:, T1:], dt_bias, A, Bm[:, T1:], Cm[:, T1:], D, f1)
    assert close(np.concatenate([y1, y2], axis=1), y, 1e-12) and close(f2, final, 1e-12)


def test_forward_linear_in_x():
    x, dt, dt_bias, A, Bm, Cm, D, _ = rand_problem()
    x2 = np.random.default_rng(5).standard_normal(x.shape)
    ya, _ = oracle.ssd_fwd(x, dt, dt_bias, A, Bm, Cm, D, None)
    yb, _ = oracle.ssd_fwd(x2, dt, dt_bias, A, Bm, Cm, D, None)
    yc, _ = oracle.ssd_fwd(2.0 * x - 3.0 * x2, dt, dt_bias, A, Bm, Cm, D, None)
    assert close(yc, 2.0 * ya - 3.0 * yb)


def test_forward_head_and_batch_permutation():
    x, dt, dt_bias, A, Bm, Cm, D, init = rand_problem(G=1)
    y, final = oracle.ssd_fwd(x, dt, dt_bias, A, Bm, Cm, D, init)
    hp, bp = np.array([2, 0, 3, 1]), np.array([1, 0])
    y2, f2 = oracle.ssd_fwd(x[bp][:, :, hp], dt[bp][:, :, hp], dt_bias[hp], A[hp], Bm[bp],
                            Cm[bp], D[hp], init[bp][:, hp])
    assert close(y2, y[bp][:, :, hp], 1e-14) and close(f2, final[bp][:, hp], 1e-14)


def test_forward_groups_replicated_equal_single_group():
    x, dt, dt_bias, A, Bm, Cm, D, init = rand_problem(G=1)
    y1, f1 = oracle.ssd_fwd(x, dt, dt_bias, A, Bm, Cm, D, init)
    Brep, Crep = np.repeat(Bm, 4, axis=2), np.repeat(Cm, 4, axis=2)
    y4, f4 = oracle.ssd_fwd(x, dt, dt_bias, A, Brep, Crep, D, init)
    assert close(y4, y1, 1e-14) and close(f4, f1, 1e-14)


def test_forward_large_negative_cumsum_does_not_overflow():
    # The in-chunk cumulative decay reaches ~ -410 on the workloads; make it far larger.
    x, dt, dt_bias, A, Bm, Cm, D, init = rand_problem(T=300, G=1)
    A = np.full_like(A, -16.0)
    dt = np.full_like(dt, 1.5)
    y, final = oracle.ssd_fwd(x, dt, dt_bias, A, Bm, Cm, D, init)
    assert np.isfinite(y).all() and np.isfinite(final).all()
    out = chunked.ssd_chunked_fwd(x, dt, dt_bias, A, Bm, Cm, D, init, 128)
    assert close(out["y"], y, 1e-10)


# --------------------------------------------------------- chunked algorithm

@pytest.mark.parametrize("L", [1, 2, 7, 16, 64, 100])
def test_chunked_forward_chunk_size_invariance(L):
    args = rand_problem(T=100)
    y, final = oracle.ssd_fwd(*args)
    out = chunked.ssd_chunked_fwd(*args, L)
    assert close(out["y"], y) and close(out["final"], final)


@pytest.mark.parametrize("L", [1, 7, 16, 100])
def test_chunked_backward_matches_oracle(L):
    args = rand_problem(T=100)
    dy = np.random.default_rng(9).standard_normal(args[0].shape)
    dfinal = np.random.default_rng(10).standard_normal(args[-1].shape)
    ref = oracle.ssd_bwd(*args, dy, dfinal)
    got = chunked.ssd_chunked_bwd(*args, dy, dfinal, L)
    for k in ("dx", "ddt", "dA", "dB", "dC", "dD", "ddt_bias", "dinit"):
        assert close(got[k], ref[k], 1e-10), k


# ------------------------------------ the chunked oracle's own intermediates
# Each intermediate of the chunked algorithm is the answer to a smaller
# question the sequential recurrence (the C++ oracle) answers on its own:
# the states on a prefix or on one chunk, gradients of a suffix.

def _slice(args, t0, t1, init):
    x, dt, dt_bias, A, Bm, Cm, D, _ = args
    return (x[:, t0:t1], dt[:, t0:t1], dt_bias, A, Bm[:, t0:t1], Cm[:, t0:t1], D, init)


@pytest.mark.parametrize("L", [16, 32])
def test_chunked_states_are_recurrence_states(L):
    """Hprev[c] is the recurrence's state after the prefix [0, cL); S_c its
    state after chunk c alone from a zero start; e^{a_c[L-1]} the decay a
    chunk applies to the state entering it (a run with x = 0 from init = 1);
    delta is softplus(dt + dt_bias) with zeros past seqlen."""
    args = rand_problem(T=100, P=5, N=7)
    x, dt, dt_bias, A, Bm, Cm, D, init = args
    T, H = x.shape[1], x.shape[2]
    f = chunked.ssd_chunked_fwd(*args, L)
    nc = f["S"].shape[1]
    for c in range(nc):
        t0, t1 = c * L, min(T, (c + 1) * L)
        want = init if c == 0 else oracle.ssd_fwd(*_slice(args, 0, t0, init))[1]
        assert close(f["Hprev"][:, c], want, 1e-10), c
        zero = np.zeros_like(init)
        assert close(f["S"][:, c], oracle.ssd_fwd(*_slice(args, t0, t1, zero))[1], 1e-10), c
        ones = np.ones_like(init)
        sl = list(_slice(args, t0, t1, ones))
        sl[0] = np.zeros_like(sl[0])
        decay = oracle.ssd_fwd(*sl)[1][:, :, 0, 0]               # (B, H)
        assert close(np.exp(f["a"][:, :, c, -1]), decay, 1e-12), c
    v = dt + dt_bias[None, None, :]
    want_delta = np.log1p(np.exp(v)).transpose(0, 2, 1)          # (B, H, T)
    got = f["delta"].reshape(x.shape[0], H, -1)
    assert close(got[:, :, :T], want_delta, 1e-14)
    assert np.all(got[:, :, T:] == 0.0)


@pytest.mark.parametrize("L", [16, 32])
def test_chunked_backward_intermediates_are_recurrence_gradients(L):
    """dS_c (the gradient entering chunk c from later chunks) is the
    recurrence's dinit of the suffix from chunk c + 1 on (dfinal at the last
    chunk); dHs_c is the dinit of chunk c alone with no dfinal."""
    args = rand_problem(T=100, P=5, N=7, seed=3)
    x, dt, dt_bias, A, Bm, Cm, D, init = args
    T = x.shape[1]
    rng = np.random.default_rng(11)
    dy = rng.standard_normal(x.shape)
    dfinal = rng.standard_normal(init.shape)
    g = chunked.ssd_chunked_bwd(*args, dy, dfinal, L)
    Hprev = g["fwd"]["Hprev"]
    nc = Hprev.shape[1]
    for c in range(nc):
        t0, t1 = c * L, min(T, (c + 1) * L)
        if c == nc - 1:
            want = dfinal
        else:
            want = oracle.ssd_bwd(*_slice(args, t1, T, Hprev[:, c + 1]), dy[:, t1:], dfinal)["dinit"]
        assert close(g["dS"][:, c], want, 1e-10), c
        own = oracle.ssd_bwd(*_slice(args, t0, t1, Hprev[:, c]), dy[:, t0:t1], None)["dinit"]
        assert close(g["dHs"][:, c], own, 1e-10), c


def test_chunked_ddA_from_the_recurrence_gradients():
    """The per-position gradient w.r.t. delta_r A that the chunked backward
    forms through its "stable" sums follows from the recurrence's own
    gradients by the chain rule of delta_r = softplus(dt_r + dt_bias):
    ddt_r = (<x_r, u_r> + A ddA_r) softplus'(v_r), with u_r = (dx_r - D dy_r) /
    delta_r (dx_r = delta_r u_r + D dy_r)."""
    args = rand_problem(T=70, P=5, N=7, seed=5)
    x, dt, dt_bias, A, Bm, Cm, D, init = args
    Bt, T, H, _ = x.shape
    rng = np.random.default_rng(12)
    dy = rng.standard_normal(x.shape)
    dfinal = rng.standard_normal(init.shape)
    L = 16
    g = chunked.ssd_chunked_bwd(*args, dy, dfinal, L)
    ref = oracle.ssd_bwd(*args, dy, dfinal)
    v = dt + dt_bias[None, None, :]
    delta = np.log1p(np.exp(v))
    sig = 1.0 / (1.0 + np.exp(-v))
    u = (ref["dx"] - D[None, None, :, None] * dy) / delta[..., None]
    want = (ref["ddt"] / sig - np.einsum("bthp,bthp->bth", x, u)) / A[None, None, :]
    got = g["ddA"].reshape(Bt, H, -1)[:, :, :T].transpose(0, 2, 1)
    assert close(got, want, 1e-8)


# ------------------------------------------------------------- backward pins

def _loss(args, dy, dfinal):
    y, final = oracle.ssd_fwd(*args)
    return float(np.sum(y * dy) + np.sum(final * dfinal))


@pytest.mark.parametrize("G", [1, 2])
def test_backward_matches_central_finite_differences(G):
    args = list(rand_problem(Bt=2, T=9, H=2, P=2, N=3, G=G, seed=3))
    rng = np.random.default_rng(4)
    dy = rng.standard_normal(args[0].shape)
    dfinal = rng.standard_normal(args[7].shape)
    g = oracle.ssd_bwd(*args, dy, dfinal)
    names = ["x", "dt", "dt_bias", "A", "B", "C", "D", "init"]
    gnames = ["dx", "ddt", "ddt_bias", "dA", "dB", "dC", "dD", "dinit"]
    eps = 1e-6
    for i, (nm, gn) in enumerate(zip(names, gnames)):
        base = args[i]
        fd = np.zeros_like(base)
        for idx in np.ndindex(base.shape):
            plus = [a.copy() if j == i else a for j, a in enumerate(args)]
            minus = [a.copy() if j == i else a for j, a in enumerate(args)]
            plus[i][idx] += eps
            minus[i][idx] -= eps
            fd[idx] = (_loss(plus, dy, dfinal) - _loss(minus, dy, dfinal)) / (2 * eps)
        err = np.abs(fd - g[gn]).max() / max(np.abs(fd).max(), 1e-12)
        assert err < 1e-6, (nm, err)


def test_backward_dD_closed_form():
    args = rand_problem()
    dy = np.random.default_rng(1).standard_normal(args[0].shape)
    g = oracle.ssd_bwd(*args, dy, None)
    assert close(g["dD"], np.einsum("bthp,bthp->h", dy, args[0]))


def test_backward_matches_torch_autograd_of_dual_form():
    torch = pytest.importorskip("torch")
    x, dt, dt_bias, A, Bm, Cm, D, init = rand_problem(Bt=2, T=23, H=4, P=3, N=5, G=2, seed=7)
    rng = np.random.default_rng(8)
    dy = rng.standard_normal(x.shape)
    dfinal = rng.standard_normal(init.shape)
    g = oracle.ssd_bwd(x, dt, dt_bias, A, Bm, Cm, D, init, dy, dfinal)

    tx, tdt, tbias, tA, tB, tC, tD, tinit = (torch.tensor(a, dtype=torch.float64, requires_grad=True)
                                             for a in (x, dt, dt_bias, A, Bm, Cm, D, init))
    Bt, T, H, P = x.shape
    gh = torch.arange(H) // 2
    delta = torch.nn.functional.softplus(tdt + tbias)
    cs = torch.cumsum(delta * tA, dim=1)                           # (B, T, H)
    Bh, Ch = tB[:, :, gh, :], tC[:, :, gh, :]
    CB = torch.einsum("bthn,bshn->bhts", Ch, Bh)
    seg = cs.permute(0, 2, 1)[..., :, None] - cs.permute(0, 2, 1)[..., None, :]
    mask = torch.tril(torch.ones(T, T, dtype=torch.bool))
    Lm = torch.where(mask, torch.exp(torch.where(mask, seg, torch.zeros_like(seg))),
                     torch.zeros_like(seg))
    W = CB * Lm * delta.permute(0, 2, 1)[:, :, None, :]
    y = torch.einsum("bhts,bshp->bthp", W, tx)
    y = y + torch.exp(cs)[..., None] * torch.einsum("bhpn,bthn->bthp", tinit, Ch)
    y = y + tD[None, None, :, None] * tx
    w_end = torch.exp(cs[:, -1:, :] - cs) * delta                  # (B, T, H)
    final = torch.einsum("bth,bthp,bthn->bhpn", w_end, tx, Bh)
    final = final + torch.exp(cs[:, -1])[:, :, None, None] * tinit
    loss = (y * torch.tensor(dy)).sum() + (final * torch.tensor(dfinal)).sum()
    loss.backward()
    for t, k in ((tx, "dx"), (tdt, "ddt"), (tbias, "ddt_bias"), (tA, "dA"), (tB, "dB"),
                 (tC, "dC"), (tD, "dD"), (tinit, "dinit")):
        assert close(g[k], t.grad.numpy(), 1e-10), k


# ------------------------------------------------------- workload generator

def test_inputs_are_bf16_representable_and_dt_in_range():
    inp = make_inputs(SSDShape(1, 64, 4, 8, 8, 1, 64), seed=0, dtype="bf16", with_dy=True)
    for a in (inp.x, inp.dt, inp.B, inp.C, inp.dy):
        assert (a.view(np.uint32) & 0xFFFF == 0).all()
    delta = np.log1p(np.exp(inp.dt.astype(np.float64) + inp.dt_bias))
    assert delta.min() > 0.9e-3 and delta.max() < 1.1e-1
    assert (inp.A < 0).all() and (inp.A >= -16.0).all()


def test_golden_tiny_workload():
    """Regression fixture written by tests/golden/make_golden.py (oracle only)."""
    import json
    import os
    path = os.path.join(os.path.dirname(__file__), "golden", "tiny_f32_oracle.json")
    gold = json.load(open(path))
    inp = make_inputs(SSDShape(1, 256, 4, 16, 16, 1, 64), seed=0, dtype="f32")
    y, final = oracle.ssd_fwd(*oracle.from_inputs(inp))
    for k, v in gold["y_samples"].items():
        t, h, p = map(int, k.split(","))
        assert abs(y[0, t, h, p] - v) <= 1e-12 * max(1.0, abs(v))
    assert abs(float(np.sum(y)) - gold["y_sum"]) <= 1e-9 * max(1.0, abs(gold["y_sum"]))
    assert abs(float(np.sum(final ** 2)) - gold["final_sq"]) <= 1e-9 * gold["final_sq"]


def test_random_shapes_recurrence_dual_and_chunked_agree():
    """Property check over random small shapes, group counts, chunk sizes,
    with and without init / D: the recurrence oracle equals the quadratic
    dual form (forward) and the chunked algorithm (forward and backward)."""
    hyp = pytest.importorskip("hypothesis")
    st = pytest.importorskip("hypothesis.strategies")

    @hyp.settings(max_examples=25, deadline=None, derandomize=True)
    @hyp.given(Bt=st.integers(1, 2), T=st.integers(1, 40), hg=st.sampled_from([(1, 1), (2, 1),
                                                                              (4, 2), (4, 4)]),
               P=st.integers(1, 4), N=st.integers(1, 5), L=st.integers(1, 48),
               init=st.booleans(), D=st.booleans(), seed=st.integers(0, 2 ** 16))
    def check(Bt, T, hg, P, N, L, init, D, seed):
        H, G = hg
        args = rand_problem(Bt=Bt, T=T, H=H, P=P, N=N, G=G, seed=seed, init=init, D=D)
        y, final = oracle.ssd_fwd(*args)
        yq, fq = quadratic_form(*args)
        assert close(y, yq) and close(final, fq)
        out = chunked.ssd_chunked_fwd(*args, L)
        assert close(out["y"], y) and close(out["final"], final)
        rng = np.random.default_rng(seed + 1)
        dy = rng.standard_normal(args[0].shape)
        dfinal = rng.standard_normal((Bt, H, P, N))
        ref = oracle.ssd_bwd(*args, dy, dfinal)
        got = chunked.ssd_chunked_bwd(*args, dy, dfinal, L)
        keys = ["dx", "ddt", "dA", "dB", "dC", "ddt_bias"] + (["dD"] if D else []) + \
            (["dinit"] if init else [])
        for k in keys:
            assert close(got[k], ref[k], 1e-9), k
    check()
