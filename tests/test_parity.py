"""GPU parity: the CUDA path through the C ABI against the CPU oracle.

Small cases (several tiles, ragged tails, edge shapes) are compared element by
element, intermediates included; the full-size workloads are compared in full
(the oracle finishes them in seconds on the host cores).
"""
import numpy as np
import pytest

import oracle
from oracle import chunked
from parity_util import assert_close, stats, to_np
from state_space_model_sm_gb300.inputs import WORKLOADS, SSDShape, make_inputs, make_workload, to_torch

pytestmark = pytest.mark.gpu


def run_fwd(ssd, inp, out_dtype=None):
    import torch
    t = to_torch(inp)
    y, final = ssd.ssd_fwd(t["x"], t["dt"], t["dt_bias"], t["A"], t["B"], t["C"], t["D"],
                           chunk_size=inp.shape.chunk_size, init_states=t["init"],
                           out_dtype=out_dtype)
    torch.cuda.synchronize()
    assert ssd.device_status() == 0
    return y, final


def run_bwd(ssd, inp):
    import torch
    t = to_torch(inp)
    g = ssd.ssd_bwd(t["x"], t["dt"], t["dt_bias"], t["A"], t["B"], t["C"], t["D"],
                    inp.shape.chunk_size, t["init"], t["dy"], t["dfinal"])
    torch.cuda.synchronize()
    assert ssd.device_status() == 0
    return {k: to_np(v) for k, v in g.items()}


def oracle_fwd(inp):
    return oracle.ssd_fwd(*oracle.from_inputs(inp))


def oracle_bwd(inp):
    args = oracle.from_inputs(inp)
    return oracle.ssd_bwd(*args, np.asarray(inp.dy, np.float64),
                          None if inp.dfinal is None else np.asarray(inp.dfinal, np.float64))


SMALL = [
    # (name, shape, dtype, init_std)
    ("tiny_f32", SSDShape(1, 256, 4, 16, 16, 1, 64), "f32", 0.0),
    ("tail_f32", SSDShape(2, 250, 4, 16, 8, 2, 64), "f32", 0.5),
    ("odd_f32", SSDShape(1, 77, 3, 5, 7, 1, 16), "f32", 0.3),
    ("tail_bf16", SSDShape(2, 300, 4, 64, 128, 2, 128), "bf16", 0.1),
    ("multi_bf16", SSDShape(2, 1024, 8, 64, 128, 1, 256), "bf16", 0.0),
    ("g_eq_h_bf16", SSDShape(1, 512, 4, 64, 64, 4, 64), "bf16", 0.2),
    ("single_token", SSDShape(1, 1, 2, 16, 16, 1, 64), "f32", 0.5),
    ("chunk1_f32", SSDShape(1, 20, 2, 4, 4, 1, 1), "f32", 0.5),
]


@pytest.mark.parametrize("name,shape,dtype,init_std", SMALL, ids=[s[0] for s in SMALL])
def test_forward_small(cuda_lib, name, shape, dtype, init_std):
    inp = make_inputs(shape, seed=11, dtype=dtype, init_std=init_std)
    y, final = run_fwd(cuda_lib, inp)
    y_ref, f_ref = oracle_fwd(inp)
    assert_close("y", to_np(y), y_ref, dtype)
    assert_close("final", to_np(final), f_ref, dtype)


@pytest.mark.parametrize("name,shape,dtype,init_std", SMALL, ids=[s[0] for s in SMALL])
def test_backward_small(cuda_lib, name, shape, dtype, init_std):
    inp = make_inputs(shape, seed=12, dtype=dtype, init_std=init_std, with_dy=True,
                      dfinal_std=0.5)
    g = run_bwd(cuda_lib, inp)
    ref = oracle_bwd(inp)
    keys = ["dx", "ddt", "dA", "dB", "dC", "dD", "ddt_bias"]
    if inp.init is not None:
        keys.append("dinit")
    for k in keys:
        got = g["dinit_states"] if k == "dinit" else g[k]
        assert_close(k, got, ref[k], dtype)


@pytest.mark.parametrize("P", [64, 128])
def test_forward_intermediates_match_chunked_reference(cuda_lib, P):
    """Per-kernel parity: delta, dA_cumsum (chunk_cumsum), states (chunk_state)
    and hprev (state_passing), read from the documented workspace layout (at
    headdim 128 the tensor-core path writes delta / dA_cumsum once per head
    and a state image per 64-wide half of a head)."""
    import torch
    Bt, T, H, N, G, L = 2, 300, 4, 128, 2, 128
    inp = make_inputs(SSDShape(Bt, T, H, P, N, G, L), seed=5, dtype="bf16", init_std=0.1)
    t = to_torch(inp)
    nc = 3
    shape = cuda_lib.make_shape(Bt, T, H, P, N, G, L, cuda_lib.SSD_BF16, cuda_lib.SSD_F32)
    lay = cuda_lib.fwd_workspace_layout(shape)
    ws = torch.zeros(lay["total"], dtype=torch.uint8, device="cuda")
    cuda_lib.ssd_fwd(t["x"], t["dt"], t["dt_bias"], t["A"], t["B"], t["C"], t["D"],
                     chunk_size=L, init_states=t["init"], workspace=ws)
    torch.cuda.synchronize()

    def view(off, shp):
        n = int(np.prod(shp))
        return to_np(ws[off:off + 4 * n].view(torch.float32).reshape(shp))
    ref = chunked.ssd_chunked_fwd(*oracle.from_inputs(inp), L)
    s = stats(view(lay["delta"], (Bt, H, nc, L)), ref["delta"])
    assert s["rel_l2"] < 1e-6, s
    s = stats(view(lay["dA_cumsum"], (Bt, H, nc, L)), ref["a"])
    assert s["rel_l2"] < 1e-5, s
    s = stats(view(lay["states"], (Bt, nc, H, P, N)), ref["S"])
    assert s["rel_l2"] < 1e-3, s
    if cuda_lib.last_path() == 1:
        raw = ws[lay["hprev"]:lay["hprev"] + 4 * Bt * nc * H * P * N].cpu().numpy()
        hprev = decode_state_images(raw, Bt * nc * H * (P // 64), N).reshape(Bt, nc, H, P, N)
    else:
        hprev = view(lay["hprev"], (Bt, nc, H, P, N))
    s = stats(hprev, ref["Hprev"])
    assert s["rel_l2"] < 1e-3, s


def decode_state_images(raw, nstates, N):
    """Split-bf16 state images (hi panels, then lo panels; 64 rows of 128
    bytes; chunk j of row p at chunk j ^ (p % 8)) back to (nstates, 64, N)."""
    u16 = raw.view(np.uint16).reshape(nstates, 2, N // 64, 64, 64)
    f = (u16.astype(np.uint32) << 16).view(np.float32).astype(np.float64)
    tot = f[:, 0] + f[:, 1]                        # (nstates, panel, row, 64)
    out = np.empty((nstates, 64, N))
    for p in range(64):
        for j in range(8):
            src = j ^ (p & 7)
            for panel in range(N // 64):
                out[:, p, panel * 64 + 8 * j:panel * 64 + 8 * j + 8] = \
                    tot[:, panel, p, 8 * src:8 * src + 8]
    return out


def test_backward_is_deterministic(cuda_lib):
    inp = make_inputs(SSDShape(2, 512, 8, 64, 128, 2, 128), seed=3, dtype="bf16", with_dy=True)
    g1 = run_bwd(cuda_lib, inp)
    g2 = run_bwd(cuda_lib, inp)
    for k in g1:
        assert np.array_equal(g1[k], g2[k]), k


def test_bf16_output_mode(cuda_lib):
    import torch
    inp = make_inputs(SSDShape(2, 512, 8, 64, 128, 1, 256), seed=4, dtype="bf16")
    y, _ = run_fwd(cuda_lib, inp, out_dtype=torch.bfloat16)
    y_ref, _ = oracle_fwd(inp)
    s = stats(to_np(y), y_ref)
    assert s["page_ok"] and s["rel_l2"] < 1e-2, s


# ------------------------------------------------------------ full workloads

@pytest.mark.parametrize("name", ["tiny_f32", "layer_bf16", "hybrid_bf16", "long_bf16"])
def test_forward_workload(cuda_lib, name):
    inp = make_workload(name)
    y, final = run_fwd(cuda_lib, inp)
    y_ref, f_ref = oracle_fwd(inp)
    s = assert_close("y", to_np(y), y_ref, inp.dtype)
    assert_close("final", to_np(final), f_ref, inp.dtype)
    print(name, s)


@pytest.mark.parametrize("name", ["layer_fwdbwd_bf16", "layer_p128_fwdbwd_bf16"])
def test_forward_backward_workload(cuda_lib, name):
    inp = make_workload(name)
    y, final = run_fwd(cuda_lib, inp)
    y_ref, f_ref = oracle_fwd(inp)
    assert_close("y", to_np(y), y_ref, "bf16")
    g = run_bwd(cuda_lib, inp)
    ref = oracle_bwd(inp)
    for k in ["dx", "ddt", "dA", "dB", "dC", "dD", "ddt_bias"]:
        s = assert_close(k, g[k], ref[k], "bf16")
        print(k, s)


def test_forward_backward_hybrid_shape(cuda_lib):
    """The backward at the hybrid-model shape (batch 2, seqlen 8192, 64 heads in
    8 groups, chunk 128) with nonzero initial states and a final-state
    gradient: the group sums of dB / dC over 8 heads each and dinit."""
    shape, dtype, init_std, seed, _ = WORKLOADS["hybrid_bf16"]
    inp = make_inputs(shape, seed=seed + 100, dtype=dtype, init_std=init_std, with_dy=True,
                      dfinal_std=0.5)
    g = run_bwd(cuda_lib, inp)
    ref = oracle_bwd(inp)
    for k in ["dx", "ddt", "dA", "dB", "dC", "dD", "ddt_bias", "dinit"]:
        s = assert_close(k, g["dinit_states"] if k == "dinit" else g[k], ref[k], "bf16")
        print(k, s)


# ------------------------------------------------- tensor-core vs generic path

TC_CASES = [
    ("tc_n128_l256", SSDShape(2, 1024, 8, 64, 128, 1, 256), 0.0),
    ("tc_n128_l128_tail", SSDShape(2, 700, 8, 64, 128, 2, 128), 0.2),
    ("tc_n64_l128_tail", SSDShape(1, 333, 6, 64, 64, 3, 128), 0.1),
    ("tc_n64_l256", SSDShape(3, 512, 4, 64, 64, 1, 256), 0.0),
    ("tc_partial_second_tile", SSDShape(1, 300, 2, 64, 128, 1, 256), 0.0),
    # headdim 128: a head runs as two 64-wide parts sharing its dt / A / D
    ("tc_p128_n128_l256", SSDShape(2, 1024, 4, 128, 128, 1, 256), 0.2),
    ("tc_p128_n64_l128_tail", SSDShape(1, 333, 3, 128, 64, 3, 128), 0.1),
]


@pytest.mark.parametrize("name,shape,init_std", TC_CASES, ids=[c[0] for c in TC_CASES])
def test_tensor_core_forward_against_oracle_and_generic(cuda_lib, monkeypatch, name, shape,
                                                       init_std):
    inp = make_inputs(shape, seed=31, dtype="bf16", init_std=init_std)
    y, final = run_fwd(cuda_lib, inp)
    assert cuda_lib.last_path() == 1, "bf16 problem did not take the tcgen05 path"
    y_ref, f_ref = oracle_fwd(inp)
    s = assert_close("y", to_np(y), y_ref, "bf16")
    assert s["rel_l2"] < 1e-4, s      # split-bf16 operands keep ~fp32 accuracy
    assert_close("final", to_np(final), f_ref, "bf16")
    monkeypatch.setenv("SSD_FORCE_SIMT", "1")
    y2, f2 = run_fwd(cuda_lib, inp)
    assert cuda_lib.last_path() == 0
    s2 = stats(to_np(y), to_np(y2))
    assert s2["rel_l2"] < 1e-4, s2


def test_workloads_take_tensor_core_path(cuda_lib):
    for name in ("layer_bf16", "hybrid_bf16"):
        inp = make_workload(name)
        inp.x, inp.B = inp.x[:, :512], inp.B[:, :512]
        inp.C, inp.dt = inp.C[:, :512], inp.dt[:, :512]
        inp.shape = SSDShape(inp.shape.batch, 512, inp.shape.nheads, inp.shape.headdim,
                             inp.shape.dstate, inp.shape.ngroups, inp.shape.chunk_size)
        run_fwd(cuda_lib, inp)
        assert cuda_lib.last_path() == 1, name


TC_BWD_CASES = [
    ("tcb_n128_l256", SSDShape(2, 1024, 8, 64, 128, 1, 256), 0.0, 0.0),
    ("tcb_n128_l128_tail_init", SSDShape(2, 700, 8, 64, 128, 2, 128), 0.2, 0.5),
    ("tcb_n64_l128_tail", SSDShape(1, 333, 6, 64, 64, 3, 128), 0.1, 0.3),
    ("tcb_n64_l256_heads", SSDShape(2, 512, 12, 64, 64, 1, 256), 0.0, 0.0),
    ("tcb_partial_tile", SSDShape(1, 300, 2, 64, 128, 1, 256), 0.3, 0.2),
    ("tcb_p128_n128_l256_init", SSDShape(2, 1024, 4, 128, 128, 1, 256), 0.2, 0.5),
    ("tcb_p128_n64_l128_tail", SSDShape(1, 333, 3, 128, 64, 3, 128), 0.1, 0.3),
    # 2 x 64 heads x 4 blocks of 256 = 512 state-passing blocks, more than
    # three per SM hold in one wave: the walks run as 128-thread blocks
    ("tcb_wide_walk_tail_init", SSDShape(2, 333, 64, 64, 128, 8, 128), 0.2, 0.5),
    # one chunk shorter than its 128-row tile: every TMA load past seqlen
    # reads zeros and every dx / y store is clipped
    ("tcb_short_l128", SSDShape(1, 100, 2, 64, 64, 1, 128), 0.2, 0.3),
]


@pytest.mark.parametrize("name,shape,init_std,dfinal_std", TC_BWD_CASES,
                         ids=[c[0] for c in TC_BWD_CASES])
def test_tensor_core_backward_against_oracle_and_generic(cuda_lib, monkeypatch, name, shape,
                                                        init_std, dfinal_std):
    inp = make_inputs(shape, seed=41, dtype="bf16", init_std=init_std, with_dy=True,
                      dfinal_std=dfinal_std)
    g = run_bwd(cuda_lib, inp)
    assert cuda_lib.last_path() == 1
    ref = oracle_bwd(inp)
    keys = ["dx", "ddt", "dA", "dB", "dC", "dD", "ddt_bias"]
    for k in keys:
        s = assert_close(k, g[k], ref[k], "bf16")
        assert s["rel_l2"] < 1e-4, (k, s)
    if inp.init is not None:
        s = assert_close("dinit", g["dinit_states"], ref["dinit"], "bf16")
        assert s["rel_l2"] < 1e-4, s
    monkeypatch.setenv("SSD_FORCE_SIMT", "1")
    g2 = run_bwd(cuda_lib, inp)
    assert cuda_lib.last_path() == 0
    for k in keys:
        s = stats(g[k], g2[k])
        assert s["rel_l2"] < 1e-4, (k, s)


# ---------------------- optional inputs absent, steps past softplus's 20

OPT_CASES = [
    # tensor-core family (bf16, headdim 64) and generic family (fp32)
    ("opt_tc", SSDShape(1, 300, 4, 64, 128, 1, 128), "bf16", 1),
    ("opt_simt", SSDShape(2, 200, 4, 16, 16, 2, 64), "f32", 0),
]


@pytest.mark.parametrize("name,shape,dtype,path", OPT_CASES, ids=[c[0] for c in OPT_CASES])
def test_no_bias_no_skip_and_large_steps(cuda_lib, name, shape, dtype, path):
    """D = None and dt_bias = None (both optional in the ABI), with a few
    steps whose dt is above 20 so softplus takes its linear branch (delta = dt)
    on both sides; forward and backward against the oracle.  Those tokens'
    x is scaled by 1/21 so delta * x stays in the workload's range (the
    absolute bar is stated for that range; a step of 30 on N(0,1) inputs gives
    |y| in the thousands)."""
    from state_space_model_sm_gb300.inputs import round_to_bf16
    inp = make_inputs(shape, seed=51, dtype=dtype, init_std=0.2, with_dy=True, dfinal_std=0.3)
    inp.D = None
    inp.dt_bias = None
    pos = [0, shape.seqlen // 2, shape.seqlen - 1]
    dt = np.array(inp.dt)
    dt[:, pos, :] = np.array([20.5, 21.0, 21.5, 22.0][:shape.nheads])  # exact in bf16
    inp.dt = dt.astype(np.float32)
    x = np.array(inp.x)
    x[:, pos] = x[:, pos] / 21.0
    inp.x = round_to_bf16(x) if dtype == "bf16" else x.astype(np.float32)
    y, final = run_fwd(cuda_lib, inp)
    assert cuda_lib.last_path() == path
    y_ref, f_ref = oracle_fwd(inp)
    assert_close("y", to_np(y), y_ref, dtype)
    assert_close("final", to_np(final), f_ref, dtype)
    g = run_bwd(cuda_lib, inp)
    assert cuda_lib.last_path() == path
    ref = oracle_bwd(inp)
    for k in ["dx", "ddt", "dA", "dB", "dC", "dD", "dinit"]:
        got = g["dinit_states"] if k == "dinit" else g[k]
        assert_close(k, got, ref[k], dtype)


# ------------------------------------- two-level state passing (few heads)

SEG_CASES = [
    # (batch x heads) small and enough chunks: the chunks are split into
    # segments (8 of 4, 6 of 5 with a ragged last one, 2 with N = 64)
    ("seg_8x4", SSDShape(1, 4000, 2, 64, 128, 1, 128), 0.3),
    ("seg_ragged", SSDShape(1, 3800, 2, 64, 128, 1, 128), 0.3),
    ("seg_n64", SSDShape(1, 1100, 2, 64, 64, 1, 128), 0.3),
    # one head of headdim 128 (two 64-wide parts sharing its decay)
    ("seg_p128", SSDShape(1, 4000, 1, 128, 128, 1, 128), 0.3),
]


@pytest.mark.parametrize("name,shape,init_std", SEG_CASES, ids=[c[0] for c in SEG_CASES])
def test_two_level_state_passing(cuda_lib, name, shape, init_std):
    """Forward (y, final) and backward (whose recompute runs the same state
    passing) at shapes whose (batch, head) grid is small, with an initial
    state and a final-state gradient; the segment kernels must have run."""
    inp = make_inputs(shape, seed=41, dtype="bf16", init_std=init_std, with_dy=True,
                      dfinal_std=0.5)
    cuda_lib.profile_enable(True)
    y, final = run_fwd(cuda_lib, inp)
    g = run_bwd(cuda_lib, inp)
    prof = cuda_lib.profile_read()
    cuda_lib.profile_enable(False)
    assert prof.get("k_state_passing_seg", (0, 0))[1] == 4, prof  # 2 kernels, fwd + recompute
    assert prof.get("k_state_passing_bwd_seg", (0, 0))[1] == 2, prof
    y_ref, f_ref = oracle_fwd(inp)
    assert_close("y", to_np(y), y_ref, "bf16")
    assert_close("final", to_np(final), f_ref, "bf16")
    ref = oracle_bwd(inp)
    for k in ["dx", "ddt", "dA", "dB", "dC", "dD", "ddt_bias", "dinit"]:
        assert_close(k, g["dinit_states"] if k == "dinit" else g[k], ref[k], "bf16")
    assert cuda_lib.device_status() == 0


def test_two_level_backward_only(cuda_lib):
    """A (batch, head) grid of 128 blocks (32 heads): too many for a
    two-level forward (more than half the SMs), too few for the backward's
    longer walk, so only the backward's state passing is cut into segments."""
    inp = make_inputs(SSDShape(1, 2000, 32, 64, 128, 1, 256), seed=43, dtype="bf16",
                      init_std=0.3, with_dy=True, dfinal_std=0.5)
    cuda_lib.profile_enable(True)
    y, final = run_fwd(cuda_lib, inp)
    g = run_bwd(cuda_lib, inp)
    prof = cuda_lib.profile_read()
    cuda_lib.profile_enable(False)
    assert prof.get("k_state_passing_seg", (0, 0))[1] == 0, prof
    assert prof.get("k_state_passing_bwd_seg", (0, 0))[1] == 2, prof
    y_ref, f_ref = oracle_fwd(inp)
    assert_close("y", to_np(y), y_ref, "bf16")
    assert_close("final", to_np(final), f_ref, "bf16")
    ref = oracle_bwd(inp)
    for k in ["dx", "ddt", "dA", "dB", "dC", "dD", "ddt_bias", "dinit"]:
        assert_close(k, g["dinit_states"] if k == "dinit" else g[k], ref[k], "bf16")
    assert cuda_lib.device_status() == 0
