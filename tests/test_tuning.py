"""The launch tables of the gated-norm and the SSD chunk kernels: validation,
the per-shape tables inside the library (set / get / remove through the C
ABI, host-only calls that need no GPU), the packaged tables, and on the GPU
that a tuned launch computes the same result as the built-in one."""
import json
import os

import numpy as np
import pytest

from state_space_model_sm_gb300 import tuning


def _entry(**kw):
    e = dict(features=4096, group_size=512, in_dtype="bf16", out_dtype="bf16", rows_per_item=1,
             ring_kb=64, ctas_per_sm=2)
    e.update(kw)
    return e


def _table(*entries):
    return {"kind": tuning.TABLE_KIND, "entries": list(entries)}


def test_validate_accepts_a_good_table():
    tuning.validate_table(_table(_entry(), _entry(features=1536, group_size=1536,
                                                  rows_per_item=2)))


@pytest.mark.parametrize("bad", [
    dict(rows_per_item=2),                  # 2 x 512 threads: more than a CTA
    dict(features=1536, group_size=1536, rows_per_item=3),  # 576 threads
    dict(features=64, group_size=16, rows_per_item=3),      # 24 threads: not whole warps
    dict(ring_kb=4), dict(ring_kb=300), dict(ctas_per_sm=9), dict(ctas_per_sm=-1),
    dict(group_size=500), dict(in_dtype="fp16"),
])
def test_validate_rejects(bad):
    with pytest.raises(ValueError):
        tuning.validate_table(_table(_entry(**bad)))


def test_validate_rejects_duplicates_and_wrong_kind():
    with pytest.raises(ValueError):
        tuning.validate_table(_table(_entry(), _entry()))
    with pytest.raises(ValueError):
        tuning.validate_table({"kind": "other", "entries": []})


def test_library_table_set_get_remove():
    F, G = 2048, 256
    tuning.clear_norm_config(F, G)
    cfg, from_table = tuning.get_norm_config(F, G)
    assert not from_table and cfg["rows_per_item"] == 512 // (F // 8)
    tuning.set_norm_config(F, G, rows_per_item=1, ring_kb=48, ctas_per_sm=3)
    cfg, from_table = tuning.get_norm_config(F, G)
    assert from_table and cfg == dict(rows_per_item=1, ring_kb=48, ctas_per_sm=3)
    # a zero field keeps the built-in choice
    tuning.set_norm_config(F, G, ring_kb=40)
    cfg, _ = tuning.get_norm_config(F, G)
    assert cfg["rows_per_item"] == 2 and cfg["ring_kb"] == 40
    # other dtypes are other entries
    assert not tuning.get_norm_config(F, G, "f32")[1]
    tuning.clear_norm_config(F, G)
    assert not tuning.get_norm_config(F, G)[1]


@pytest.mark.parametrize("kw", [dict(rows_per_item=3), dict(ring_kb=201), dict(ctas_per_sm=9)])
def test_library_rejects_invalid_fields(kw):
    with pytest.raises(ValueError):
        tuning.set_norm_config(2048, 256, **kw)


def test_table_file_roundtrip_and_apply(tmp_path):
    t = _table(_entry(features=1024, group_size=128, rows_per_item=4, ring_kb=32, ctas_per_sm=1))
    p = tmp_path / "t.json"
    p.write_text(json.dumps(t))
    assert tuning.apply_table(json.loads(p.read_text())) == 1
    cfg, from_table = tuning.get_norm_config(1024, 128)
    assert from_table and cfg == dict(rows_per_item=4, ring_kb=32, ctas_per_sm=1)
    tuning.clear_norm_config(1024, 128)


def test_default_table_env_control(tmp_path, monkeypatch):
    monkeypatch.setenv("SSD_TUNING_TABLE", "none")
    assert tuning.apply_default(None) is None
    p = tmp_path / "t.json"
    p.write_text(json.dumps(_table(_entry(features=512, group_size=64, rows_per_item=2))))
    monkeypatch.setenv("SSD_TUNING_TABLE", str(p))
    assert tuning.apply_default(tuning._native.load()) == str(p)
    assert tuning.get_norm_config(512, 64)[1]
    tuning.clear_norm_config(512, 64)


def test_packaged_table_is_valid_and_loaded():
    if not os.path.exists(tuning.DEFAULT_TABLE):
        pytest.skip("no packaged table")
    with open(tuning.DEFAULT_TABLE) as f:
        t = json.load(f)
    tuning.validate_table(t)
    assert t.get("generated_by", "").startswith("python -m state_space_model_sm_gb300.tuning")
    if os.environ.get("SSD_TUNING_TABLE", tuning.DEFAULT_TABLE) == tuning.DEFAULT_TABLE:
        for e in t["entries"]:
            cfg, from_table = tuning.get_norm_config(e["features"], e["group_size"],
                                                     e["in_dtype"], e["out_dtype"])
            assert from_table
            assert cfg["ring_kb"] == e["ring_kb"] and cfg["ctas_per_sm"] == e["ctas_per_sm"]


@pytest.mark.gpu
@pytest.mark.parametrize("F,G,cfg", [
    (4096, 512, dict(rows_per_item=1, ring_kb=32, ctas_per_sm=1)),
    (1536, 1536, dict(rows_per_item=1, ring_kb=48, ctas_per_sm=3)),
    (256, 64, dict(rows_per_item=4, ring_kb=16, ctas_per_sm=4)),
])
def test_tuned_launch_computes_the_same(cuda_lib, F, G, cfg):
    """Every row is computed by the same per-thread arithmetic whatever the
    launch, so out, rstd, dy and dz are bit-identical; dw is summed over a
    different CTA partition, equal to rounding."""
    import torch
    rows = 777
    g = torch.Generator().manual_seed(F + G)
    y, z, dout = (torch.randn(rows, F, generator=g).to("cuda", torch.bfloat16) for _ in range(3))
    w = (1.0 + 0.1 * torch.randn(F, generator=g)).cuda()
    saved, had = tuning.get_norm_config(F, G)

    def run():
        out, rstd = cuda_lib.gated_norm_fwd(y, z, w, G)
        gr = cuda_lib.gated_norm_bwd(y, z, w, dout, G, rstd=rstd)
        torch.cuda.synchronize()
        return out, rstd, gr
    try:
        tuning.clear_norm_config(F, G)
        a = run()
        tuning.set_norm_config(F, G, **cfg)
        b = run()
    finally:
        if had:
            tuning.set_norm_config(F, G, **saved)
        else:
            tuning.clear_norm_config(F, G)
    assert torch.equal(a[0], b[0]) and torch.equal(a[1], b[1])
    assert torch.equal(a[2]["dy"], b[2]["dy"]) and torch.equal(a[2]["dz"], b[2]["dz"])
    np.testing.assert_allclose(b[2]["dw"].cpu().numpy(), a[2]["dw"].cpu().numpy(), rtol=1e-5,
                               atol=1e-5)
    assert cuda_lib.device_status() == 0


# ------------------------------------------------------ SSD chunk kernels
_SSD_KEY = dict(batch=2, seqlen=1000, nheads=12, headdim=64, dstate=128, ngroups=2,
                chunk_size=128)


def _scan_table(*entries):
    return {"kind": tuning.SCAN_TABLE_KIND, "entries": list(entries)}


def _scan_entry(**kw):
    e = dict(_SSD_KEY, scan_head_blocks=3, bc_head_blocks=2)
    e.update(kw)
    return e


def _model_rule(key, sms=152, partials=False):
    """The built-in rule re-derived here: list scheduling of the launch (the
    heavy row tile's CTAs first, each to the SM that frees first), a CTA
    costing (column panels + 4) per head plus 6; for dC / dB (partials) more
    than one block adds the tail's pass over the partials (2 B T G N 4 bytes
    per slot read and per sum written, at 6.8e12 B/s, in units of 1100
    cycles at 2.07 GHz); the best (heavy, light) pair, fewer CTAs on a tie."""
    import heapq
    hpg = key["nheads"] // key["ngroups"] * (2 if key["headdim"] == 128 else 1)
    nc = -(-key["seqlen"] // key["chunk_size"])
    units = key["batch"] * nc * key["ngroups"]
    divs = [d for d in range(1, min(hpg, 32) + 1) if hpg % d == 0]

    def span(jobs):
        heap = [0.0] * sms
        end = 0.0
        for n, c in jobs:
            for _ in range(n):
                t = heapq.heappop(heap) + c
                heapq.heappush(heap, t)
                end = max(end, t)
        return end
    row_bytes = 2.0 * key["batch"] * key["seqlen"] * key["ngroups"] * key["dstate"] * 4.0

    def tail(nmax):
        if not partials or nmax <= 1:
            return 0.0
        return row_bytes * (nmax + 1) / 6.8e12 / (1100.0 / 2.07e9)
    best = None
    if key["chunk_size"] <= 128:
        cands = [((d, d), span([(units * d, hpg // d * 6 + 6)]) + tail(d), units * d)
                 for d in divs]
    else:
        hu = key["chunk_size"] // 64 + 4
        cands = [((h, l), span([(units * h, hpg // h * hu + 6), (units * l, hpg // l * 6 + 6)])
                  + tail(max(h, l)), units * (h + l)) for h in divs for l in divs]
    for pair, t, n in cands:
        if best is None or t < best[1] - 1e-9 or (t < best[1] + 1e-9 and n < best[2]):
            best = (pair, t, n)
    return best[0]


def test_scan_validate():
    tuning.validate_scan_table(_scan_table(_scan_entry(), _scan_entry(seqlen=2000)))
    for bad in (dict(scan_head_blocks=4), dict(bc_head_blocks=-1), dict(bc_head_blocks=33),
                dict(ngroups=5), dict(headdim=0)):
        with pytest.raises(ValueError):
            tuning.validate_scan_table(_scan_table(_scan_entry(**bad)))
    with pytest.raises(ValueError):
        tuning.validate_scan_table(_scan_table(_scan_entry(), _scan_entry()))
    with pytest.raises(ValueError):
        tuning.validate_scan_table(_table())


def test_scan_table_counts_headdim_128_heads_twice():
    """At headdim 128 the head blocks split two 64-wide heads per head: 3
    heads in 3 groups give 2 kernel heads per group, so 2 blocks are valid
    and 4 are not (library and Python validation agree)."""
    key = dict(batch=1, seqlen=333, nheads=3, headdim=128, dstate=64, ngroups=3, chunk_size=128)
    try:
        tuning.set_scan_config(key, 2, 2)
        got, from_table = tuning.get_scan_config(key)
        assert from_table and got["scan_head_blocks"] == 2 and got["bc_head_blocks"] == 2
        tuning.validate_scan_table(_scan_table(dict(key, scan_head_blocks=2, bc_head_blocks=2)))
        with pytest.raises(ValueError):
            tuning.set_scan_config(key, 4, 0)
        with pytest.raises(ValueError):
            tuning.validate_scan_table(_scan_table(dict(key, scan_head_blocks=4,
                                                        bc_head_blocks=0)))
    finally:
        tuning.clear_scan_config(key)


def test_scan_table_set_get_remove():
    """Host-only calls: the entry overrides the built-in head-block rule, a
    zero field keeps the rule's choice, and removing the entry restores it."""
    tuning.clear_scan_config(_SSD_KEY)
    rule, from_table = tuning.get_scan_config(_SSD_KEY)
    assert not from_table
    h, _ = _model_rule(_SSD_KEY)
    hb, _ = _model_rule(_SSD_KEY, partials=True)
    # chunk 128: one row tile, so the light count equals the heavy one
    assert rule == dict(scan_head_blocks=h, bc_head_blocks=hb, scan_head_blocks_light=h,
                        bc_head_blocks_light=hb)
    tuning.set_scan_config(_SSD_KEY, 2, 3)
    got, from_table = tuning.get_scan_config(_SSD_KEY)
    assert from_table and got["scan_head_blocks"] == 2 and got["bc_head_blocks"] == 3
    tuning.set_scan_config(_SSD_KEY, 0, 1)
    got = tuning.get_scan_config(_SSD_KEY)[0]
    assert got["scan_head_blocks"] == h and got["bc_head_blocks"] == 1
    for bad in ((4, 0), (0, 5), (-1, 0), (33, 0), (0, 0, 4, 0), (0, 0, 0, 5)):
        with pytest.raises(ValueError):
            tuning.set_scan_config(_SSD_KEY, *bad)
    tuning.clear_scan_config(_SSD_KEY)
    assert tuning.get_scan_config(_SSD_KEY) == (rule, False)


@pytest.mark.parametrize("key", [
    dict(batch=4, seqlen=4096, nheads=24, headdim=64, dstate=128, ngroups=1, chunk_size=256),
    dict(batch=1, seqlen=700, nheads=12, headdim=64, dstate=64, ngroups=2, chunk_size=256),
    dict(batch=2, seqlen=8192, nheads=64, headdim=64, dstate=128, ngroups=8, chunk_size=128),
    dict(batch=1, seqlen=131072, nheads=32, headdim=64, dstate=128, ngroups=1, chunk_size=256),
    # headdim 128: the kernels split a group's 2 x 6 64-wide heads
    dict(batch=4, seqlen=4096, nheads=12, headdim=128, dstate=128, ngroups=1, chunk_size=256),
])
def test_scan_rule_is_the_list_scheduling_model(key):
    """The library's built-in (heavy, light) head blocks equal the model's,
    re-derived in Python; table fields override one tile at a time."""
    saved = _table_entry(key)
    try:
        tuning.clear_scan_config(key)
        rule, from_table = tuning.get_scan_config(key)
        h, l = _model_rule(key)
        bh, bl = _model_rule(key, partials=True)
        assert not from_table
        assert (rule["scan_head_blocks"], rule["scan_head_blocks_light"]) == (h, l)
        assert (rule["bc_head_blocks"], rule["bc_head_blocks_light"]) == (bh, bl)
        if key["chunk_size"] > 128:
            tuning.set_scan_config(key, 0, 0, 1, 0)
            got = tuning.get_scan_config(key)[0]
            assert got["scan_head_blocks"] == h and got["scan_head_blocks_light"] == 1
            assert got["bc_head_blocks_light"] == bl
    finally:
        tuning.clear_scan_config(key)
        if saved is not None:
            tuning.set_scan_config(key, **saved)


def _table_entry(key):
    """The packaged table's fields for key (as loaded), or None."""
    if not os.path.exists(tuning.DEFAULT_SCAN_TABLE):
        return None
    with open(tuning.DEFAULT_SCAN_TABLE) as f:
        for e in json.load(f)["entries"]:
            if all(e[k] == key[k] for k in tuning._SCAN_KEYS):
                return {k: int(e.get(k, 0)) for k in tuning._SCAN_FIELDS}
    return None


def test_scan_table_apply_and_env(tmp_path, monkeypatch):
    p = tmp_path / "s.json"
    p.write_text(json.dumps(_scan_table(_scan_entry(seqlen=777))))
    monkeypatch.setenv("SSD_TUNING_TABLE", "none")
    monkeypatch.setenv("SSD_SCAN_TABLE", str(p))
    tuning.apply_default(tuning._native.load())
    key = dict(_SSD_KEY, seqlen=777)
    got, from_table = tuning.get_scan_config(key)
    assert from_table and got["scan_head_blocks"] == 3 and got["bc_head_blocks"] == 2
    tuning.clear_scan_config(key)


def test_packaged_scan_table_is_valid_and_loaded():
    if not os.path.exists(tuning.DEFAULT_SCAN_TABLE):
        pytest.skip("no packaged table")
    with open(tuning.DEFAULT_SCAN_TABLE) as f:
        t = json.load(f)
    tuning.validate_scan_table(t)
    assert t.get("generated_by", "").startswith("SSD_SCAN_TABLE=none python -m")
    if os.environ.get("SSD_SCAN_TABLE", tuning.DEFAULT_SCAN_TABLE) == tuning.DEFAULT_SCAN_TABLE:
        for e in t["entries"]:
            cfg, from_table = tuning.get_scan_config({k: e[k] for k in tuning._SCAN_KEYS})
            assert from_table
            for k in tuning._SCAN_FIELDS:
                if e.get(k, 0) > 0 and not (k.endswith("_light") and e["chunk_size"] <= 128):
                    assert cfg[k] == e[k], k


@pytest.mark.gpu
@pytest.mark.parametrize("key,cfg", [
    (_SSD_KEY, (1, 1, 0, 0)), (_SSD_KEY, (2, 3, 0, 0)), (_SSD_KEY, (6, 2, 0, 0)),
    (dict(batch=1, seqlen=700, nheads=12, headdim=64, dstate=64, ngroups=2, chunk_size=256),
     (2, 3, 3, 1)),
    (dict(batch=1, seqlen=700, nheads=12, headdim=64, dstate=64, ngroups=2, chunk_size=256),
     (6, 1, 1, 6)),
])
def test_tuned_ssd_launch_computes_the_same(cuda_lib, key, cfg):
    """Each head of a chunk tile is computed by the same arithmetic whichever
    head block holds it, so y, final_states, dx and ddt are bit-identical under
    any table entry (including different counts for the two row tiles of a
    256-row chunk); dB and dC sum the heads of a group over a different
    partition (per block, then over blocks), equal to rounding."""
    import torch

    from state_space_model_sm_gb300.inputs import SSDShape, make_inputs, to_torch
    k = key
    inp = make_inputs(SSDShape(k["batch"], k["seqlen"], k["nheads"], k["headdim"], k["dstate"],
                               k["ngroups"], k["chunk_size"]), seed=31, dtype="bf16",
                      init_std=0.1, with_dy=True, dfinal_std=0.1)
    t = to_torch(inp)
    saved, had = tuning.get_scan_config(k)

    def run():
        y, fin = cuda_lib.ssd_fwd(t["x"], t["dt"], t["dt_bias"], t["A"], t["B"], t["C"], t["D"],
                                  chunk_size=k["chunk_size"], init_states=t["init"])
        g = cuda_lib.ssd_bwd(t["x"], t["dt"], t["dt_bias"], t["A"], t["B"], t["C"], t["D"],
                             k["chunk_size"], t["init"], t["dy"], t["dfinal"])
        torch.cuda.synchronize()
        return y, fin, g
    try:
        tuning.clear_scan_config(k)
        a = run()
        tuning.set_scan_config(k, *cfg)
        b = run()
    finally:
        if had:
            tuning.set_scan_config(k, **saved)
        else:
            tuning.clear_scan_config(k)
    assert cuda_lib.device_status() == 0
    assert torch.equal(a[0], b[0]) and torch.equal(a[1], b[1])
    for name in ("dx", "ddt"):
        assert torch.equal(a[2][name], b[2][name]), name
    for name in ("dB", "dC", "dA", "ddt_bias", "dD", "dinit_states"):
        np.testing.assert_allclose(b[2][name].cpu().numpy(), a[2][name].cpu().numpy(),
                                   rtol=1e-5, atol=1e-5 * float(a[2][name].abs().max()),
                                   err_msg=name)
