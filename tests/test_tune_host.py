"""The tuning table on the host, without a GPU: the JSON reader, the matching
rules of cs_tune_match, and the schedule a plan with a tuned desc builds."""
from __future__ import annotations

import json
import os

import pytest


@pytest.fixture(scope="module")
def cs():
    import __graft_entry__
    __graft_entry__._build_module().build()
    import consumer_gemm_chain_gb300 as cs
    return cs


@pytest.fixture
def table(cs, tmp_path):
    """Writes a table file, loads it, and empties the table again afterwards."""
    def load(entries, **top):
        doc = {"format": "cs_chain_tuning", "version": 1, "entries": entries}
        doc.update(top)
        path = tmp_path / "t.json"
        path.write_text(json.dumps(doc))
        return cs.cs_tune_load(str(path))
    yield load
    cs.cs_tune_clear()


def E(M, tile_m=128, tile_n=128, split_k=1, **kw):
    e = {"kind": "gelu", "dtype": "f16", "H": 12288, "F": 6144, "M": M, "sms": 152,
         "tile_m": tile_m, "tile_n": tile_n, "split_k": split_k}
    e.update(kw)
    return e


def gpt3(cs, M, **kw):
    kw.setdefault("weight_layout", "nk")
    kw.setdefault("dtype", 0)
    return cs.cs_chain_desc_init(kind="gelu", M=M, H=12288, F=6144, **kw)


def test_empty_table_leaves_built_in_rules(cs):
    cs.cs_tune_clear()
    assert cs.cs_tune_size() == 0
    e, r = cs.cs_tune_match(gpt3(cs, 2048, policy="auto"), 152)
    assert e == -1 and r.policy == cs.CS_SYNC_TILE and r.tile_m == 0


def test_exact_and_nearest_m_on_a_log_scale(cs, table):
    assert table([E(16, split_k=12), E(64, split_k=3), E(1024, 512, 256), E(2048, 256, 256)]) == 4
    for M, want in [(16, 0), (64, 2 - 1), (1024, 2), (2048, 3), (1, 0), (40, 1), (200, 1), (300, 2), (4096, 3),
                    (32, 0),     # 16 and 64 are equally near: the smaller M
                    (1448, 2)]:  # below sqrt(1024 * 2048) = 1448.2
        e, _ = cs.cs_tune_match(gpt3(cs, M), 152)
        assert e == want, M
    _, r = cs.cs_tune_match(gpt3(cs, 2000), 152)
    assert (r.tile_m, r.tile_n, r.split_k, r.group_m) == (256, 256, 1, 0)


def test_shape_dtype_grid_and_layout_must_match(cs, table):
    table([E(64, layout="kn"), E(64, split_k=2, layout="nk"), E(64, split_k=4, sms=148)])
    assert cs.cs_tune_match(gpt3(cs, 64, weight_layout="nk"), 152)[0] == 1
    assert cs.cs_tune_match(gpt3(cs, 64, weight_layout="kn"), 152)[0] == 0
    assert cs.cs_tune_match(gpt3(cs, 64), 148)[0] == 2
    assert cs.cs_tune_match(gpt3(cs, 64), 132)[0] == -1
    assert cs.cs_tune_match(gpt3(cs, 64, dtype=1), 152)[0] == -1
    other = cs.cs_chain_desc_init(kind="gelu", M=64, H=8192, F=6144, weight_layout="nk")
    assert cs.cs_tune_match(other, 152)[0] == -1
    swiglu = cs.cs_chain_desc_init(kind="swiglu", M=64, H=12288, F=6144, weight_layout="nk")
    assert cs.cs_tune_match(swiglu, 152)[0] == -1


def test_policy_rules(cs, table):
    table([E(512, policy="tile", us=150.0), E(512, 256, 256, policy="row", us=140.0),
           E(512, 512, 256, policy="stream", us=120.0), E(512, split_k=2, policy="any", us=200.0)])
    # auto: the fastest fused policy; the two-kernel control is never chosen
    e, r = cs.cs_tune_match(gpt3(cs, 512, policy="auto"), 152)
    assert e == 1 and r.policy == cs.CS_SYNC_ROW and (r.tile_m, r.tile_n) == (256, 256)
    # a given policy: its own entry before an "any" entry, even a slower one
    assert cs.cs_tune_match(gpt3(cs, 512, policy="tile"), 152)[0] == 0
    assert cs.cs_tune_match(gpt3(cs, 512, policy="stream"), 152)[0] == 2
    e, r = cs.cs_tune_match(gpt3(cs, 512, policy="strided"), 152)
    assert e == 3 and r.split_k == 2 and r.policy == cs.CS_SYNC_STRIDED


def test_fields_set_by_the_caller_are_kept(cs, table):
    table([E(512, 256, 256, split_k=3, policy="row", us=1.0)])
    # any of the five tile fields given: the table does not touch them
    for field, value in [("tile_m", 128), ("tile_n", 128), ("split_k", 1), ("split_k_first", 2), ("group_m", 2)]:
        e, r = cs.cs_tune_match(gpt3(cs, 512, policy="row", **{field: value}), 152)
        assert e == -1 and getattr(r, field) == value
    # ... but an auto policy is still resolved from it
    e, r = cs.cs_tune_match(gpt3(cs, 512, policy="auto", tile_m=128), 152)
    assert e == 0 and r.policy == cs.CS_SYNC_ROW and r.tile_m == 128 and r.split_k == 0
    # tuned = -1: never consulted
    e, r = cs.cs_tune_match(gpt3(cs, 512, policy="auto", tuned=-1), 152)
    assert e == -1 and r.policy == cs.CS_SYNC_TILE


def test_entry_the_desc_rejects_is_ignored(cs, table):
    attn = {"kind": "attn", "dtype": "f16", "H": 12288, "F": 1536, "M": 1024, "sms": 152,
            "tile_m": 512, "tile_n": 256, "split_k": 1}
    table([attn])
    d = cs.cs_chain_desc_init(kind="attn", M=1024, H=12288, F=1536, heads=12, policy="auto")
    e, r = cs.cs_tune_match(d, 152)
    assert e == -1 and r.tile_m == 0 and r.policy == cs.CS_SYNC_TILE
    assert cs.cs_last_error_string() == ""  or "attention" not in cs.cs_last_error_string()


def test_first_stage_splits_and_order_come_from_the_entry(cs, table):
    """split_k_first and raster are optional keys: applied with the tile fields,
    the order only where the desc leaves it on auto."""
    table([E(1, split_k=6, split_k_first=8, raster=3, us=1.0), E(16, split_k=3, us=1.0)])
    e, r = cs.cs_tune_match(gpt3(cs, 1), 152)
    assert e == 0 and (r.split_k, r.split_k_first, r.raster) == (6, 8, 3)
    q = cs.cs_chain_plan_info(gpt3(cs, 1), 152)
    assert q["split_k"][:2] == [8, 6] and q["raster"] == 3
    e, r = cs.cs_tune_match(gpt3(cs, 1, raster=2), 152)
    assert e == 0 and r.raster == 2 and r.split_k_first == 8
    e, r = cs.cs_tune_match(gpt3(cs, 16), 152)   # keys absent: defaults
    assert e == 1 and (r.split_k, r.split_k_first, r.raster) == (3, 0, 0)
    assert cs.cs_chain_plan_info(gpt3(cs, 16), 152)["raster"] == 1


def test_schedule_follows_the_tuned_tiles(cs, table):
    d = gpt3(cs, 2048)
    n_builtin = len(cs.cs_schedule_build(d, 152))   # 512 x 256 tiles: 4 x (24 + 48)
    assert n_builtin == 4 * (24 + 48)
    table([E(2048, 128, 128, split_k=1)])
    assert len(cs.cs_schedule_build(d, 152)) == 16 * (48 + 96)
    d.tuned = -1
    assert len(cs.cs_schedule_build(d, 152)) == n_builtin


@pytest.mark.parametrize("text,what", [
    ("{", "expected a string at byte 1"),
    ("", "unexpected end"),
    ('{"format": "cs_chain_tuning", "version": 1, "entries": [1,]}', "byte"),
    ('{"format": "x", "version": 1, "entries": []}', "format"),
    ('{"format": "cs_chain_tuning", "version": 2, "entries": []}', "version"),
    ('{"format": "cs_chain_tuning", "version": 1}', "entries"),
    ('{"format": "cs_chain_tuning", "version": 1, "entries": [], } ', "byte"),
    ('{"format": "cs_chain_tuning", "version": 1, "entries": []} x', "trailing"),
    ('{"format": "cs_chain_tuning", "version": 1, "entries": [{"kind": "gelu"}]}', "entry 0: missing"),
])
def test_malformed_files_are_rejected_and_keep_the_table(cs, table, tmp_path, text, what):
    table([E(64)])
    bad = tmp_path / "bad.json"
    bad.write_text(text)
    with pytest.raises(cs.CSError) as err:
        cs.cs_tune_load(str(bad))
    assert err.value.status == cs.CS_ERR_INVALID_ARG and what in str(err.value)
    assert cs.cs_tune_size() == 1


@pytest.mark.parametrize("field,value", [("tile_m", 384), ("tile_n", 32), ("split_k", 16), ("M", 0),
                                         ("H", 12.5), ("kind", "conv"), ("dtype", "f32"), ("policy", "none"),
                                         ("layout", "mk"), ("us", -1), ("group_m", -1), ("sms", "152"),
                                         ("split_k_first", 16), ("raster", 4), ("raster", -1)])
def test_bad_entries_name_their_field(cs, table, field, value):
    bad = E(128)
    bad[field] = value
    with pytest.raises(cs.CSError) as err:
        table([E(64), bad])
    assert "entry 1" in str(err.value) and field in str(err.value)
    assert cs.cs_tune_size() == 0


def test_reader_accepts_json_details(cs, table):
    # escapes, exponents, nested unknown keys, whitespace
    n = table([dict(E(64), note='a"b\u00e9\n/', extra={"x": [1, 2.5e3, None, True]}, us=1.25e2)],
              device={"name": "GB300", "sms": 152})
    assert n == 1


def test_number_edges(cs, table, tmp_path):
    # an underflowing number is read (as a subnormal or zero), an overflowing one refused
    assert table([dict(E(64), us=1e-320, extra=2.2e-311)]) == 1
    bad = tmp_path / "big.json"
    bad.write_text('{"format": "cs_chain_tuning", "version": 1, "entries": [], "x": 1e400}')
    with pytest.raises(cs.CSError) as err:
        cs.cs_tune_load(str(bad))
    assert "number out of range" in str(err.value)


@pytest.mark.parametrize("text,ok", [("128", True), ("128.0", True), ("1.28e2", True), ("12.8e1", True),
                                     ("128.5", False), ("1e2", False)])
def test_integer_fields_in_any_json_number_form(cs, table, tmp_path, text, ok):
    """Integer fields are read exactly whatever form the number takes (the reader
    does not go through the C library's locale-dependent conversion)."""
    path = tmp_path / "t.json"
    path.write_text('{"format": "cs_chain_tuning", "version": 1, "entries": [' +
                    json.dumps(E(64))[:-1].replace('"tile_m": 128', '"tile_m": ' + text) + '}]}')
    if ok:
        assert cs.cs_tune_load(str(path)) == 1
    else:
        with pytest.raises(cs.CSError):
            cs.cs_tune_load(str(path))


def test_missing_file(cs, tmp_path):
    with pytest.raises(cs.CSError) as err:
        cs.cs_tune_load(str(tmp_path / "nope.json"))
    assert "cannot open" in str(err.value)


def test_packaged_table_matches_its_own_entries(cs):
    """Every entry of the shipped table loads, and a desc of exactly its shape, M
    and policy resolves to an entry with the same choices."""
    path = cs.chain.TUNE_TABLE
    if not os.path.exists(path):
        pytest.skip("no tuning table shipped")
    with open(path) as f:
        doc = json.load(f)
    try:
        assert cs.cs_tune_load() == len(doc["entries"])
        kinds = {"gelu": 0, "swiglu": 1, "attn": 2}
        for e in doc["entries"]:
            d = cs.cs_chain_desc_init(kind=kinds[e["kind"]], M=e["M"], H=e["H"], F=e["F"],
                                      dtype=0 if e["dtype"] == "f16" else 1, policy=e["policy"],
                                      weight_layout=e["layout"], heads=e["F"] // 128 if e["kind"] == "attn" else 12)
            idx, r = cs.cs_tune_match(d, e["sms"])
            assert idx >= 0, e
            assert (r.tile_m, r.tile_n, r.split_k) == (e["tile_m"], e["tile_n"], e["split_k"]), e
            assert (r.split_k_first, r.raster) == (e.get("split_k_first", 0), e.get("raster", 0)), e
            assert e["us"] <= e["builtin_us"] * 1.0001
    finally:
        cs.cs_tune_clear()


def test_tuner_k_range_candidates(cs):
    """The K-range phase times each (split, first-stage split) pair once, and
    tells candidates apart by every stage's tile width and splits: 128 x 128 and
    128 x 256 tiles with the same splits are two candidates."""
    from consumer_gemm_chain_gb300 import tune
    assert tune.k_range_combos(3) == [(0, 0), (3, 0), (4, 0), (6, 0), (8, 0), (3, 6), (3, 8), (3, 12), (1, 3), (1, 6)]
    c6 = tune.k_range_combos(6)
    assert len(c6) == len(set(c6)) and (6, 12) in c6 and (6, 6) not in c6
    keys = set()
    for tn in (128, 256):
        d = cs.cs_chain_desc_init(kind="gelu", M=1, H=12288, F=6144, tile_m=128, tile_n=tn, split_k=6, raster=3,
                                  tuned=-1)
        keys.add(tune.plan_key(cs.cs_chain_plan_info(d, 152)))
    assert len(keys) == 2


def test_tuner_shapes_of_ones_own():
    from consumer_gemm_chain_gb300 import tune
    assert tune.parse_shape("gelu, 8192, 4096, bf16") == ("gelu", 8192, 4096, "bf16", 0)
    assert tune.parse_shape("attn,12288,1536,f16,12") == ("attn", 12288, 1536, "f16", 12)
    for bad in ("gelu,8192,4096", "conv,8,8,f16", "gelu,8190,4096,f16", "attn,12288,1536,f16",
                "gelu,8,8,f32", "gelu,x,8,f16"):
        with pytest.raises(ValueError):
            tune.parse_shape(bad)
    # the command line refuses before it looks for a GPU
    for argv in ([], ["--shape", "gelu,1,2"], ["--preset", "gpt3", "--layout", "mk"]):
        with pytest.raises(SystemExit) as e:
            tune.main(argv)
        assert e.value.code == 2
