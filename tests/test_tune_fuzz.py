"""Property tests of the tuning-table reader (a C++ JSON parser that reads files
from outside the library) and of the tuner's table writer, on the host.

Random documents must either load or be refused with CS_ERR_INVALID_ARG and a
message; the process must survive every input, and a refused file must leave
the loaded table as it was.  Valid documents written by Python's json module
must load with the entries they hold."""
from __future__ import annotations

import json
import os

import pytest

try:
    from hypothesis import HealthCheck, given, settings
    from hypothesis import strategies as st
except ImportError:  # the property tests need hypothesis; the plain tests below run without it
    given = None


@pytest.fixture(scope="module")
def cs():
    import __graft_entry__
    __graft_entry__._build_module().build()
    import consumer_gemm_chain_gb300 as cs
    return cs


BASE = {"kind": "gelu", "dtype": "f16", "H": 12288, "F": 6144, "M": 64, "sms": 152,
        "tile_m": 128, "tile_n": 128, "split_k": 1}
# optional fields the reader checks when present (random documents must not name them)
OPTIONAL = ("group_m", "layout", "policy", "us", "sk_tiles", "sk_units")


def _load_text(cs, tmp_path, text: bytes):
    p = tmp_path / "t.json"
    p.write_bytes(text)
    return cs.cs_tune_load(str(p))


if given is not None:
    SETTINGS = settings(max_examples=300, deadline=None, suppress_health_check=[HealthCheck.function_scoped_fixture])

    @SETTINGS
    @given(st.binary(max_size=400))
    def test_random_bytes_never_crash(cs, tmp_path, data):
        cs.cs_tune_clear()
        try:
            n = _load_text(cs, tmp_path, data)
        except cs.CSError as e:
            assert e.status == cs.CS_ERR_INVALID_ARG and str(e)
            assert cs.cs_tune_size() == 0
        else:  # only a well-formed table with an empty entry list can come out of noise
            assert n == cs.cs_tune_size()


    json_scalars = st.none() | st.booleans() | st.integers(-10**6, 10**6) | st.floats(allow_nan=False, allow_infinity=False) \
        | st.text(max_size=12)
    json_values = st.recursive(json_scalars, lambda c: st.lists(c, max_size=4) | st.dictionaries(st.text(max_size=6), c, max_size=4),
                               max_leaves=20)


    @SETTINGS
    @given(extra=st.dictionaries(st.text(max_size=8).filter(lambda k: k not in OPTIONAL), json_values, max_size=4),
           ws=st.sampled_from(["", " ", "\n\t", "  \r\n"]))
    def test_valid_tables_with_unknown_keys_load(cs, tmp_path, extra, ws):
        entry = dict(extra)
        entry.update(BASE)  # the required fields win over random ones of the same name
        doc = {"format": "cs_chain_tuning", "version": 1, "entries": [entry, dict(BASE, M=128)], "notes": extra}
        text = json.dumps(doc, indent=1 if ws else None).replace("\n", "\n" + ws)
        assert _load_text(cs, tmp_path, text.encode()) == 2
        cs.cs_tune_clear()


    @SETTINGS
    @given(field=st.sampled_from(sorted(BASE)), value=json_values)
    def test_random_field_values_load_or_name_the_field(cs, tmp_path, field, value):
        cs.cs_tune_clear()
        keep = {"format": "cs_chain_tuning", "version": 1, "entries": [BASE]}
        assert _load_text(cs, tmp_path, json.dumps(keep).encode()) == 1
        entry = dict(BASE)
        entry[field] = value
        doc = {"format": "cs_chain_tuning", "version": 1, "entries": [entry]}
        try:
            n = _load_text(cs, tmp_path, json.dumps(doc).encode())
        except cs.CSError as e:
            assert e.status == cs.CS_ERR_INVALID_ARG and f'"{field}"' in str(e)
            assert cs.cs_tune_size() == 1  # the earlier table stays
        else:
            assert n == 1
        cs.cs_tune_clear()


    @SETTINGS
    @given(cut=st.integers(0, 200))
    def test_truncated_files_are_refused(cs, tmp_path, cut):
        cs.cs_tune_clear()
        text = json.dumps({"format": "cs_chain_tuning", "version": 1, "entries": [BASE, dict(BASE, M=2)]})
        cut = min(cut, len(text) - 1)
        with pytest.raises(cs.CSError) as e:
            _load_text(cs, tmp_path, text[:cut].encode())
        assert e.value.status == cs.CS_ERR_INVALID_ARG

else:
    @pytest.mark.skip(reason="hypothesis is not installed")
    def test_property_tests_need_hypothesis():
        pass


def test_deep_nesting_is_refused_not_overflowed(cs, tmp_path):
    deep = "[" * 100000 + "]" * 100000
    text = '{"format": "cs_chain_tuning", "version": 1, "x": ' + deep + ', "entries": []}'
    with pytest.raises(cs.CSError) as e:
        _load_text(cs, tmp_path, text.encode())
    assert "nested too deeply" in str(e.value)


def test_writer_merges_by_key_and_the_reader_reads_it(cs, tmp_path):
    from consumer_gemm_chain_gb300 import tune
    path = str(tmp_path / "sub" / "table.json")
    dev = {"name": "test", "sms": 152, "cc": "10.3"}
    a = [dict(BASE, M=m, layout="nk", policy="tile", us=10.0 + m, builtin_us=11.0 + m) for m in (1, 64)]
    assert tune.write_table(path, a, merge=False, device=dev) == 2
    # a second shape merged in, and one entry of the first re-measured
    b = [dict(BASE, M=64, layout="nk", policy="tile", tile_m=256, tile_n=256, us=5.0, builtin_us=9.0),
         dict(BASE, kind="swiglu", dtype="bf16", H=8192, F=2752, M=16, layout="nk", policy="row", us=1.0, builtin_us=2.0)]
    assert tune.write_table(path, b, merge=True, device=dev) == 3
    with open(path) as f:
        doc = json.load(f)
    assert doc["format"] == "cs_chain_tuning" and doc["device"] == dev
    got = {(e["kind"], e["M"]): e for e in doc["entries"]}
    assert got[("gelu", 64)]["tile_m"] == 256 and got[("gelu", 1)]["tile_m"] == 128
    try:
        assert cs.cs_tune_load(path) == 3
        d = cs.cs_chain_desc_init(kind="gelu", M=64, H=12288, F=6144, weight_layout="nk", policy="tile")
        e, r = cs.cs_tune_match(d, 152)
        assert e >= 0 and r.tile_m == 256
    finally:
        cs.cs_tune_clear()
    # without merge the file holds only the new entries
    assert tune.write_table(path, b[:1], merge=False, device=dev) == 1
    assert os.path.exists(path)
