"""Host-side checks of the C-ABI library that need no GPU: it loads, exports every
symbol include/cs_chain.h declares, validates descriptors and builds a
dependency-respecting schedule."""
from __future__ import annotations

import ctypes
import os
import re

import pytest

ROOT = os.path.dirname(os.path.dirname(os.path.abspath(__file__)))


@pytest.fixture(scope="module")
def cs():
    import __graft_entry__
    __graft_entry__._build_module().build()
    import consumer_gemm_chain_gb300 as cs
    return cs


def header_functions():
    text = open(os.path.join(ROOT, "include", "cs_chain.h")).read()
    text = re.sub(r"/\*.*?\*/", "", text, flags=re.S)
    return sorted(set(re.findall(r"\b(cs_[a-z0-9_]+)\s*\(", text)))


def test_every_declared_symbol_is_exported(cs):
    lib = ctypes.CDLL(cs.chain.LIB_PATH)
    names = header_functions()
    assert "cs_chain_plan" in names and "cs_mlp_forward" in names and "cs_chain_destroy" in names
    for n in names:
        assert hasattr(lib, n), f"{n} declared in cs_chain.h but not exported"
    assert set(cs.chain.EXPORTED) == set(names)
    assert cs.cs_abi_version() == 1


def test_desc_defaults(cs):
    d = cs.cs_chain_desc_init()
    assert (d.kind, d.dtype, d.policy, d.weight_layout, d.lag) == (0, 0, 0, 0, -1)
    assert d.head_dim == 128


@pytest.mark.parametrize("field,value", [("M", 0), ("H", 12), ("F", 0), ("dtype", 7), ("policy", 9),
                                         ("kind", 5), ("weight_layout", 3), ("lag", -2), ("num_sms", -1)])
def test_invalid_descs_are_rejected_without_a_gpu(cs, field, value):
    d = cs.cs_chain_desc_init(M=64, H=256, F=1024)
    setattr(d, field, value)
    with pytest.raises(cs.CSError) as e:
        cs.cs_chain_plan(d)
    assert e.value.status == cs.CS_ERR_INVALID_ARG
    with pytest.raises(cs.CSError):
        cs.cs_schedule_build(d, 148)


def test_null_arguments(cs):
    lib = cs.chain._lib
    assert lib.cs_chain_plan(None, None) == cs.CS_ERR_INVALID_ARG
    assert lib.cs_chain_destroy(None) == cs.CS_OK
    assert lib.cs_mlp_forward(None, None, None) == cs.CS_ERR_INVALID_ARG
    assert lib.cs_chain_status(None) == cs.CS_ERR_INVALID_ARG
    assert lib.cs_chain_desc_init(None) == cs.CS_ERR_INVALID_ARG
    assert "NULL" in cs.cs_last_error_string()


def _deps(stage_kind, s, m, n, d, q):
    """Producer units (stage, m, n) a unit waits on, under the plan's policy (TILE: the
    tiles its K-slices read; every policy waits on a superset of those)."""
    if s == 0:
        return []
    if stage_kind == "attn" and s == 1:
        heads = d.heads
        return [(0, j, t) for j in range(m + 1) for t in (n, n + heads, n + 2 * heads)]
    ntp = q[s - 1]
    return [(s - 1, m, t) for t in range(ntp)]


@pytest.mark.parametrize("tile_m,tile_n", [(128, 128), (128, 256), (256, 256)])
@pytest.mark.parametrize("M,H,F,sms,lag,group", [(64, 256, 1024, 148, -1, 0), (2048, 12288, 6144, 148, -1, 0),
                                                 (2048, 12288, 6144, 152, 0, 3), (1, 12288, 6144, 148, -1, 0),
                                                 (1000, 8192, 2752, 148, 2, 1), (1536, 8192, 8192, 148, 5, 5)])
def test_schedule_is_dependency_ordered(cs, M, H, F, sms, lag, group, tile_n, tile_m):
    d = cs.cs_chain_desc_init(M=M, H=H, F=F, lag=lag, group_m=group, tile_n=tile_n, tile_m=tile_m)
    units = cs.cs_schedule_build(d, sms)
    m_tiles = -(-M // tile_m)
    n0, n1 = -(-F // tile_n), -(-H // tile_n)
    dec = [cs.decode_unit(u) for u in units]
    # every unit exactly once
    expect = {(0, m, n) for m in range(m_tiles) for n in range(n0)} | {(1, m, n) for m in range(m_tiles) for n in range(n1)}
    assert len(dec) == len(expect) and set(dec) == expect
    pos = {u: i for i, u in enumerate(dec)}
    for (s, m, n), i in pos.items():
        for dep in _deps("mlp", s, m, n, d, [n0, n1]):
            assert pos[dep] < i, f"unit {(s, m, n)} at {i} precedes its producer {dep}"


@pytest.mark.parametrize("M,lag,group", [(1, -1, 0), (300, -1, 0), (2048, -1, 0), (2048, 2, 3), (1000, 0, 1)])
def test_attention_schedule_is_dependency_ordered(cs, M, lag, group):
    d = cs.cs_chain_desc_init(kind="attn", M=M, H=12288, F=1536, heads=12, head_dim=128, lag=lag, group_m=group)
    dec = [cs.decode_unit(u) for u in cs.cs_schedule_build(d, 148)]
    m_tiles = -(-M // 128)
    nt = [36, 12, 96]
    expect = {(s, m, n) for s in range(3) for m in range(m_tiles) for n in range(nt[s])}
    assert len(dec) == len(expect) and set(dec) == expect
    pos = {u: i for i, u in enumerate(dec)}
    for (s, m, n), i in pos.items():
        deps = []
        if s == 1:   # causal: key blocks 0..m of head n (Q, K and V tiles)
            deps = [(0, j, t) for j in range(m + 1) for t in (n, n + 12, n + 24)]
        elif s == 2:  # every head of the same row block
            deps = [(1, m, h) for h in range(12)]
        for dep in deps:
            assert pos[dep] < i, (s, m, n, dep)


def test_attention_desc_validation(cs):
    d = cs.cs_chain_desc_init(kind="attn", M=64, H=256, F=256, heads=2, head_dim=64)
    with pytest.raises(cs.CSError) as e:
        cs.cs_schedule_build(d, 148)
    assert e.value.status == cs.CS_ERR_UNSUPPORTED
    d = cs.cs_chain_desc_init(kind="attn", M=64, H=256, F=384, heads=2, head_dim=128)
    with pytest.raises(cs.CSError) as e:
        cs.cs_schedule_build(d, 148)
    assert e.value.status == cs.CS_ERR_INVALID_ARG


def test_schedule_rasterises_column_major_within_a_group(cs):
    d = cs.cs_chain_desc_init(M=2048, H=12288, F=6144, group_m=4, lag=1, tile_n=128)
    dec = [cs.decode_unit(u) for u in cs.cs_schedule_build(d, 148)]
    # first group of producers: (n, m) with m fastest
    assert dec[:8] == [(0, 0, 0), (0, 1, 0), (0, 2, 0), (0, 3, 0), (0, 0, 1), (0, 1, 1), (0, 2, 1), (0, 3, 1)]
    # then the second producer group, then the first consumer group
    assert dec[192] == (0, 4, 0) and dec[384] == (1, 0, 0)


def test_auto_tile_shape(cs):
    big = cs.cs_schedule_build(cs.cs_chain_desc_init(M=2048, H=12288, F=6144), 148)
    mid = cs.cs_schedule_build(cs.cs_chain_desc_init(M=640, H=12288, F=6144), 148)
    small = cs.cs_schedule_build(cs.cs_chain_desc_init(M=256, H=12288, F=6144), 148)
    assert len(big) == 8 * 24 + 8 * 48      # 256 x 256 tiles on CTA pairs for large M
    assert len(mid) == 5 * 24 + 5 * 48      # 128 x 256 tiles on single SMs in between
    assert len(small) == 2 * 48 + 2 * 96    # 128 x 128 tiles for small M


def test_pair_tiles_need_wide_gelu_tiles(cs):
    d = cs.cs_chain_desc_init(M=512, H=512, F=512, tile_m=256, tile_n=128)
    with pytest.raises(cs.CSError) as e:
        cs.cs_schedule_build(d, 148)
    assert e.value.status == cs.CS_ERR_UNSUPPORTED
