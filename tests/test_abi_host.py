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
    assert cs.cs_abi_version() == 7


def test_desc_defaults(cs):
    d = cs.cs_chain_desc_init()
    assert (d.kind, d.dtype, d.policy, d.weight_layout, d.lag) == (0, 0, 0, 0, -1)
    assert d.head_dim == 128


@pytest.mark.parametrize("field,value", [("M", 0), ("H", 12), ("F", 0), ("dtype", 7), ("policy", 9),
                                         ("kind", 5), ("weight_layout", 3), ("lag", -2), ("num_sms", -1),
                                         ("split_k", 16), ("tile_n", 192), ("tile_m", 64), ("tile_m", 1024), ("M", 128 * 4096),
                                         ("raster", 4), ("raster", -1), ("split_k_first", 16),
                                         ("split_k_first", -1), ("prefetch", -2), ("pdl", 2), ("pdl", -2),
                                         ("policy", -2), ("tuned", 1), ("tuned", -2), ("out_release", 2),
                                         ("out_release", -1)])
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


def _check_order(dec, deps_of):
    """Every unit appears once and after every producer unit it depends on."""
    pos = {u: i for i, u in enumerate(dec)}
    assert len(pos) == len(dec)
    for u, i in pos.items():
        for dep in deps_of(u):
            assert pos[dep] < i, f"unit {u} at {i} precedes its producer {dep}"


@pytest.mark.parametrize("tile_m,tile_n", [(128, 64), (128, 128), (128, 256), (256, 256), (512, 256)])
@pytest.mark.parametrize("M,H,F,sms,lag,group,split", [(64, 256, 1024, 148, -1, 0, 1), (2048, 12288, 6144, 148, -1, 0, 1),
                                                       (2048, 12288, 6144, 152, 0, 3, 1), (1, 12288, 6144, 148, -1, 0, 3),
                                                       (1000, 8192, 2752, 148, 2, 1, 2), (1536, 8192, 8192, 148, 5, 5, 1)])
@pytest.mark.parametrize("raster", [1, 2, 3])
def test_schedule_is_dependency_ordered(cs, M, H, F, sms, lag, group, split, tile_n, tile_m, raster):
    d = cs.cs_chain_desc_init(M=M, H=H, F=F, lag=lag, group_m=group, tile_n=tile_n, tile_m=tile_m, split_k=split,
                              raster=raster)
    dec = [cs.decode_unit(u) for u in cs.cs_schedule_build(d, sms)]
    m_tiles = -(-M // tile_m)
    n0, n1 = -(-F // tile_n), -(-H // tile_n)
    # with an explicit split_k every GEMM stage gets that many splits (enough K-slices here)
    expect = {(0, m, n, k) for m in range(m_tiles) for n in range(n0) for k in range(split)} | \
             {(1, m, n, k) for m in range(m_tiles) for n in range(n1) for k in range(split)}
    assert len(dec) == len(expect) and set(dec) == expect

    def deps(u):
        s, m, n, _ = u
        return [] if s == 0 else [(0, m, t, k) for t in range(n0) for k in range(split)]
    _check_order(dec, deps)


@pytest.mark.parametrize("tile_m", [128, 256])
@pytest.mark.parametrize("M,lag,group", [(1, -1, 0), (300, -1, 0), (2048, -1, 0), (2048, 2, 3), (1000, 0, 1)])
@pytest.mark.parametrize("kv", [-1, 0, 2])
def test_attention_schedule_is_dependency_ordered(cs, M, lag, group, tile_m, kv):
    d = cs.cs_chain_desc_init(kind="attn", M=M, H=12288, F=1536, heads=12, head_dim=128, lag=lag, group_m=group,
                              tile_m=tile_m, kv_chunk=kv)
    dec = [cs.decode_unit(u) for u in cs.cs_schedule_build(d, 148)]
    kv_arg, kv = kv, cs.cs_chain_plan_info(d, 148)["kv_chunk"]
    m_tiles = -(-M // tile_m)
    tn = tile_m  # 128 x 128 single-SM tiles or 256 x 256 pair tiles
    nt = [4608 // tn, 12, 12288 // tn]
    splits = {}
    for s, m, n, k in dec:
        splits[(s, m, n)] = max(splits.get((s, m, n), 0), k + 1)
    assert len(dec) == len(set(dec))
    assert set(splits) == {(s, m, n) for s in range(3) for m in range(m_tiles) for n in range(nt[s])}
    # attention units: one per row and head, or ceil((m + 1) / kv) key-range pieces
    assert all(v == (-(-(m + 1) // kv) if kv else 1) for (s, m, _), v in splits.items() if s == 1)
    if kv_arg <= 0:
        assert kv == 0  # auto and -1: whole rows

    def deps(u):
        s, m, n, _ = u
        if s == 1:   # causal: key blocks up to the unit's last query block (Q, K and V tiles of head n)
            tiles = {(p * 12 + n) * 128 // tn for p in range(3)}
            return [(0, j, t, k) for j in range(m + 1) for t in tiles for k in range(splits[(0, j, t)])]
        if s == 2:   # every piece of every head of the same row block
            return [(1, m, h, k) for h in range(12) for k in range(splits[(1, m, h)])]
        return []
    _check_order(dec, deps)


def test_small_m_splits_k_automatically(cs):
    d = cs.cs_chain_desc_init(M=64, H=12288, F=6144)
    dec = [cs.decode_unit(u) for u in cs.cs_schedule_build(d, 152)]
    s0 = [u for u in dec if u[0] == 0]
    assert {u[3] for u in s0} == {0, 1, 2}        # 48 tiles, 152 SMs: 3 splits fill one wave
    assert len(s0) == 48 * 3
    s1 = [u for u in dec if u[0] == 1]
    assert {u[3] for u in s1} == {0, 1, 2}        # 96 tiles: 3 splits = 2 waves of 32 K-slices
    # the splits of a tile are consecutive
    assert s0[:3] == [(0, 0, 0, 0), (0, 0, 0, 1), (0, 0, 0, 2)]
    big = [cs.decode_unit(u) for u in cs.cs_schedule_build(cs.cs_chain_desc_init(M=2048, H=12288, F=6144), 152)]
    assert {u[3] for u in big} == {0}             # enough tiles: no split at large M


@pytest.mark.parametrize("kind,M,H,F,split,first", [
    ("gelu", 1, 12288, 6144, 6, 9), ("gelu", 1, 12288, 6144, 0, 6), ("swiglu", 16, 8192, 2752, 4, 6),
    ("attn", 16, 12288, 1536, 3, 8), ("gelu", 64, 12288, 6144, 3, 1)])
def test_split_k_first_sets_the_first_stage_only(cs, kind, M, H, F, split, first):
    """split_k_first replaces split_k (explicit or automatic) for the first
    GEMM stage alone; the later stages keep what split_k gives them."""
    extra = dict(heads=F // 128, head_dim=128) if kind == "attn" else {}
    base = cs.cs_chain_desc_init(kind=kind, M=M, H=H, F=F, split_k=split, tile_m=128, tile_n=128, tuned=-1, **extra)
    d = cs.cs_chain_desc_init(kind=kind, M=M, H=H, F=F, split_k=split, split_k_first=first, tile_m=128, tile_n=128,
                              tuned=-1, **extra)
    qb, q = cs.cs_chain_plan_info(base, 152), cs.cs_chain_plan_info(d, 152)
    assert q["split_k"][0] == first and q["split_k"][1:] == qb["split_k"][1:]
    units = [cs.decode_unit(u) for u in cs.cs_schedule_build(d, 152)]
    assert {k for s, _, _, k in units if s == 0} == set(range(first))
    assert q["sched_units"][0] == q["n_tiles"][0] * -(-M // 128) * first


def test_64_wide_tiles_on_single_sms_only(cs):
    """tile_n = 64: single-SM MLP tiles (twice the tiles of 128, the SwiGLU
    producer keeping its 128-wide gate|up tiles); refused for pairs, clusters
    and the attention chain, and never chosen automatically."""
    for kind, F, n0 in (("gelu", 6144, 96), ("swiglu", 2752, 22)):
        d = cs.cs_chain_desc_init(kind=kind, M=64, H=8192, F=F, tile_m=128, tile_n=64, tuned=-1)
        q = cs.cs_chain_plan_info(d, 152)
        assert q["tile_n"][:2] == [64 if kind == "gelu" else 128, 64] and q["n_tiles"][:2] == [n0, 128]
    for tm in (256, 512):
        with pytest.raises(cs.CSError) as e:
            cs.cs_schedule_build(cs.cs_chain_desc_init(M=1024, H=8192, F=8192, tile_m=tm, tile_n=64), 152)
        assert e.value.status == cs.CS_ERR_UNSUPPORTED
    with pytest.raises(cs.CSError) as e:
        cs.cs_schedule_build(cs.cs_chain_desc_init(kind="attn", M=64, H=1024, F=512, heads=4, head_dim=128,
                                                   tile_m=128, tile_n=64), 152)
    assert e.value.status == cs.CS_ERR_UNSUPPORTED
    for M in (1, 64, 1024, 8192):
        for kind in ("gelu", "swiglu"):
            q = cs.cs_chain_plan_info(cs.cs_chain_desc_init(kind=kind, M=M, H=8192, F=2752, tuned=-1), 152)
            assert 64 not in q["tile_n"]


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
    dec = [cs.decode_unit(u)[:3] for u in cs.cs_schedule_build(d, 148)]
    # first group of producers: (n, m) with m fastest
    assert dec[:8] == [(0, 0, 0), (0, 1, 0), (0, 2, 0), (0, 3, 0), (0, 0, 1), (0, 1, 1), (0, 2, 1), (0, 3, 1)]
    # then the second producer group, then the first consumer group
    assert dec[192] == (0, 4, 0) and dec[384] == (1, 0, 0)


def test_row_major_raster_completes_rows_in_turn(cs):
    d = cs.cs_chain_desc_init(M=1024, H=12288, F=6144, group_m=4, lag=1, tile_n=256, tile_m=256, raster=2)
    dec = [cs.decode_unit(u)[:3] for u in cs.cs_schedule_build(d, 152)]
    assert dec[:25] == [(0, 0, n) for n in range(24)] + [(0, 1, 0)]


def test_auto_tile_shape(cs):
    def units(M):
        return len(cs.cs_schedule_build(cs.cs_chain_desc_init(M=M, H=12288, F=6144, split_k=1), 148))
    assert units(2048) == 4 * 24 + 4 * 48   # 512 x 256 tiles: two CTA pairs sharing weight boxes
    assert units(1536) == 3 * 24 + 3 * 48
    assert units(1280) == 5 * 24 + 5 * 48   # 256 x 256 pairs where 512 rows would add padding
    assert units(640) == 5 * 24 + 5 * 48    # 128 x 256 tiles on single SMs in between
    assert units(256) == 1 * 24 + 1 * 48    # two row blocks: one 256 x 256 pair tile row
    assert units(128) == 1 * 48 + 1 * 96    # one row block: 128 x 128 tiles
    # SwiGLU (gate|up split over each pair): 512 x 256 tiles from M = 512, padding or not
    swiglu = cs.cs_chain_desc_init(kind="swiglu", M=768, H=8192, F=2752, split_k=1)
    assert len(cs.cs_schedule_build(swiglu, 148)) == 2 * 22 + 2 * 32


def test_pair_tiles_need_wide_gelu_tiles(cs):
    d = cs.cs_chain_desc_init(M=512, H=512, F=512, tile_m=256, tile_n=128)
    with pytest.raises(cs.CSError) as e:
        cs.cs_schedule_build(d, 148)
    assert e.value.status == cs.CS_ERR_UNSUPPORTED


def test_the_abi_from_plain_c99(cs, tmp_path):
    """tests/c/abi_host_check.c includes only include/cs_chain.h, compiles as
    strict C99 and links the library: the boundary is a C ABI, usable without
    Python (host-only entry points, no GPU)."""
    import shutil
    import subprocess
    gcc = shutil.which("gcc")
    if gcc is None:
        pytest.skip("no C compiler")
    libdir = os.path.dirname(cs.chain.LIB_PATH)
    exe = str(tmp_path / "abi_host_check")
    subprocess.run([gcc, "-std=c99", "-Wall", "-Wextra", "-pedantic", "-Werror", "-I", os.path.join(ROOT, "include"),
                    os.path.join(ROOT, "tests", "c", "abi_host_check.c"), "-o", exe, "-L", libdir, "-lcs_chain",
                    f"-Wl,-rpath,{libdir}"], check=True)
    p = subprocess.run([exe, cs.chain.TUNE_TABLE], capture_output=True, text=True, timeout=60)
    assert p.returncode == 0 and p.stdout.strip() == "ok", p.stderr


def _loop_order(stages, m_tiles, group_m, lag, n_tiles, splits, row_major, kv=0, ks_major=False):
    """The fused dispatch order written as nested loops (steps, stages, a
    group's tiles), independently of the library's closed form.  kv > 0: the
    attention stage's units of tile row m are ceil((m + 1) / kv) key-range
    pieces per head, listed row by row, head, then piece.  ks_major: a split
    stage after the first lists K-split, then column tile, then row."""
    groups = -(-m_tiles // group_m)
    out = []
    for t in range(groups + (stages - 1) * lag):
        for s in range(stages):
            g = t - s * lag
            if not 0 <= g < groups:
                continue
            rows = range(g * group_m, min(m_tiles, (g + 1) * group_m))
            if kv > 0 and stages == 3 and s == 1:
                out += [(s, m, n, k) for m in rows for n in range(n_tiles[s]) for k in range(-(-(m + 1) // kv))]
            elif row_major:
                out += [(s, m, n, k) for m in rows for n in range(n_tiles[s]) for k in range(splits[s])]
            elif ks_major and s > 0:
                out += [(s, m, n, k) for k in range(splits[s]) for n in range(n_tiles[s]) for m in rows]
            else:
                out += [(s, m, n, k) for n in range(n_tiles[s]) for m in rows for k in range(splits[s])]
    return out


_ORDER_CASES = [
    ("gelu", 2048, 12288, 6144, -1, 0, 0, 0, 0), ("gelu", 1, 12288, 6144, -1, 0, 0, 0, 0),
    ("gelu", 1000, 8192, 2752, 2, 1, 2, 128, 1), ("gelu", 1536, 8192, 8192, 5, 5, 1, 256, 2),
    ("swiglu", 777, 8192, 2752, 0, 3, 3, 128, 2), ("gelu", 130000, 256, 512, 3, 7, 1, 128, 1),
    ("attn", 2048, 12288, 1536, -1, 0, 0, 256, 0), ("attn", 300, 12288, 1536, 2, 1, 0, 128, 2),
    ("attn", 2048, 12288, 1536, -1, 3, 0, 128, 0), ("attn", 1900, 1024, 512, 1, 2, 0, 256, 2),
    ("attn", 640, 1024, 256, 0, 1, 0, 128, 0),
    # K-range-major split consumers
    ("gelu", 1, 12288, 6144, -1, 0, 6, 0, 3), ("swiglu", 16, 8192, 2752, -1, 0, 4, 128, 3),
    ("gelu", 1000, 8192, 2752, 2, 1, 2, 128, 3), ("gelu", 700, 4096, 1024, 1, 2, 3, 256, 3),
    ("attn", 16, 12288, 1536, -1, 0, 3, 128, 3), ("attn", 900, 1024, 512, 1, 2, 2, 256, 3)]


# attention cases also with key-range pieces: auto, every group alone, three groups
@pytest.mark.parametrize("kind,M,H,F,lag,group,split,tile_m,raster,kv",
                         [c + (kv,) for c in _ORDER_CASES for kv in ((-1, 0, 1, 3) if c[0] == "attn" else (-1,))])
def test_closed_form_schedule_equals_the_loop_order(cs, kind, M, H, F, lag, group, split, tile_m, raster, kv):
    """The schedule entries are computed one by one from a closed form (so the
    allocation-free forward can write them on the device, one thread each):
    they must equal the nested-loop order entry for entry."""
    extra = dict(heads=F // 128, head_dim=128, kv_chunk=kv) if kind == "attn" else {}
    d = cs.cs_chain_desc_init(kind=kind, M=M, H=H, F=F, lag=lag, group_m=group, split_k=split, tile_m=tile_m,
                              raster=raster, weight_layout="nk", tuned=-1, **extra)
    q = cs.cs_chain_plan_info(d, 152)
    m_tiles = -(-M // q["tile_m"])
    if kind == "attn":
        want_kv = max(kv, -(-m_tiles // 15)) if kv > 0 else 0  # auto: whole rows
        assert q["kv_chunk"] == (want_kv if want_kv < m_tiles else 0)
    want = _loop_order(q["stages"], m_tiles, q["group_m"], q["lag"], q["n_tiles"], q["split_k"], raster == 2,
                       q.get("kv_chunk", 0), raster == 3)
    assert q["raster"] == (raster or 1)
    got = [cs.decode_unit(u) for u in cs.cs_schedule_build(d, 152)]
    assert got == [(s, m, n, k) for s, m, n, k in want]
    assert q["n_units"] == len(got)
    for s in range(q["stages"]):
        assert q["sched_units"][s] == sum(1 for e in got if e[0] == s)


def _sk_pieces(u, q, K, tiles):
    """(tile, first slice, end slice, contributor, contributors) of Stream-K unit u."""
    a, b = u * q, min(tiles * K, (u + 1) * q)
    out = []
    for j in range(a // K, (b - 1) // K + 1):
        first, last = (j * K) // q, ((j + 1) * K - 1) // q
        out.append((j, max(a, j * K) - j * K, min(b, (j + 1) * K) - j * K, u - first, last - first + 1))
    return out


@pytest.mark.parametrize("M,H,F,tile_m,sk_tiles,sk_units", [
    (1024, 8192, 8192, 512, 14, 0), (1024, 8192, 8192, 512, 52, 0), (896, 8192, 8192, 512, 100, 0),
    (1536, 8192, 8192, 256, 20, 76), (700, 1024, 2048, 128, 9, 40), (300, 512, 1024, 128, 3, 1000)])
def test_stream_k_tail_schedule(cs, M, H, F, tile_m, sk_tiles, sk_units):
    """The last sk_tiles tiles of the last stage leave the dispatch order and
    Stream-K units (K-split field 15) take their place at its end; their K
    ranges cover every K-slice of those tiles exactly once, each unit's share
    is contiguous and at least 8 slices (or all of a shorter K), and each
    tile's contributors are numbered in K order."""
    d = cs.cs_chain_desc_init(M=M, H=H, F=F, tile_m=tile_m, tile_n=256 if tile_m > 128 else 128,
                              sk_tiles=sk_tiles, sk_units=sk_units, weight_layout="nk", tuned=-1)
    q = cs.cs_chain_plan_info(d, 152)
    K = -(-F // 64)  # K-slices of the last stage (H = X W2: K = F)
    tn = q["tile_n"][1]
    last_group_tiles = (-(-M // tile_m) - (q["group_m"] * (-(-(-(-M // tile_m)) // q["group_m"]) - 1))) * -(-H // tn)
    assert q["sk_tiles"] == min(sk_tiles, last_group_tiles)
    assert q["sk_q"] >= min(8, K)
    plain = cs.cs_chain_desc_init(M=M, H=H, F=F, tile_m=tile_m, tile_n=d.tile_n, sk_tiles=-1, weight_layout="nk",
                                  tuned=-1)
    base = [cs.decode_unit(u) for u in cs.cs_schedule_build(plain, 152)]
    got = [cs.decode_unit(u) for u in cs.cs_schedule_build(d, 152)]
    t, U = q["sk_tiles"], q["sk_units"]
    assert got[:len(base) - t] == base[:len(base) - t]
    assert got[len(base) - t:] == [(1, 0, u, 15) for u in range(U)]
    assert q["n_units"] == len(got)
    assert all(s == 1 and k == 0 for s, _, _, k in base[len(base) - t:])  # the replaced entries: last-stage tiles
    cover = {}
    for u in range(U):
        pieces = _sk_pieces(u, q["sk_q"], K, t)
        assert sum(e - b for _, b, e, _, _ in pieces) == min(q["sk_q"], t * K - u * q["sk_q"])
        for j, b, e, c, nc in pieces:
            assert 0 <= b < e <= K and 0 <= c < nc
            cover.setdefault(j, []).append((b, e, c, nc))
    for j in range(t):
        parts = sorted(cover[j])
        assert parts[0][0] == 0 and parts[-1][1] == K
        assert all(a[1] == b[0] for a, b in zip(parts, parts[1:]))  # contiguous, no overlap
        assert [c for _, _, c, _ in parts] == list(range(len(parts)))
        assert all(nc == len(parts) for _, _, _, nc in parts)


def test_stream_k_with_automatic_splits_leaves_the_last_stage_unsplit(cs):
    """At small M the automatic rule splits every stage; asking for a Stream-K
    tail with split_k 0 keeps the producers' splits and leaves the last stage
    unsplit, its tiles shared out as Stream-K units."""
    for kind, H, F, M in (("gelu", 12288, 6144, 1), ("swiglu", 8192, 2752, 16), ("gelu", 12288, 6144, 256)):
        plain = cs.cs_chain_plan_info(cs.cs_chain_desc_init(kind=kind, M=M, H=H, F=F, tuned=-1), 152)
        assert plain["split_k"][1] > 1
        d = cs.cs_chain_desc_init(kind=kind, M=M, H=H, F=F, tuned=-1, sk_tiles=4096)
        q = cs.cs_chain_plan_info(d, 152)
        assert q["split_k"][0] == plain["split_k"][0] and q["split_k"][1] == 1
        assert q["sk_tiles"] == q["n_tiles"][1] * -(-M // q["tile_m"]) and q["sk_units"] > 0
        units = [cs.decode_unit(u) for u in cs.cs_schedule_build(d, 152)]
        assert sum(1 for s, _, _, k in units if s == 1 and k == 15) == q["sk_units"]


def test_stream_k_needs_an_unsplit_last_stage(cs):
    d = cs.cs_chain_desc_init(M=64, H=4096, F=4096, split_k=4, sk_tiles=8, tuned=-1)
    q = cs.cs_chain_plan_info(d, 152)
    assert q["split_k"][1] == 4 and q["sk_tiles"] == 0 and q["sk_units"] == 0
    for field, value in (("sk_tiles", -2), ("sk_tiles", 70000), ("sk_units", -1), ("sk_units", 20000)):
        bad = cs.cs_chain_desc_init(M=64, H=256, F=1024)
        setattr(bad, field, value)
        with pytest.raises(cs.CSError) as e:
            cs.cs_chain_plan_info(bad, 152)
        assert e.value.status == cs.CS_ERR_INVALID_ARG


def test_attention_piece_bounds(cs):
    """kv_chunk is refused outside -1..4095, raised so that no row has more than
    15 pieces (the unit's K-split field), and pieces never cover a whole row."""
    for v in (-2, 4096):
        d = cs.cs_chain_desc_init(kind="attn", M=2048, H=12288, F=1536, heads=12, head_dim=128, kv_chunk=v)
        with pytest.raises(cs.CSError) as e:
            cs.cs_chain_plan_info(d, 152)
        assert e.value.status == cs.CS_ERR_INVALID_ARG
    d = cs.cs_chain_desc_init(kind="attn", M=128 * 40, H=1024, F=256, heads=2, head_dim=128, tile_m=128, kv_chunk=1)
    q = cs.cs_chain_plan_info(d, 152)
    assert q["kv_chunk"] == 3  # ceil(40 / 15)
    assert max(cs.decode_unit(u)[3] for u in cs.cs_schedule_build(d, 152) if cs.decode_unit(u)[0] == 1) == 13
    for M, kv in ((512, 2), (512, 5), (128, 1)):  # two 256-row tile rows, one 128-row row: nothing to split
        d = cs.cs_chain_desc_init(kind="attn", M=M, H=1024, F=256, heads=2, head_dim=128, kv_chunk=kv)
        assert cs.cs_chain_plan_info(d, 152)["kv_chunk"] == 0
