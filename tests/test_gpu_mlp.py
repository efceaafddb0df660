"""GPU parity of the fused MLP chain against the fp64 oracle, through the C ABI.

Bar: max|gpu - oracle| / max|oracle| <= 5e-3 (fp16/bf16 inputs, fp32
accumulate, intermediate rounded to the input dtype).  Outputs of every sync
policy are compared with one another bit for bit: tile synchronisation only
changes when a consumer tile runs, never what it computes.
"""
from __future__ import annotations

import numpy as np
import pytest
import torch

import cs_inputs
import oracle
from tests.gpu_util import TOL, device_tensors, forward, intermediate, plan_for

pytestmark = pytest.mark.gpu

cs = pytest.importorskip("consumer_gemm_chain_gb300")


def _oracle(inp, rows=None):
    X = inp.X if rows is None else inp.X[rows]
    if inp.kind == "gelu":
        return oracle.mlp_gelu(X, inp.W1, inp.b1, inp.W2, return_hidden=True)
    return oracle.mlp_swiglu(X, inp.Wg, inp.Wu, inp.W2, return_hidden=True)


def test_tiny_chain_tile_sync():
    inp = cs_inputs.make_inputs("tiny", seed=0)
    dev = device_tensors(inp)
    with plan_for(inp, "tile") as plan:
        Y = forward(plan, dev)
        H = intermediate(plan, 0, inp.M, inp.F, inp.dtype)
    Yref, Href = _oracle(inp)
    assert oracle.rel_err(H.cpu(), Href) <= TOL
    assert oracle.rel_err(Y.cpu(), Yref) <= TOL


def test_tiny_chain_golden_values():
    from tests.test_golden import load_tiny_golden
    inp = cs_inputs.make_inputs("tiny", seed=0)
    dev = device_tensors(inp)
    with plan_for(inp, "tile") as plan:
        Y = forward(plan, dev).double().cpu().numpy()
    g = load_tiny_golden()
    ref = np.array([v for _, _, v in g])
    got = np.array([Y[r, c] for r, c, _ in g])
    full_ref = _oracle(inp)[0]
    assert np.max(np.abs(got - ref)) <= TOL * np.max(np.abs(full_ref))


# (tile_m, tile_n): 256 rows = a 2-SM pair; 512 rows = two pairs in a 4-CTA
# cluster sharing every weight box by multicast
TILES = [(128, 128), (128, 256), (256, 256), (512, 256)]


@pytest.mark.parametrize("tile_m,tile_n", TILES)
@pytest.mark.parametrize("layout", ["kn", "nk"])
@pytest.mark.parametrize("dtype", [torch.float16, torch.bfloat16])
@pytest.mark.parametrize("M,H,F", [(1, 256, 1024), (100, 320, 392), (200, 200, 136), (384, 512, 640),
                                   (129, 1024, 2752), (700, 264, 520)])
def test_ragged_shapes(M, H, F, dtype, layout, tile_m, tile_n):
    inp = cs_inputs.make_custom("gelu", M, H, F, dtype=dtype, seed=3)
    dev = device_tensors(inp, layout)
    with plan_for(inp, "tile", layout, tile_n=tile_n, tile_m=tile_m) as plan:
        Y = forward(plan, dev)
    Yref, _ = _oracle(inp)
    assert oracle.rel_err(Y.cpu(), Yref) <= TOL


@pytest.mark.parametrize("tile_m,tile_n", TILES)
def test_policies_bit_identical_and_layouts_agree(tile_m, tile_n):
    inp = cs_inputs.make_custom("gelu", 300, 768, 1536, seed=5)
    outs = {}
    for layout in ("kn", "nk"):
        dev = device_tensors(inp, layout)
        for pol in ("tile", "row", "strided", "stream"):
            with plan_for(inp, pol, layout, tile_n=tile_n, tile_m=tile_m, group_m=1) as plan:
                outs[(layout, pol)] = forward(plan, dev).cpu()
    Yref, _ = _oracle(inp)
    base = outs[("kn", "tile")]
    assert oracle.rel_err(base, Yref) <= TOL
    for k, v in outs.items():
        assert torch.equal(v, base), f"{k} differs from kn/tile"


@pytest.mark.parametrize("tile_m,tile_n", TILES)
def test_flags_end_at_expected_counts(tile_m, tile_n):
    inp = cs_inputs.make_custom("gelu", 520, 512, 1280, seed=6)
    dev = device_tensors(inp)
    with plan_for(inp, "tile", tile_n=tile_n, tile_m=tile_m) as plan:
        q = cs.cs_chain_query(plan)
        Y = torch.empty_like(dev["X"])
        for e in range(1, 6):
            forward(plan, dev, Y)
            tiles, rows, epoch = cs.cs_chain_debug_read_sems(plan, 0)
            assert epoch == e
            assert all(v == e for r in tiles for v in r), tiles
            assert rows == [e * q["n_tiles"][0]] * q["m_tiles"]


def test_policies_and_control_keep_flags_consistent():
    inp = cs_inputs.make_custom("gelu", 256, 512, 512, seed=7)
    dev = device_tensors(inp)
    for pol in ("row", "strided", "stream"):
        with plan_for(inp, pol, tile_n=128) as plan:
            for _ in range(3):
                forward(plan, dev)
            tiles, rows, epoch = cs.cs_chain_debug_read_sems(plan, 0)
            assert epoch == 3 and all(v == 3 for r in tiles for v in r) and rows == [3 * 4] * 2


def poisoned_forward(plan, dev, Y=None):
    """A forward whose plan-owned intermediate (and split-K partials) hold NaN
    when it starts: every element a consumer reads before its producer has
    stored and released it is NaN, and NaN reaches the output through the
    MMA, so one premature read anywhere turns Y NaN."""
    cs.cs_chain_debug_poison_intermediate(plan, -1)
    Y = forward(plan, dev, Y)
    return Y


def test_poison_reaches_a_consumer_that_reads_without_its_producer():
    """The positive control of the poisoned delay tests: the consumer stage run
    alone after a poison (no producer in between) reads NaN and writes NaN."""
    inp = cs_inputs.make_custom("gelu", 300, 512, 1024, seed=12)
    dev = device_tensors(inp)
    with plan_for(inp, "tile") as plan:
        good = forward(plan, dev).cpu()
        assert not torch.isnan(good).any()
        cs.cs_chain_debug_poison_intermediate(plan, 0)
        Y = torch.zeros_like(dev["X"])
        cs.cs_chain_forward_stage(plan, 1, Y=Y, **dev)
        torch.cuda.synchronize()
        assert torch.isnan(Y.cpu()).all(dim=1).all()  # every row read poisoned K-slices
        assert torch.equal(poisoned_forward(plan, dev).cpu(), good)


@pytest.mark.parametrize("tile_m,tile_n", TILES)
def test_delay_injection_never_changes_a_bit(tile_m, tile_n):
    """Random producer delays (up to 200 us) before each release, the
    intermediate poisoned before every forward: a consumer that loaded any
    K-slice before its producer tile was released would produce NaN."""
    inp = cs_inputs.make_custom("gelu", 640, 1024, 2048, seed=8)
    dev = device_tensors(inp)
    ref = None
    for pol in ("tile", "row", "strided"):
        with plan_for(inp, pol, tile_n=tile_n, tile_m=tile_m, group_m=1) as plan:
            q = cs.cs_chain_query(plan)
            for seed in range(3):
                g = torch.Generator().manual_seed(100 + seed)
                delays = (torch.rand(q["units"][0], generator=g) * 200_000).to(torch.int64).tolist()
                cs.cs_chain_debug_set_delays(plan, 0, delays)
                Y = poisoned_forward(plan, dev).cpu()
                assert not torch.isnan(Y).any(), (pol, seed)
                if ref is None:
                    ref = Y
                    Yref, _ = _oracle(inp)
                    assert oracle.rel_err(Y, Yref) <= TOL
                assert torch.equal(Y, ref), (pol, seed)
            cs.cs_chain_debug_set_delays(plan, 0, None)
            tiles, rows, epoch = cs.cs_chain_debug_read_sems(plan, 0)
            assert epoch == 3 and all(v == 3 for r in tiles for v in r)


@pytest.mark.parametrize("tile_m,tile_n,split", [(128, 128, 1), (256, 256, 2), (512, 256, 1), (128, 256, 3)])
@pytest.mark.parametrize("policy", ["tile", "row", "strided", "stream"])
def test_epoch_counters_wrap_at_two_to_the_32(policy, tile_m, tile_n, split):
    """Semaphores are epoch-counted and never reset: a forward waits for
    counts of epoch + 1 (times the tiles per row block, or the splits per tile),
    compared modulo 2^32.  Seeded two forwards before the wrap, four forwards
    (with the output released per tile too) cross it: every counter ends at its
    expected value modulo 2^32 and every output has the bits of a fresh plan."""
    inp = cs_inputs.make_custom("gelu", 520, 2048, 1280, seed=13)
    dev = device_tensors(inp, "nk")
    kw = dict(tile_m=tile_m, tile_n=tile_n, split_k=split, out_release=1)
    with plan_for(inp, policy, "nk", **kw) as fresh:
        ref = forward(fresh, dev).cpu()
    with plan_for(inp, policy, "nk", **kw) as plan:
        q = cs.cs_chain_query(plan)
        assert q["split_k"][0] == split
        start = 0xFFFFFFFE
        cs.cs_chain_debug_set_epoch(plan, start)
        for i in range(1, 5):
            Y = poisoned_forward(plan, dev).cpu()
            assert torch.equal(Y, ref), i
            e = (start + i) & 0xFFFFFFFF
            for b in (0, 1):  # the intermediate's counters, then the output's
                tiles, rows, epoch = cs.cs_chain_debug_read_sems(plan, b)
                assert epoch == e
                assert all(v == e for r in tiles for v in r), (i, b)
                assert rows == [(e * q["n_tiles"][b]) & 0xFFFFFFFF] * q["m_tiles"], (i, b)


@pytest.mark.parametrize("tile_m,tile_n", TILES)
def test_missing_release_times_out_and_reset_recovers(tile_m, tile_n):
    inp = cs_inputs.make_custom("gelu", 256, 512, 512, seed=9)
    dev = device_tensors(inp)
    with plan_for(inp, "tile", spin_timeout_ns=20_000_000, tile_m=tile_m, tile_n=tile_n) as plan:
        good = forward(plan, dev).cpu()
        cs.cs_chain_debug_skip_release(plan, 0, 1)
        Y = torch.empty_like(dev["X"])
        cs.cs_mlp_forward(plan, Y=Y, **dev)
        torch.cuda.synchronize()
        assert cs.cs_chain_status(plan) == cs.CS_ERR_TIMEOUT
        with pytest.raises(cs.CSError) as e:
            cs.cs_mlp_forward(plan, Y=Y, **dev)
        assert e.value.status == cs.CS_ERR_NEEDS_RESET
        cs.cs_chain_debug_skip_release(plan, 0, -1)
        cs.cs_chain_reset(plan)
        again = forward(plan, dev).cpu()
        assert torch.equal(again, good)
        tiles, rows, epoch = cs.cs_chain_debug_read_sems(plan, 0)
        assert epoch == 1 and all(v == 1 for r in tiles for v in r)


@pytest.mark.parametrize("tile_m,tile_n", TILES)
def test_forward_stage_matches_chain(tile_m, tile_n):
    inp = cs_inputs.make_custom("gelu", 300, 512, 1024, seed=10)
    dev = device_tensors(inp)
    with plan_for(inp, "tile", tile_m=tile_m, tile_n=tile_n) as plan:
        Y = forward(plan, dev).clone()
        H = intermediate(plan, 0, inp.M, inp.F, inp.dtype).clone()
        Y2 = torch.zeros_like(Y)
        cs.cs_chain_forward_stage(plan, 0, Y=Y2, **dev)
        cs.cs_chain_forward_stage(plan, 1, Y=Y2, **dev)
        torch.cuda.synchronize()
        assert cs.cs_chain_status(plan) == cs.CS_OK
        assert torch.equal(intermediate(plan, 0, inp.M, inp.F, inp.dtype), H)
        assert torch.equal(Y2, Y)
        _, _, epoch = cs.cs_chain_debug_read_sems(plan, 0)
        assert epoch == 1


def test_shape_and_dtype_checks_in_binding():
    inp = cs_inputs.make_custom("gelu", 64, 256, 512, seed=11)
    dev = device_tensors(inp)
    with plan_for(inp, "tile") as plan:
        with pytest.raises(ValueError):
            cs.cs_mlp_forward(plan, Y=torch.empty(64, 256, dtype=torch.bfloat16, device="cuda"), **dev)
        bad = dict(dev)
        bad["W1"] = dev["W1"].t()
        with pytest.raises(ValueError):
            cs.cs_mlp_forward(plan, Y=torch.empty_like(dev["X"]), **bad)


@pytest.mark.parametrize("M", cs_inputs.GPT3_M_SWEEP)
def test_gpt3_shard_sampled_rows(M):
    inp = cs_inputs.make_inputs("gpt3", M=M, seed=0)
    dev = device_tensors(inp)
    with plan_for(inp, "tile") as plan:  # the bench configuration (auto tile width, grouping)
        Y = forward(plan, dev).cpu()
    rows = cs_inputs.sample_rows(M, 64)
    Yref, _ = _oracle(inp, rows)
    assert oracle.rel_err(Y[rows], Yref) <= TOL


@pytest.mark.parametrize("M", [1024, 1536, 2048])
def test_gpt3_shard_two_pair_clusters(M):
    """512-row tiles (two 2-SM pairs per 4-CTA cluster, weight boxes multicast)
    on the full GPT-3 shard: sampled rows against the oracle, and the same bits
    as the 256-row pair tiles (same K order per output element)."""
    inp = cs_inputs.make_inputs("gpt3", M=M, seed=0)
    dev = device_tensors(inp)
    outs = {}
    for tm in (256, 512):
        with plan_for(inp, "tile", tile_m=tm, tile_n=256) as plan:
            assert cs.cs_chain_query(plan)["tile_m"] == tm
            outs[tm] = forward(plan, dev).cpu()
    rows = cs_inputs.sample_rows(M, 64)
    Yref, _ = _oracle(inp, rows)
    assert oracle.rel_err(outs[512][rows], Yref) <= TOL
    assert torch.equal(outs[512], outs[256])


@pytest.mark.parametrize("M", [128 * 3, 128 * 7, 128 * 12])
def test_stress_shape_all_policies(M):
    inp = cs_inputs.make_inputs("stress", M=M, seed=0)
    rows = cs_inputs.sample_rows(M, 32)
    Yref, _ = _oracle(inp, rows)
    dev = device_tensors(inp)
    base = None
    for pol in ("tile", "row", "strided", "stream"):
        with plan_for(inp, pol) as plan:
            Y = forward(plan, dev).cpu()
        if base is None:
            base = Y
            assert oracle.rel_err(Y[rows], Yref) <= TOL
        assert torch.equal(Y, base), pol


@pytest.mark.parametrize("split", [2, 3, 5])
@pytest.mark.parametrize("tile_m,tile_n", TILES)
@pytest.mark.parametrize("M,H,F", [(1, 1024, 1024), (200, 968, 392), (300, 2048, 1280)])
def test_split_k_parity(M, H, F, tile_m, tile_n, split):
    inp = cs_inputs.make_custom("gelu", M, H, F, seed=51)
    dev = device_tensors(inp, "nk")
    with plan_for(inp, "tile", "nk", tile_m=tile_m, tile_n=tile_n, split_k=split) as plan:
        q = cs.cs_chain_query(plan)
        assert q["split_k"][0] > 1
        Y1 = forward(plan, dev).cpu()
        H1 = intermediate(plan, 0, inp.M, inp.F, inp.dtype).cpu()
        Y2 = forward(plan, dev).cpu()
        tiles, rows, epoch = cs.cs_chain_debug_read_sems(plan, 0)
        assert epoch == 2 and all(v == 2 for r in tiles for v in r)
    Yref, Href = _oracle(inp)
    assert oracle.rel_err(H1, Href) <= TOL
    assert oracle.rel_err(Y1, Yref) <= TOL
    assert torch.equal(Y1, Y2)  # fixed split order: the same bits every time


@pytest.mark.parametrize("kind,M,H,F,split", [
    ("gelu", 24, 8192, 256, 12),    # cooperative reduction, 9..15 splits
    ("gelu", 32, 4096, 512, 7),     # cooperative, 5..8 splits, 32 valid rows
    ("gelu", 1, 2048, 384, 3),      # cooperative, a single row
    ("gelu", 17, 2048, 384, 2),     # cooperative, two splits
    ("gelu", 40, 8192, 256, 12),    # 40 rows: row per thread, the chunks shared by all four warps
    ("gelu", 48, 4096, 512, 3),     # 48 rows, shared
    ("gelu", 64, 4096, 512, 3),     # 64 rows, shared
    ("swiglu", 32, 2048, 256, 3),   # cooperative, gate and up parts
    ("swiglu", 33, 4096, 344, 6),   # 33 rows, shared, ragged F
    ("swiglu", 48, 2048, 256, 3),   # 48 rows, shared
    ("swiglu", 64, 2048, 256, 3),   # 64 rows, shared
    ("swiglu", 130, 2048, 256, 2),  # a full row block (row per thread), then a block of 2 rows
    ("gelu", 100, 2048, 384, 4),    # 100 rows: row per thread
])
def test_split_k_few_valid_rows(kind, M, H, F, split):
    """Ragged row blocks: partials are written for the valid rows only; the last
    split of a block of at most 32 valid rows reduces cooperatively (every
    epilogue thread fetches elements of every split) and stores its rows
    directly, a larger block sums row per thread (up to 64 rows with the chunks
    shared by all four warps); the result matches the oracle and is the same
    bits on every call."""
    inp = cs_inputs.make_custom(kind, M, H, F, dtype=torch.bfloat16, seed=54)
    dev = device_tensors(inp, "nk")
    with plan_for(inp, "tile", "nk", split_k=split) as plan:
        q = cs.cs_chain_query(plan)
        assert q["split_k"][0] == split
        Y1 = forward(plan, dev).cpu()
        H1 = intermediate(plan, 0, inp.M, inp.F, inp.dtype).cpu()
        Y2 = forward(plan, dev).cpu()
    Yref, Href = _oracle(inp)
    assert oracle.rel_err(H1, Href) <= TOL
    assert oracle.rel_err(Y1, Yref) <= TOL
    assert torch.equal(Y1, Y2)


def test_split_k_swiglu_and_policies():
    inp = cs_inputs.make_custom("swiglu", 100, 1024, 688, dtype=torch.bfloat16, seed=52)
    dev = device_tensors(inp, "nk")
    outs = {}
    for pol in ("tile", "row", "strided", "stream"):
        with plan_for(inp, pol, "nk", split_k=4, group_m=1) as plan:
            outs[pol] = forward(plan, dev).cpu()
    Yref, _ = _oracle(inp)
    assert oracle.rel_err(outs["tile"], Yref) <= TOL
    for k, v in outs.items():
        assert torch.equal(v, outs["tile"]), k


def test_split_k_delay_injection_never_changes_a_bit():
    inp = cs_inputs.make_custom("gelu", 64, 2048, 1024, seed=53)
    dev = device_tensors(inp, "nk")
    with plan_for(inp, "tile", "nk", split_k=4) as plan:
        q = cs.cs_chain_query(plan)
        ref = forward(plan, dev).cpu()
        for seed in range(3):
            g = torch.Generator().manual_seed(300 + seed)
            cs.cs_chain_debug_set_delays(plan, 0, (torch.rand(q["units"][0], generator=g) * 100_000).long().tolist())
            assert torch.equal(poisoned_forward(plan, dev).cpu(), ref), seed


@pytest.mark.parametrize("kind,M,H,F,split,first", [
    ("gelu", 1, 12288, 6144, 6, 6),    # GPT-3 shard at one row: producers in two waves
    ("gelu", 16, 4096, 2048, 3, 8),    # more producer splits than consumer splits
    ("swiglu", 16, 8192, 2752, 4, 6),  # LLaMA shard: gate and up, a ragged consumer K
    ("gelu", 200, 2048, 1024, 2, 4),   # two row blocks, row-per-thread reductions
])
def test_k_range_major_consumers_and_first_stage_splits(kind, M, H, F, split, first):
    """raster 3 lists a split consumer stage K-split by K-split, and
    split_k_first gives the producers their own split count: every consumer
    still waits for exactly the producer tiles of its K range (delayed
    producers, the intermediate poisoned before each forward), the output
    matches the oracle, and the order changes no bit (raster 1, same splits)."""
    inp = cs_inputs.make_custom(kind, M, H, F, seed=56)
    dev = device_tensors(inp, "nk")
    outs = {}
    for raster in (1, 3):
        with plan_for(inp, "tile", "nk", split_k=split, split_k_first=first, raster=raster) as plan:
            q = cs.cs_chain_query(plan)
            assert q["raster"] == raster and q["split_k"][:2] == [first, split]
            outs[raster] = poisoned_forward(plan, dev).cpu()
            if raster == 3:
                for seed in range(2):
                    g = torch.Generator().manual_seed(400 + seed)
                    delays = (torch.rand(q["units"][0], generator=g) * 100_000).long().tolist()
                    cs.cs_chain_debug_set_delays(plan, 0, delays)
                    assert torch.equal(poisoned_forward(plan, dev).cpu(), outs[3]), seed
    Yref, _ = _oracle(inp)
    assert oracle.rel_err(outs[3], Yref) <= TOL
    assert torch.equal(outs[1], outs[3])


@pytest.mark.parametrize("layout", ["nk", "kn"])
@pytest.mark.parametrize("kind,M,H,F,split,policy", [
    ("gelu", 1, 2048, 1024, 3, "tile"),     # up to 8 rows: the 17 KB-stage kernel, K-splits
    ("gelu", 100, 2048, 1152, 1, "tile"),   # ragged rows, unsplit
    ("gelu", 300, 1024, 640, 2, "row"),     # three row blocks, K-splits, RowSync
    ("gelu", 300, 1024, 640, 1, "strided"),
    ("gelu", 130, 1024, 640, 2, "stream"),  # the two-kernel control
    ("swiglu", 64, 2048, 688, 3, "tile"),   # 128-wide gate|up producer, 64-wide consumer tiles
])
def test_64_wide_tiles(kind, M, H, F, split, policy, layout):
    """64-column tiles on single SMs: the output matches the oracle and the
    128-wide tiles' (the same K order per element) to fp16 rounding, and
    delayed producers over a poisoned intermediate change no bit."""
    inp = cs_inputs.make_custom(kind, M, H, F, dtype=torch.bfloat16 if kind == "swiglu" else torch.float16, seed=59)
    dev = device_tensors(inp, layout)
    outs = {}
    for tn in (64, 128):
        with plan_for(inp, policy, layout, tile_m=128, tile_n=tn, split_k=split) as plan:
            q = cs.cs_chain_query(plan)
            assert q["tile_n"][1] == tn and q["tile_n"][0] == (128 if kind == "swiglu" else tn)
            outs[tn] = poisoned_forward(plan, dev).cpu()
            if tn == 64:
                g = torch.Generator().manual_seed(420)
                delays = (torch.rand(q["units"][0], generator=g) * 100_000).long().tolist()
                cs.cs_chain_debug_set_delays(plan, 0, delays)
                assert torch.equal(poisoned_forward(plan, dev).cpu(), outs[64])
    Yref, _ = _oracle(inp)
    assert oracle.rel_err(outs[64], Yref) <= TOL
    assert oracle.rel_err(outs[64], outs[128]) <= 1e-3


@pytest.mark.parametrize("layout", ["nk", "kn"])
@pytest.mark.parametrize("policy", ["row", "strided", "stream"])
def test_k_range_order_under_every_policy(policy, layout):
    """The K-range order is a dispatch order only: under RowSync, Strided and the
    two-kernel control, in both weight layouts, with the output release on,
    it gives raster 1's bits and the oracle's values, and every Y tile and row
    block is released once per forward."""
    inp = cs_inputs.make_custom("swiglu", 24, 4096, 2048, dtype=torch.bfloat16, seed=58)
    dev = device_tensors(inp, layout)
    outs = {}
    for raster in (1, 3):
        with plan_for(inp, policy, layout, split_k=3, split_k_first=5, raster=raster, out_release=1) as plan:
            q = cs.cs_chain_query(plan)
            assert q["raster"] == raster and q["split_k"][:2] == [5, 3]
            outs[raster] = poisoned_forward(plan, dev).cpu()
            assert torch.equal(poisoned_forward(plan, dev).cpu(), outs[raster])
            tiles, rows, epoch = cs.cs_chain_debug_read_sems(plan, 1)  # the output's counters
            assert epoch == 2 and all(v == 2 for r in tiles for v in r)
    Yref, _ = _oracle(inp)
    assert oracle.rel_err(outs[3], Yref) <= TOL
    assert torch.equal(outs[1], outs[3])


@pytest.mark.parametrize("policy", ["tile", "stream"])
def test_back_to_back_forwards_with_programmatic_launch(policy):
    """Forwards queued back to back (each one's output is the next one's input,
    no host synchronisation in between) give the same bits with programmatic
    dependent launch on and off: a grid reads global memory only after the
    grid before it has completed."""
    inp = cs_inputs.make_custom("gelu", 300, 1024, 768, seed=55)
    dev = device_tensors(inp, "nk")
    outs = {}
    for pdl in (1, -1):
        with plan_for(inp, policy, "nk", pdl=pdl) as plan:
            xs = [dev["X"].clone()]
            for _ in range(4):
                Y = torch.empty_like(xs[-1])
                cs.cs_mlp_forward(plan, X=xs[-1], W1=dev["W1"], b1=dev["b1"], W2=dev["W2"], Y=Y)
                xs.append(Y)
            torch.cuda.synchronize()
            assert cs.cs_chain_status(plan) == cs.CS_OK
            outs[pdl] = [x.cpu() for x in xs[1:]]
    Yref, _ = _oracle(inp)
    assert oracle.rel_err(outs[1][0], Yref) <= TOL
    for a, b in zip(outs[1], outs[-1]):
        assert torch.equal(a, b)


@pytest.mark.parametrize("kind,split", [("gelu", 2), ("gelu", 3), ("swiglu", 2)])
def test_split_consumers_wait_for_their_own_producer_tiles(kind, split):
    """A K-split consumer waits only for the producer tiles of its own K range.
    The intermediate still holds the previous input's values, so a consumer
    that read a tile too early would mix them in: with every producer delayed,
    the second input's output must equal an undelayed run of it."""
    a = cs_inputs.make_custom(kind, 64, 2048, 1536, seed=56)
    b = cs_inputs.make_custom(kind, 64, 2048, 1536, seed=57)
    dev_a = device_tensors(a, "nk")
    with plan_for(a, "tile", "nk", split_k=split) as plan:
        q = cs.cs_chain_query(plan)
        assert q["split_k"][0] == split and q["split_k"][1] == split
        clean_b = forward(plan, dict(dev_a, X=b.X.cuda())).cpu()
        forward(plan, dev_a)
        g = torch.Generator().manual_seed(58)
        cs.cs_chain_debug_set_delays(plan, 0, (torch.rand(q["units"][0], generator=g) * 300_000).long().tolist())
        delayed_b = forward(plan, dict(dev_a, X=b.X.cuda())).cpu()
    assert torch.equal(delayed_b, clean_b)


@pytest.mark.parametrize("kind,tile_n", [("gelu", 128), ("gelu", 256), ("swiglu", 0)])
@pytest.mark.parametrize("layout", ["nk", "kn"])
@pytest.mark.parametrize("M", [2, 5, 8])
def test_up_to_eight_rows_use_one_a_row_group(M, layout, kind, tile_n):
    """Up to 8 rows, a stage holds only the one 8-row group of A (the MMA reads it
    for all of its 128 rows; the rows past M are never stored), which leaves room
    for 11 (or 5 with 256 rows of B) stages of weights: parity against the oracle,
    every policy the same bits, producer delays change nothing."""
    inp = cs_inputs.make_custom(kind, M, 2048, 1280 if kind == "gelu" else 688, seed=59)
    dev = device_tensors(inp, layout)
    outs = {}
    for pol in ("tile", "row", "stream"):
        with plan_for(inp, pol, layout, tile_n=tile_n) as plan:
            q = cs.cs_chain_query(plan)
            outs[pol] = forward(plan, dev).cpu()
            if pol == "tile":
                g = torch.Generator().manual_seed(60)
                cs.cs_chain_debug_set_delays(plan, 0, (torch.rand(q["units"][0], generator=g) * 100_000).long().tolist())
                assert torch.equal(poisoned_forward(plan, dev).cpu(), outs[pol])
    Yref, _ = _oracle(inp)
    assert oracle.rel_err(outs["tile"], Yref) <= TOL
    for k, v in outs.items():
        assert torch.equal(v, outs["tile"]), k


@pytest.mark.parametrize("kind", ["gelu", "swiglu"])
def test_host_memory_forward_matches_device_forward(kind):
    """cs_mlp_forward_host: inputs and outputs in pinned host memory, four calls
    back to back with different inputs (the plan's two device buffers each serve
    two calls, the copies overlap the kernels); after the join every output
    equals the device-memory forward bit for bit."""
    inp = cs_inputs.make_custom(kind, 300, 1024, 768 if kind == "gelu" else 688, seed=61)
    dev = device_tensors(inp, "nk")
    wts = {k: v for k, v in dev.items() if k != "X"}
    g = torch.Generator().manual_seed(62)
    xs = [(torch.randn(inp.M, inp.H, generator=g) * 0.02).to(inp.dtype).pin_memory() for _ in range(4)]
    ys = [torch.full((inp.M, inp.H), float("nan"), dtype=inp.dtype).pin_memory() for _ in range(4)]
    with plan_for(inp, "tile", "nk") as plan:
        refs = [forward(plan, dict(dev, X=x.cuda())).cpu() for x in xs]
        for x, y in zip(xs, ys):
            cs.cs_mlp_forward_host(plan, X=x, Y=y, **wts)
        cs.cs_chain_host_join(plan)
        torch.cuda.synchronize()
        assert cs.cs_chain_status(plan) == cs.CS_OK
        for y, r in zip(ys, refs):
            assert torch.equal(y, r)
        with pytest.raises(ValueError):
            cs.cs_mlp_forward_host(plan, X=xs[0].cuda(), Y=ys[0], **wts)


REPLICA_CHECK = r"""
import sys, torch
sys.path.insert(0, sys.argv[1])
import consumer_gemm_chain_gb300 as cs, cs_inputs, oracle
from tests.gpu_util import device_tensors, forward, plan_for
assert cs.chain.LIB_PATH.endswith("libcs_chain_nomc.so"), cs.chain.LIB_PATH
assert cs.cs_library_features() & cs.CS_FEATURE_CLUSTER_MULTICAST == 0
inp = cs_inputs.make_custom("gelu", 1024, 512, 1024, seed=14)
dev = device_tensors(inp, "nk")
with plan_for(inp, "tile", "nk") as plan:
    tm = cs.cs_chain_query(plan)["tile_m"]
    Y = forward(plan, dev).cpu()
try:
    plan_for(inp, "tile", "nk", tile_m=512, tile_n=256)
    raise SystemExit("tile_m=512 accepted")
except cs.CSError as e:
    assert e.status == cs.CS_ERR_UNSUPPORTED
Yref = oracle.mlp_gelu(inp.X, inp.W1, inp.b1, inp.W2)
print(tm, oracle.rel_err(Y, Yref))
"""


def test_replica_build_runs_the_chain_without_multicast():
    """The replica build (no TMA cluster multicast; what N-rank processes load)
    in a process of its own: the shape that takes 512-row 4-CTA tiles in the
    full build runs on single-SM or 256-row pair tiles there, matches the
    oracle, and an explicit tile_m = 512 is refused."""
    import os
    import subprocess
    import sys
    root = os.path.dirname(os.path.dirname(os.path.abspath(__file__)))
    env = dict(os.environ, CS_CHAIN_LIBRARY="nomc")
    p = subprocess.run([sys.executable, "-c", REPLICA_CHECK, root], cwd=root, env=env, capture_output=True,
                       text=True, timeout=600)
    assert p.returncode == 0, p.stderr[-3000:]
    tm, err = p.stdout.split()[-2:]
    assert int(tm) in (128, 256)
    assert float(err) <= TOL
    full = cs.cs_chain_desc_init(kind="gelu", M=1024, H=512, F=1024, weight_layout="nk", tuned=-1)
    assert cs.cs_chain_plan_info(full, 152)["tile_m"] == 512  # this process: the full build


@pytest.mark.parametrize("kind,tile_m,tile_n,sk_tiles,sk_units", [
    ("gelu", 128, 128, 9, 40), ("gelu", 128, 256, 20, 0), ("gelu", 256, 256, 13, 76), ("gelu", 512, 256, 14, 0),
    ("gelu", 512, 256, 52, 0), ("swiglu", 512, 256, 20, 0), ("swiglu", 128, 128, 30, 7)])
def test_stream_k_tail(kind, tile_m, tile_n, sk_tiles, sk_units):
    """The last stage's trailing tiles shared out as Stream-K units (K ranges
    crossing tile boundaries, partial tiles summed in K order by the last
    contributor): parity with the oracle, the same bits under every policy
    (the two-kernel control's last launch carries the same tail), under
    producer delays with the intermediate and every partial poisoned, and
    across the 2^32 wrap of the arrival counters."""
    inp = cs_inputs.make_custom(kind, 1000, 1024, 2048 if kind == "gelu" else 1376, seed=15)
    dev = device_tensors(inp, "nk")
    kw = dict(tile_m=tile_m, tile_n=tile_n, sk_tiles=sk_tiles, sk_units=sk_units, group_m=1)
    outs = {}
    for pol in ("tile", "row", "strided", "stream"):
        with plan_for(inp, pol, "nk", **kw) as plan:
            q = cs.cs_chain_query(plan)
            assert q["sk_tiles"] > 0 and q["sk_units"] > 0, q
            outs[pol] = forward(plan, dev).cpu()
            if pol == "tile":
                g = torch.Generator().manual_seed(16)
                cs.cs_chain_debug_set_delays(plan, 0, (torch.rand(q["units"][0], generator=g) * 100_000).long().tolist())
                for _ in range(2):
                    assert torch.equal(poisoned_forward(plan, dev).cpu(), outs[pol])
                cs.cs_chain_debug_set_delays(plan, 0, None)
                cs.cs_chain_debug_set_epoch(plan, 0xFFFFFFFE)
                for _ in range(3):
                    assert torch.equal(poisoned_forward(plan, dev).cpu(), outs[pol])
    Yref, _ = _oracle(inp)
    assert oracle.rel_err(outs["tile"], Yref) <= TOL
    for k, v in outs.items():
        assert torch.equal(v, outs["tile"]), k
    with plan_for(inp, "tile", "nk", tile_m=tile_m, tile_n=tile_n, sk_tiles=-1, group_m=1) as plain:
        assert cs.cs_chain_query(plain)["sk_units"] == 0
        Yplain = forward(plain, dev).cpu()
    assert oracle.rel_err(outs["tile"], Yplain) <= 1e-3  # only the tail tiles' summation order differs


@pytest.mark.parametrize("M", [896, 1024, 1408, 1536])
def test_stream_k_on_the_stress_shape(M):
    inp = cs_inputs.make_inputs("stress", M=M, seed=0)
    dev = device_tensors(inp, "nk")
    rows = cs_inputs.sample_rows(M, 32)
    Yref, _ = _oracle(inp, rows)
    with plan_for(inp, "tile", "nk", sk_tiles=64, tuned=-1) as plan:
        q = cs.cs_chain_query(plan)
        assert q["sk_units"] > 0
        Y = poisoned_forward(plan, dev).cpu()
        assert torch.equal(poisoned_forward(plan, dev).cpu(), Y)
    assert oracle.rel_err(Y[rows], Yref) <= TOL
