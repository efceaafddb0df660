"""GPU parity of the attention chain (QKV GEMM -> causal attention -> Wo GEMM)
against the fp64 oracle, through the C ABI.

Stage by stage: the QKV intermediate, the attention output O and Y are each
compared with the oracle; outputs of every sync policy agree bit for bit, and
the semaphores of both boundaries end at their expected counts."""
from __future__ import annotations

import pytest
import torch

import cs_inputs
import oracle
from tests.gpu_util import TOL, device_tensors, forward, intermediate, plan_for

pytestmark = pytest.mark.gpu

cs = pytest.importorskip("consumer_gemm_chain_gb300")


def _oracle(inp):
    return oracle.attention_chain(inp.X, inp.Wqkv, inp.Wo, heads=inp.F // 128, head_dim=128, return_parts=True)


@pytest.mark.parametrize("tile_m", [128, 256])
@pytest.mark.parametrize("layout", ["nk", "kn"])
@pytest.mark.parametrize("M,H,heads", [(1, 256, 1), (100, 256, 2), (128, 512, 1), (300, 384, 3), (513, 256, 2)])
def test_attention_chain_parity(M, H, heads, layout, tile_m):
    """tile_m 256: 256 x 256 GEMM tiles and attention units of two query blocks
    on CTA pairs (each CTA holds half of every key block and half of V's head
    dimensions; S and O borrow a 256-column accumulator buffer)."""
    inp = cs_inputs.make_custom("attn", M, H, heads * 128, seed=31)
    dev = device_tensors(inp, layout)
    with plan_for(inp, "row", layout, tile_m=tile_m) as plan:
        assert cs.cs_chain_query(plan)["tile_m"] == tile_m
        Y = forward(plan, dev)
        QKV = intermediate(plan, 0, M, 3 * inp.F, inp.dtype)
        O = intermediate(plan, 1, M, inp.F, inp.dtype)
    Yref, QKVref, Oref = _oracle(inp)
    assert oracle.rel_err(QKV.cpu(), QKVref) <= TOL
    assert oracle.rel_err(O.cpu(), Oref) <= TOL
    assert oracle.rel_err(Y.cpu(), Yref) <= TOL


@pytest.mark.parametrize("tile_m", [128, 256])
def test_attention_policies_bit_identical_and_flags(tile_m):
    inp = cs_inputs.make_custom("attn", 520, 512, 256, seed=32)
    dev = device_tensors(inp, "nk")
    outs = {}
    for pol in ("tile", "row", "strided", "stream"):
        with plan_for(inp, pol, "nk", group_m=1, tile_m=tile_m) as plan:
            for _ in range(2):
                outs[pol] = forward(plan, dev).cpu()
            q = cs.cs_chain_query(plan)
            for b in (0, 1):
                tiles, rows, epoch = cs.cs_chain_debug_read_sems(plan, b)
                assert epoch == 2
                assert all(v == 2 for r in tiles for v in r)
                assert rows == [2 * q["n_tiles"][b]] * q["m_tiles"]
    Yref, _, _ = _oracle(inp)
    assert oracle.rel_err(outs["row"], Yref) <= TOL
    for k, v in outs.items():
        assert torch.equal(v, outs["row"]), k


@pytest.mark.parametrize("kv", [-1, 1])
@pytest.mark.parametrize("tile_m", [128, 256])
def test_attention_delay_injection_never_changes_a_bit(tile_m, kv):
    """Random delays before the QKV tiles' and the attention units' releases,
    QKV, O and the pieces' workspace poisoned with NaN before every forward: an
    attention unit that read a QKV row block, a Wo tile that read an O block,
    or a merging piece that read another piece's state, before it was released
    would turn Y NaN.  kv 1: every key group its own piece."""
    inp = cs_inputs.make_custom("attn", 400 if tile_m == 128 else 800, 512, 384, seed=33)
    dev = device_tensors(inp, "nk")
    ref = None
    for pol in ("row", "tile", "strided"):
        with plan_for(inp, pol, "nk", group_m=1, tile_m=tile_m, kv_chunk=kv) as plan:
            q = cs.cs_chain_query(plan)
            assert q["kv_chunk"] == (1 if kv == 1 else 0)
            for seed in range(2):
                g = torch.Generator().manual_seed(200 + seed)
                for stage in (0, 1):
                    d = (torch.rand(q["units"][stage], generator=g) * 200_000).to(torch.int64).tolist()
                    cs.cs_chain_debug_set_delays(plan, stage, d)
                cs.cs_chain_debug_poison_intermediate(plan, -1)
                Y = forward(plan, dev).cpu()
                assert not torch.isnan(Y).any(), (pol, seed)
                if ref is None:
                    ref = Y
                    Yref, _, _ = _oracle(inp)
                    assert oracle.rel_err(Y, Yref) <= TOL
                assert torch.equal(Y, ref), (pol, seed)


@pytest.mark.parametrize("tile_m", [128, 256])
def test_attention_poison_reaches_stages_run_without_producers(tile_m):
    """Positive control of the poisoned attention tests: run alone after a
    poison, the attention stage reads NaN QKV and the Wo stage NaN O."""
    inp = cs_inputs.make_custom("attn", 300, 512, 256, seed=35)
    dev = device_tensors(inp, "nk")
    with plan_for(inp, "row", "nk", tile_m=tile_m) as plan:
        good = forward(plan, dev).cpu()
        Y = torch.zeros_like(dev["X"])
        cs.cs_chain_debug_poison_intermediate(plan, 0)
        cs.cs_chain_forward_stage(plan, 1, Y=Y, **dev)  # attention from poisoned QKV
        O = intermediate(plan, 1, inp.M, inp.F, inp.dtype).cpu()
        assert torch.isnan(O).all()
        cs.cs_chain_debug_poison_intermediate(plan, 1)
        cs.cs_chain_forward_stage(plan, 2, Y=Y, **dev)  # Wo from poisoned O
        torch.cuda.synchronize()
        assert torch.isnan(Y.cpu()).all()
        assert torch.equal(forward(plan, dev).cpu(), good)


@pytest.mark.parametrize("kv", [-1, 1])
@pytest.mark.parametrize("tile_m", [128, 256])
@pytest.mark.parametrize("policy", ["row", "tile", "stream"])
def test_attention_epoch_counters_wrap(policy, tile_m, kv):
    """Both boundaries' counters (and the output's) across the 2^32 wrap; kv 1:
    also the pieces' arrival counters (a piece that miscounted would never
    merge, and the forward would time out)."""
    inp = cs_inputs.make_custom("attn", 300 if tile_m == 128 else 600, 512, 256, seed=36)
    dev = device_tensors(inp, "nk")
    with plan_for(inp, policy, "nk", tile_m=tile_m, out_release=1, kv_chunk=kv) as fresh:
        ref = forward(fresh, dev).cpu()
    with plan_for(inp, policy, "nk", tile_m=tile_m, out_release=1, kv_chunk=kv) as plan:
        q = cs.cs_chain_query(plan)
        start = 0xFFFFFFFF
        cs.cs_chain_debug_set_epoch(plan, start)
        for i in range(1, 4):
            cs.cs_chain_debug_poison_intermediate(plan, -1)
            assert torch.equal(forward(plan, dev).cpu(), ref), i
            assert cs.cs_chain_status(plan) == cs.CS_OK
            e = (start + i) & 0xFFFFFFFF
            for b in (0, 1, 2):
                tiles, rows, epoch = cs.cs_chain_debug_read_sems(plan, b)
                assert epoch == e and all(v == e for r in tiles for v in r), (i, b)
                assert rows == [(e * q["n_tiles"][b]) & 0xFFFFFFFF] * q["m_tiles"], (i, b)


@pytest.mark.parametrize("tile_m", [128, 256])
def test_attention_missing_release_times_out(tile_m):
    inp = cs_inputs.make_custom("attn", 256, 256, 256, seed=34)
    dev = device_tensors(inp, "nk")
    with plan_for(inp, "tile", "nk", spin_timeout_ns=20_000_000, tile_m=tile_m) as plan:
        good = forward(plan, dev).cpu()
        cs.cs_chain_debug_skip_release(plan, 1, 0)  # attention unit (block 0, head 0)
        Y = torch.empty_like(dev["X"])
        cs.cs_attn_chain_forward(plan, dev["X"], dev["Wqkv"], dev["Wo"], Y)
        torch.cuda.synchronize()
        assert cs.cs_chain_status(plan) == cs.CS_ERR_TIMEOUT
        cs.cs_chain_debug_skip_release(plan, 1, -1)
        cs.cs_chain_reset(plan)
        assert torch.equal(forward(plan, dev).cpu(), good)


@pytest.mark.parametrize("M", (1, 64, 512, 2048))
def test_gpt3_attention_shard(M):
    inp = cs_inputs.make_inputs("attn", M=M, seed=0)
    dev = device_tensors(inp, "nk")
    with plan_for(inp, "row", "nk") as plan:
        Y = forward(plan, dev).cpu()
    Yref, _, _ = _oracle(inp)
    assert oracle.rel_err(Y, Yref) <= TOL


@pytest.mark.parametrize("M,tile_m", [(16, 128), (300, 128), (600, 256)])
def test_attention_k_range_major_output_projection(M, tile_m):
    """raster 3 with split_k_first: the QKV GEMM takes its own (larger) split
    count and the split Wo stage runs K range by K range; with the QKV units
    delayed and QKV / O poisoned before every forward the output keeps its
    bits, equals raster 1 with the same splits, and matches the oracle."""
    inp = cs_inputs.make_custom("attn", M, 4096, 1024, seed=57)
    dev = device_tensors(inp, "nk")
    outs = {}
    for raster in (1, 3):
        with plan_for(inp, "row", "nk", tile_m=tile_m, split_k=2, split_k_first=4, raster=raster) as plan:
            q = cs.cs_chain_query(plan)
            assert q["raster"] == raster and q["split_k"] == [4, 1, 2]
            cs.cs_chain_debug_poison_intermediate(plan, -1)
            outs[raster] = forward(plan, dev).cpu()
            if raster == 3:
                g = torch.Generator().manual_seed(410)
                cs.cs_chain_debug_set_delays(plan, 0, (torch.rand(q["units"][0], generator=g) * 100_000).long().tolist())
                cs.cs_chain_debug_poison_intermediate(plan, -1)
                assert torch.equal(forward(plan, dev).cpu(), outs[3])
    Yref, _, _ = _oracle(inp)
    assert oracle.rel_err(outs[3], Yref) <= TOL
    assert torch.equal(outs[1], outs[3])


@pytest.mark.parametrize("M", (300, 1024, 2048))
def test_attention_pair_tiles_agree_with_single_sm_tiles(M):
    """128 x 128 single-SM tiles and 256 x 256 pair tiles (with two-query-block
    attention units) follow the same K order per output element but different
    tcgen05 instruction shapes, whose fp32 partial sums may round differently:
    the two outputs agree to a few fp16 ulps (a masking or indexing slip would
    show far above that) and each matches the oracle."""
    inp = cs_inputs.make_inputs("attn", M=M, seed=0)
    dev = device_tensors(inp, "nk")
    outs = {}
    for tm in (128, 256):
        with plan_for(inp, "row", "nk", tile_m=tm) as plan:
            outs[tm] = forward(plan, dev).cpu()
    Yref, _, _ = _oracle(inp)
    assert oracle.rel_err(outs[128], Yref) <= TOL
    assert oracle.rel_err(outs[256], Yref) <= TOL
    assert oracle.rel_err(outs[256], outs[128]) <= 1e-3


@pytest.mark.parametrize("tile_m", [128, 256])
def test_attention_stream_k_tail_on_the_output_projection(tile_m):
    inp = cs_inputs.make_custom("attn", 520, 512, 384, seed=37)
    dev = device_tensors(inp, "nk")
    outs = {}
    for pol in ("row", "tile", "stream"):
        with plan_for(inp, pol, "nk", tile_m=tile_m, sk_tiles=6, group_m=1) as plan:
            q = cs.cs_chain_query(plan)
            assert q["sk_units"] > 0
            cs.cs_chain_debug_poison_intermediate(plan, -1)
            outs[pol] = forward(plan, dev).cpu()
    Yref, _, _ = _oracle(inp)
    assert oracle.rel_err(outs["row"], Yref) <= TOL
    for k, v in outs.items():
        assert torch.equal(v, outs["row"]), k


@pytest.mark.parametrize("tile_m", [128, 256])
@pytest.mark.parametrize("M,heads,kv", [(700, 2, 1), (700, 2, 2), (1000, 1, 3), (1280, 3, 4), (2048, 2, 2)])
def test_attention_key_range_pieces(M, heads, kv, tile_m):
    """The causal units split into key-range pieces of kv key groups (tile_m
    keys each), merged by the last piece in piece order: O and Y against the
    oracle, against whole-row units (the merge reorders the fp32 sums, so to a
    few fp16 ulps, not bit for bit), and the same bits on a second forward and
    under another policy."""
    inp = cs_inputs.make_custom("attn", M, 384, heads * 128, seed=38)
    dev = device_tensors(inp, "nk")
    outs = {}
    for pol, k in (("row", kv), ("tile", kv), ("row", -1)):
        with plan_for(inp, pol, "nk", tile_m=tile_m, kv_chunk=k) as plan:
            q = cs.cs_chain_query(plan)
            m_tiles = -(-M // tile_m)
            if k == -1:
                assert q["kv_chunk"] == 0
            else:
                assert 0 < q["kv_chunk"] < m_tiles
                assert q["sched_units"][1] == heads * sum(-(-(m + 1) // q["kv_chunk"]) for m in range(m_tiles))
            cs.cs_chain_debug_poison_intermediate(plan, -1)
            Y = forward(plan, dev).cpu()
            O = intermediate(plan, 1, M, inp.F, inp.dtype).cpu()
            cs.cs_chain_debug_poison_intermediate(plan, -1)
            assert torch.equal(forward(plan, dev).cpu(), Y)
            outs[(pol, k)] = (Y, O)
    Yref, _, Oref = _oracle(inp)
    Y, O = outs[("row", kv)]
    assert oracle.rel_err(O, Oref) <= TOL
    assert oracle.rel_err(Y, Yref) <= TOL
    assert torch.equal(outs[("tile", kv)][0], Y)
    assert oracle.rel_err(O, outs[("row", -1)][1]) <= 1e-3
    assert oracle.rel_err(Y, outs[("row", -1)][0]) <= 1e-3


def _rising_logits(M, H, heads, dtype, a=8.0, seed=40):
    """Inputs whose causal logits rise with the key index: Q = a in every
    dimension (X column 1 is 1, Wq row 1 is a), K = x0 in every dimension (X
    column 0 is floor(j/4)/256, Wk row 0 is 1), so S_ij = 128 a x0_j, exact in
    fp32 from fp16 or bf16 operands.  Scaled by 1/sqrt(128) the logit grows by
    11.3 a / 8 per 128 keys: with a = 8 about 16 powers of two per key block,
    more than the 2^8 a row's maximum may rise before the kernel rescales the
    output it accumulates in tensor memory, so every block rescales.  V and Wo
    are random."""
    F = heads * 128
    g = torch.Generator().manual_seed(seed)
    X = torch.randn(M, H, generator=g) * 0.02
    X[:, 0] = torch.div(torch.arange(M), 4, rounding_mode="floor").float() / 256.0
    X[:, 1] = 1.0
    Wqkv = torch.randn(H, 3 * F, generator=g) * 0.02
    Wqkv[:, :2 * F] = 0.0
    Wqkv[1, :F] = a          # Q
    Wqkv[0, F:2 * F] = 1.0   # K
    Wo = torch.randn(F, H, generator=g) * 0.02
    return cs_inputs.ChainInputs("rising", "attn", M, H, F, dtype, X.to(dtype), Wqkv=Wqkv.to(dtype), Wo=Wo.to(dtype))


@pytest.mark.parametrize("kv", [-1, 1])
@pytest.mark.parametrize("tile_m", [128, 256])
@pytest.mark.parametrize("dtype", [torch.float16, torch.bfloat16])
def test_attention_rescales_the_tensor_memory_output(dtype, tile_m, kv):
    """Logits that rise by more than 2^8 from one key block to the next make
    every block raise the reference maximum and rescale O in TMEM (and l):
    O and Y still match the oracle, under two policies, also split into
    pieces whose merge takes different maxima."""
    inp = _rising_logits(1024, 256, 2, dtype)
    dev = device_tensors(inp, "nk")
    Yref, _, Oref = _oracle(inp)
    outs = {}
    for pol in ("row", "tile"):
        with plan_for(inp, pol, "nk", tile_m=tile_m, kv_chunk=kv) as plan:
            cs.cs_chain_debug_poison_intermediate(plan, -1)
            outs[pol] = forward(plan, dev).cpu()
            O = intermediate(plan, 1, inp.M, inp.F, inp.dtype).cpu()
            assert cs.cs_chain_status(plan) == cs.CS_OK
    assert oracle.rel_err(O, Oref) <= TOL
    assert oracle.rel_err(outs["row"], Yref) <= TOL
    assert torch.equal(outs["row"], outs["tile"])


@pytest.mark.parametrize("tile_m", [128, 256])
@pytest.mark.parametrize("M,H,heads", [(300, 384, 3), (513, 256, 2), (1100, 256, 1)])
def test_attention_chain_parity_bf16(M, H, heads, tile_m):
    """The attention chain in bf16 (P and O rounded to bf16) against the oracle."""
    inp = cs_inputs.make_custom("attn", M, H, heads * 128, dtype=torch.bfloat16, seed=39)
    dev = device_tensors(inp, "nk")
    with plan_for(inp, "row", "nk", tile_m=tile_m) as plan:
        Y = forward(plan, dev)
        QKV = intermediate(plan, 0, M, 3 * inp.F, inp.dtype)
        O = intermediate(plan, 1, M, inp.F, inp.dtype)
    Yref, QKVref, Oref = _oracle(inp)
    assert oracle.rel_err(QKV.cpu(), QKVref) <= TOL
    assert oracle.rel_err(O.cpu(), Oref) <= TOL
    assert oracle.rel_err(Y.cpu(), Yref) <= TOL
