"""GPU checks of the output release (desc.out_release): the last stage releases
Y per tile and per 128-row block the way producers release the intermediate,
for a following consumer of Y such as a collective that sends blocks of rows
as they complete (the Flux summary's GEMM + reduce-scatter fusion, here on one
GPU).  The counters end at their expected values, the output keeps its bits,
and the per-unit timeline shows blocks of Y completing before the kernel ends."""
from __future__ import annotations

import pytest
import torch

import cs_inputs
import oracle
from tests.gpu_util import TOL, device_tensors, forward, plan_for

pytestmark = pytest.mark.gpu

cs = pytest.importorskip("consumer_gemm_chain_gb300")

TILES = [(128, 128), (128, 256), (256, 256), (512, 256)]


def _check_output_sems(plan, forwards):
    q = cs.cs_chain_query(plan)
    last = q["stages"] - 1
    assert q["out_tile_sems"] and q["out_row_sems"]
    assert q["out_sem_words"] == q["m_tiles"] * q["n_tiles"][last]
    tiles, rows, epoch = cs.cs_chain_debug_read_sems(plan, last)
    assert epoch == forwards
    assert all(v == forwards for r in tiles for v in r)
    assert rows == [forwards * q["n_tiles"][last]] * q["m_tiles"]


@pytest.mark.parametrize("split", [0, 3])
@pytest.mark.parametrize("tile_m,tile_n", TILES)
def test_mlp_output_release(tile_m, tile_n, split):
    inp = cs_inputs.make_custom("gelu", 700, 512, 640, seed=61)
    dev = device_tensors(inp, "nk")
    with plan_for(inp, "tile", "nk", tile_m=tile_m, tile_n=tile_n, split_k=split) as plan:
        assert cs.cs_chain_query(plan)["out_tile_sems"] is None
        with pytest.raises(cs.CSError):
            cs.cs_chain_debug_read_sems(plan, 1)
        ref = forward(plan, dev).cpu()
    with plan_for(inp, "tile", "nk", tile_m=tile_m, tile_n=tile_n, split_k=split, out_release=1) as plan:
        outs = [forward(plan, dev).cpu() for _ in range(2)]
        _check_output_sems(plan, 2)
        cs.cs_chain_reset(plan)
        tiles, rows, epoch = cs.cs_chain_debug_read_sems(plan, 1)
        assert epoch == 0 and not any(rows) and not any(v for r in tiles for v in r)
        outs.append(forward(plan, dev).cpu())
        _check_output_sems(plan, 1)
    for Y in outs:
        assert torch.equal(Y, ref)
    Yref = oracle.mlp_gelu(inp.X, inp.W1, inp.b1, inp.W2)
    assert oracle.rel_err(ref, Yref) <= TOL


@pytest.mark.parametrize("policy", ["row", "stream"])
def test_swiglu_output_release(policy):
    inp = cs_inputs.make_custom("swiglu", 300, 1024, 1376, dtype=torch.bfloat16, seed=62)
    dev = device_tensors(inp, "nk")
    with plan_for(inp, policy, "nk") as plan:
        ref = forward(plan, dev).cpu()
    with plan_for(inp, policy, "nk", out_release=1) as plan:
        for _ in range(3):
            assert torch.equal(forward(plan, dev).cpu(), ref)
        _check_output_sems(plan, 3)


@pytest.mark.parametrize("tile_m", [128, 256])
def test_attention_output_release(tile_m):
    inp = cs_inputs.make_custom("attn", 520, 512, 256, seed=63)
    dev = device_tensors(inp, "nk")
    with plan_for(inp, "row", "nk", tile_m=tile_m) as plan:
        ref = forward(plan, dev).cpu()
    with plan_for(inp, "row", "nk", tile_m=tile_m, out_release=1) as plan:
        for _ in range(2):
            assert torch.equal(forward(plan, dev).cpu(), ref)
        _check_output_sems(plan, 2)


def test_allocation_free_forward_refuses_output_release():
    inp = cs_inputs.make_custom("gelu", 64, 256, 1024, seed=64)
    dev = device_tensors(inp, "nk")
    desc = cs.cs_chain_desc_init(kind="gelu", M=inp.M, H=inp.H, F=inp.F, dtype=inp.dtype, weight_layout="nk",
                                 out_release=1)
    with pytest.raises(cs.CSError) as e:
        cs.cs_mlp_forward_noalloc(desc, Y=torch.empty_like(dev["X"]), **dev)
    assert e.value.status == cs.CS_ERR_UNSUPPORTED


def test_row_blocks_of_y_complete_before_the_kernel_ends():
    """The per-unit timeline of a traced forward: the last consumer tile of the
    first row blocks finishes well before the last one of the last row blocks,
    which is the window a row-chunked collective could overlap."""
    inp = cs_inputs.make_inputs("gpt3", M=1024, seed=0)
    dev = device_tensors(inp, "nk")
    with plan_for(inp, "tile", "nk", out_release=1) as plan:
        forward(plan, dev)
        cs.cs_chain_debug_trace(plan, True)
        forward(plan, dev)
        recs = cs.cs_chain_debug_read_trace(plan)
        q = cs.cs_chain_query(plan)
        cs.cs_chain_debug_trace(plan, False)
    ready = {}
    for r in recs:
        stage, m_tile, _, _ = cs.decode_unit(r[0] & 0xFFFFFFFF)
        if stage == q["stages"] - 1 and r[7]:
            ready[m_tile] = max(ready.get(m_tile, 0), r[7])
    assert sorted(ready) == list(range(max(ready) + 1))
    start = min(r[2] for r in recs if r[2])
    end = max(ready.values())
    assert ready[0] < end
    assert (ready[0] - start) < 0.9 * (end - start)
