"""GPU parity of the fused SwiGLU MLP chain (LLaMA 65.2B 8-way shard shape)
against the fp64 oracle, through the C ABI.

The producer tile holds the gate and up projections of the same 128 output
columns side by side (one N = 256 tcgen05 MMA), so SiLU(gate) * up is applied
in the producer epilogue."""
from __future__ import annotations

import pytest
import torch

import cs_inputs
import oracle
from tests.gpu_util import TOL, device_tensors, forward, intermediate, plan_for

pytestmark = pytest.mark.gpu

cs = pytest.importorskip("consumer_gemm_chain_gb300")


def _oracle(inp, rows=None):
    X = inp.X if rows is None else inp.X[rows]
    return oracle.mlp_swiglu(X, inp.Wg, inp.Wu, inp.W2, return_hidden=True)


@pytest.mark.parametrize("layout", ["kn", "nk"])
@pytest.mark.parametrize("dtype", [torch.bfloat16, torch.float16])
@pytest.mark.parametrize("M,H,F", [(1, 256, 344), (64, 512, 1024), (200, 320, 392), (300, 1024, 2752)])
def test_swiglu_parity(M, H, F, dtype, layout):
    inp = cs_inputs.make_custom("swiglu", M, H, F, dtype=dtype, seed=21)
    dev = device_tensors(inp, layout)
    with plan_for(inp, "tile", layout) as plan:
        Y = forward(plan, dev)
        Hid = intermediate(plan, 0, inp.M, inp.F, inp.dtype)
    Yref, Href = _oracle(inp)
    assert oracle.rel_err(Hid.cpu(), Href) <= TOL
    assert oracle.rel_err(Y.cpu(), Yref) <= TOL


@pytest.mark.parametrize("tile_m", [128, 256, 512])
@pytest.mark.parametrize("layout", ["kn", "nk"])
@pytest.mark.parametrize("M,H,F", [(1, 512, 344), (300, 1024, 2752), (700, 768, 392)])
def test_swiglu_tile_shapes(M, H, F, layout, tile_m):
    """256-row tiles split the gate|up MMA over a CTA pair (gate rows of B on the
    first CTA, up rows on the second); 512-row tiles add a second pair that
    shares every weight box by multicast.  All shapes agree bit for bit."""
    inp = cs_inputs.make_custom("swiglu", M, H, F, dtype=torch.bfloat16, seed=23)
    dev = device_tensors(inp, layout)
    with plan_for(inp, "tile", layout, tile_m=tile_m, tile_n=256) as plan:
        assert cs.cs_chain_query(plan)["tile_m"] == tile_m
        Y = forward(plan, dev)
        Hid = intermediate(plan, 0, inp.M, inp.F, inp.dtype)
    Yref, Href = _oracle(inp)
    assert oracle.rel_err(Hid.cpu(), Href) <= TOL
    assert oracle.rel_err(Y.cpu(), Yref) <= TOL
    with plan_for(inp, "tile", layout, tile_m=128, tile_n=256) as plan:
        assert torch.equal(forward(plan, dev), Y)


def test_swiglu_policies_bit_identical():
    inp = cs_inputs.make_custom("swiglu", 384, 768, 1376, dtype=torch.bfloat16, seed=22)
    dev = device_tensors(inp, "nk")
    outs = {}
    for pol in ("tile", "row", "strided", "stream"):
        with plan_for(inp, pol, "nk", group_m=1) as plan:
            outs[pol] = forward(plan, dev).cpu()
            tiles, rows, epoch = cs.cs_chain_debug_read_sems(plan, 0)
            assert epoch == 1 and all(v == 1 for r in tiles for v in r)
    Yref, _ = _oracle(inp)
    assert oracle.rel_err(outs["tile"], Yref) <= TOL
    for k, v in outs.items():
        assert torch.equal(v, outs["tile"]), k


@pytest.mark.parametrize("M", (1, 64, 512, 2048))
def test_llama_shard_sampled_rows(M):
    inp = cs_inputs.make_inputs("llama", M=M, seed=0)
    dev = device_tensors(inp, "nk")
    with plan_for(inp, "tile", "nk") as plan:
        Y = forward(plan, dev).cpu()
    rows = cs_inputs.sample_rows(M, 64)
    Yref, _ = _oracle(inp, rows)
    assert oracle.rel_err(Y[rows], Yref) <= TOL
