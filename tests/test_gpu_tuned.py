"""GPU parity of plans whose tile shape, K-splits and policy come from the
shipped tuning table (desc fields on auto, policy AUTO), against the fp64
oracle, through the C ABI.  The table only changes how the chain is tiled and
synchronised, never what it computes."""
from __future__ import annotations

import os

import pytest
import torch

import cs_inputs
import oracle
from tests.gpu_util import TOL, device_tensors, forward, plan_for

pytestmark = pytest.mark.gpu

cs = pytest.importorskip("consumer_gemm_chain_gb300")


@pytest.fixture(scope="module")
def tuned_table():
    if not os.path.exists(cs.chain.TUNE_TABLE):
        pytest.skip("no tuning table shipped")
    n = cs.cs_tune_load()
    assert n > 0
    yield n
    cs.cs_tune_clear()


def _oracle_rows(inp, rows):
    if inp.kind == "gelu":
        return oracle.mlp_gelu(inp.X[rows], inp.W1, inp.b1, inp.W2)
    if inp.kind == "swiglu":
        return oracle.mlp_swiglu(inp.X[rows], inp.Wg, inp.Wu, inp.W2)
    Y = oracle.attention_chain(inp.X, inp.Wqkv, inp.Wo, heads=inp.F // 128, head_dim=128)
    return Y[rows]


@pytest.mark.parametrize("workload,M", [("gpt3", 1), ("gpt3", 256), ("gpt3", 512), ("gpt3", 2048), ("llama", 64),
                                        ("llama", 1024),
                                        ("attn", 16), ("attn", 512), ("stress", 384), ("stress", 1152)])
def test_tuned_plans_match_the_oracle(tuned_table, workload, M):
    inp = cs_inputs.make_inputs(workload, M=M, seed=0)
    dev = device_tensors(inp, "nk")
    outs = {}
    for tuned in (0, -1):
        with plan_for(inp, "auto", "nk", tuned=tuned) as plan:
            q = cs.cs_chain_query(plan)
            if tuned == 0:
                assert q["tuned_entry"] >= 0, "the shipped table has an entry for this shape"
                assert q["policy"] in ("tile", "row", "strided")
            else:
                assert q["tuned_entry"] == -1 and q["policy"] == "tile"
            outs[tuned] = forward(plan, dev).cpu()
    rows = cs_inputs.sample_rows(M, 64)
    Yref = _oracle_rows(inp, rows)
    for tuned, Y in outs.items():
        assert oracle.rel_err(Y[rows], Yref) <= TOL, tuned
    # tiled differently, the same sums up to fp32 rounding order and the
    # rounding of the intermediate to the input type (one bf16 ulp is 2^-8)
    assert oracle.rel_err(outs[0], outs[-1]) <= (2e-3 if inp.dtype == torch.float16 else 1e-2)


def test_the_table_selects_a_stream_k_tail_where_it_won(tuned_table):
    """Entries that recorded a Stream-K tail give plans that run it (and match
    the oracle through the tuned-plan test above); the plan reports the tail."""
    import json
    with open(cs.chain.TUNE_TABLE) as f:
        entries = [e for e in json.load(f)["entries"] if e.get("sk_tiles")]
    if not entries:
        pytest.skip("no entry of the shipped table chose a Stream-K tail")
    for e in entries:
        extra = dict(heads=e["F"] // 128, head_dim=128) if e["kind"] == "attn" else {}
        desc = cs.cs_chain_desc_init(kind=e["kind"], M=e["M"], H=e["H"], F=e["F"],
                                     dtype=torch.float16 if e["dtype"] == "f16" else torch.bfloat16,
                                     policy=e["policy"], weight_layout=e.get("layout", "nk"), **extra)
        with cs.cs_chain_plan(desc) as plan:
            q = cs.cs_chain_query(plan)
        assert q["tuned_entry"] >= 0, e
        assert q["sk_tiles"] == e["sk_tiles"], e
        # sk_units 0: one Stream-K unit per resident worker
        assert q["sk_units"] == e["sk_units"] if e["sk_units"] else 0 < q["sk_units"] <= q["workers"], e
        if e["split_k"] == 0:
            # automatic K-splits: the last stage unsplit, its tiles shared out
            assert q["split_k"][q["stages"] - 1] == 1, e
