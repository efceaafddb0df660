"""The allocation-free forward, through the C ABI, against the planned forward.

cs_mlp_forward_noalloc exists for callers that may not allocate device memory
themselves: code that runs inside another framework whose caching allocator
owns the GPU memory budget, or a latency-critical loop where cudaMalloc and
cudaFree would synchronise the device.  It keeps its intermediate, semaphores
and schedule in a fixed array inside the library instead of a plan.  Each test
runs it twice in a row (the array keeps the previous call's contents, which the
second call must not depend on) and compares Y with cs_chain_plan +
cs_mlp_forward (unsplit, like the allocation-free forward) and with the fp64
oracle, within the parity tolerance the other GPU tests use.  This file
runs last, and also passes on its own in a fresh process.
"""
from __future__ import annotations

import pytest
import torch

import cs_inputs
import oracle
from tests.gpu_util import TOL, device_tensors, forward, plan_for

pytestmark = pytest.mark.gpu

cs = pytest.importorskip("consumer_gemm_chain_gb300")


def _desc(inp, layout, policy):
    return cs.cs_chain_desc_init(kind=inp.kind, M=inp.M, H=inp.H, F=inp.F, dtype=inp.dtype, policy=policy,
                                 weight_layout=layout)


@pytest.mark.parametrize("kind,M,H,F,layout,policy", [
    ("gelu", 300, 512, 1024, "nk", "tile"),
    ("gelu", 129, 256, 392, "kn", "row"),
    ("swiglu", 200, 512, 688, "nk", "tile"),
    ("gelu", 64, 256, 1024, "nk", "stream"),
    ("gelu", 1024, 512, 1024, "nk", "tile"),      # 512-row tiles: 4-CTA clusters, multicast weights
    ("swiglu", 640, 512, 688, "kn", "tile"),      # gate|up pairs in 4-CTA clusters, padded rows
])
def test_noalloc_matches_planned_forward_twice(kind, M, H, F, layout, policy):
    inp = cs_inputs.make_custom(kind, M, H, F, dtype=torch.float16, seed=41)
    dev = device_tensors(inp, layout)
    with plan_for(inp, policy, layout, split_k=1) as plan:
        ref = forward(plan, dev).cpu()
    if kind == "gelu":
        truth = oracle.mlp_gelu(inp.X, inp.W1, inp.b1, inp.W2)
    else:
        truth = oracle.mlp_swiglu(inp.X, inp.Wg, inp.Wu, inp.W2)
    assert oracle.rel_err(ref, truth) <= TOL
    desc = _desc(inp, layout, policy)
    for call in range(2):
        Y = torch.full_like(dev["X"], float("nan"))
        cs.cs_mlp_forward_noalloc(desc, Y=Y, **dev)
        torch.cuda.synchronize()
        assert cs.cs_noalloc_status() == cs.CS_OK, cs.cs_last_error_string()
        Yc = Y.cpu()
        assert not torch.isnan(Yc).any(), call
        assert oracle.rel_err(Yc, ref) <= TOL, call   # against the planned forward
        assert oracle.rel_err(Yc, truth) <= TOL, call  # and against the fp64 oracle


def test_noalloc_refuses_k_splits():
    """The array holds no split-K workspace: split_k > 1 or split_k_first > 1
    is refused, not ignored."""
    inp = cs_inputs.make_custom("gelu", 64, 256, 512, dtype=torch.float16, seed=42)
    dev = device_tensors(inp, "nk")
    for field in ("split_k", "split_k_first"):
        desc = _desc(inp, "nk", "tile")
        setattr(desc, field, 2)
        with pytest.raises(cs.CSError) as e:
            cs.cs_mlp_forward_noalloc(desc, Y=torch.empty_like(dev["X"]), **dev)
        assert e.value.status == cs.CS_ERR_UNSUPPORTED and field in str(e.value)


def test_noalloc_rejects_shapes_beyond_its_scratch():
    # M * F * 2 bytes alone exceed the fixed scratch array: refused before any launch
    desc = cs.cs_chain_desc_init(kind="gelu", M=4096, H=256, F=8192, dtype=torch.float16)
    X = torch.zeros(4096, 256, dtype=torch.float16, device="cuda")
    W1 = torch.zeros(8192, 256, dtype=torch.float16, device="cuda")
    b1 = torch.zeros(8192, dtype=torch.float16, device="cuda")
    W2 = torch.zeros(256, 8192, dtype=torch.float16, device="cuda")
    desc.weight_layout = cs.CS_WEIGHTS_NK
    Y = torch.zeros_like(X)
    with pytest.raises(cs.CSError) as e:
        cs.cs_mlp_forward_noalloc(desc, X, W1=W1, b1=b1, W2=W2, Y=Y)
    assert e.value.status == cs.CS_ERR_INVALID_ARG
    assert "scratch" in str(e.value)
