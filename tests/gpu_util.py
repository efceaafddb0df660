"""Helpers for the GPU tests: move seeded inputs to the device in the layout a
plan expects and run one chain forward through the C ABI."""
from __future__ import annotations

import torch

import consumer_gemm_chain_gb300 as cs

TOL = 5e-3  # max|gpu - oracle| / max|oracle|, fp16/bf16 inputs, fp32 accumulate


def weight(t: torch.Tensor, layout: str) -> torch.Tensor:
    """Math-layout [K, N] weight -> device tensor in the plan's storage layout."""
    t = t if layout == "kn" else t.t().contiguous()
    return t.cuda()


def plan_for(inp, policy="tile", layout="kn", **kw):
    kind = {"gelu": "gelu", "swiglu": "swiglu", "attn": "attn"}[inp.kind]
    extra = {}
    if kind == "attn":
        extra = dict(heads=inp.F // 128, head_dim=128)
    desc = cs.cs_chain_desc_init(kind=kind, M=inp.M, H=inp.H, F=inp.F, dtype=inp.dtype, policy=policy,
                                 weight_layout=layout, **extra, **kw)
    return cs.cs_chain_plan(desc)


def device_tensors(inp, layout="kn"):
    d = {"X": inp.X.cuda()}
    if inp.kind == "gelu":
        d.update(W1=weight(inp.W1, layout), b1=inp.b1.cuda(), W2=weight(inp.W2, layout))
    elif inp.kind == "swiglu":
        d.update(Wg=weight(inp.Wg, layout), Wu=weight(inp.Wu, layout), W2=weight(inp.W2, layout))
    else:
        d.update(Wqkv=weight(inp.Wqkv, layout), Wo=weight(inp.Wo, layout))
    return d


def forward(plan, dev, Y=None, check=True):
    if Y is None:
        Y = torch.empty_like(dev["X"])
    if "Wqkv" in dev:
        cs.cs_attn_chain_forward(plan, dev["X"], dev["Wqkv"], dev["Wo"], Y)
    else:
        cs.cs_mlp_forward(plan, Y=Y, **dev)
    if check:
        torch.cuda.synchronize()
        st = cs.cs_chain_status(plan)
        assert st == cs.CS_OK, f"{cs.STATUS_NAMES.get(st)}: {cs.cs_last_error_string()}"
    return Y


def intermediate(plan, which, rows, cols, dtype):
    """Copy of a plan-owned intermediate buffer (H, or QKV / O) as a torch tensor."""
    out = torch.empty(rows, cols, dtype=dtype, device="cuda")
    cs.cs_chain_debug_copy_intermediate(plan, which, out)
    return out
