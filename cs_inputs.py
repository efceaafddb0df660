"""Seeded synthetic inputs for the GEMM-chain workloads.

This module is shared by the CUDA path's tests/bench and by the fp64 oracle's
tests.  It holds no arithmetic of the method itself: it only draws random
numbers, rounds them to the storage dtype and names the workload shapes.

Recipe (the same for every workload and every M):
  * a CPU ``torch.Generator`` seeded with ``seed`` (0 by default);
  * tensors drawn in a fixed order, each ``randn(shape, float32) * 0.02``
    (0.02 is the standard deviation), then rounded to the workload dtype;
  * weights are returned in the mathematical layout of the chain,
    ``Y = act(X @ W1 + b1) @ W2``: ``W1`` is ``[H, F]`` and ``W2`` is ``[F, H]``.

Workloads (shapes from the CuSync README, "8 way model parallelism GPT3 175B
(H=12288 FP16) and LLAMA 65.2B (H=8192)", and the FFN/attention shard widths
that follow from an 8-way split):
  tiny    X[64,256]  W1[256,1024] b1[1024] GeLU  W2[1024,256]      fp16
  gpt3    X[M,12288] W1[12288,6144] b1[6144] GeLU W2[6144,12288]   fp16
  llama   X[M,8192]  Wg,Wu[8192,2752] SiLU(g)*u  Wd[2752,8192]     bf16
  attn    X[M,12288] Wqkv[12288,4608] 12 heads x 128 causal, Wo[1536,12288]  fp16
  stress  X[M,8192]  W1[8192,8192] b1[8192] GeLU W2[8192,8192]     fp16
"""
from __future__ import annotations

import dataclasses

import torch

STD = 0.02

# name -> (kind, H, F, dtype, default M)
WORKLOADS = {
    "tiny": ("gelu", 256, 1024, torch.float16, 64),
    "gpt3": ("gelu", 12288, 6144, torch.float16, 2048),
    "llama": ("swiglu", 8192, 2752, torch.bfloat16, 2048),
    "attn": ("attn", 12288, 1536, torch.float16, 2048),
    "stress": ("gelu", 8192, 8192, torch.float16, 1536),
}
GPT3_M_SWEEP = (1, 16, 64, 256, 512, 1024, 2048)
STRESS_M_SWEEP = tuple(128 * b for b in range(1, 13))
ATTN_HEADS = 12
ATTN_HEAD_DIM = 128


@dataclasses.dataclass
class ChainInputs:
    """One workload's tensors (CPU, storage dtype, mathematical layout)."""

    name: str
    kind: str  # "gelu" | "swiglu" | "attn"
    M: int
    H: int
    F: int
    dtype: torch.dtype
    X: torch.Tensor
    W1: torch.Tensor | None = None  # [H, F]      (gelu)
    b1: torch.Tensor | None = None  # [F]         (gelu)
    W2: torch.Tensor | None = None  # [F, H]      (gelu; Wd for swiglu)
    Wg: torch.Tensor | None = None  # [H, F]      (swiglu)
    Wu: torch.Tensor | None = None  # [H, F]      (swiglu)
    Wqkv: torch.Tensor | None = None  # [H, 3*heads*d]  (attn)
    Wo: torch.Tensor | None = None  # [heads*d, H]    (attn)


def _draw(g: torch.Generator, shape, dtype) -> torch.Tensor:
    return (torch.randn(shape, generator=g, dtype=torch.float32) * STD).to(dtype)


def make_inputs(name: str, M: int | None = None, seed: int = 0, H: int | None = None,
                F: int | None = None) -> ChainInputs:
    """Draw the inputs of workload ``name`` (see module docstring)."""
    kind, H0, F0, dtype, M0 = WORKLOADS[name]
    M = M0 if M is None else M
    H = H0 if H is None else H
    F = F0 if F is None else F
    g = torch.Generator().manual_seed(seed)
    X = _draw(g, (M, H), dtype)
    if kind == "gelu":
        W1 = _draw(g, (H, F), dtype)
        b1 = _draw(g, (F,), dtype)
        W2 = _draw(g, (F, H), dtype)
        return ChainInputs(name, kind, M, H, F, dtype, X, W1=W1, b1=b1, W2=W2)
    if kind == "swiglu":
        Wg = _draw(g, (H, F), dtype)
        Wu = _draw(g, (H, F), dtype)
        Wd = _draw(g, (F, H), dtype)
        return ChainInputs(name, kind, M, H, F, dtype, X, Wg=Wg, Wu=Wu, W2=Wd)
    if kind == "attn":
        hd = F  # heads * head_dim
        Wqkv = _draw(g, (H, 3 * hd), dtype)
        Wo = _draw(g, (hd, H), dtype)
        return ChainInputs(name, kind, M, H, F, dtype, X, Wqkv=Wqkv, Wo=Wo)
    raise ValueError(name)


def make_custom(kind: str, M: int, H: int, F: int, dtype=torch.float16, seed: int = 0) -> ChainInputs:
    """Same recipe at arbitrary sizes (parity tests at sizes the oracle finishes quickly)."""
    g = torch.Generator().manual_seed(seed)
    X = _draw(g, (M, H), dtype)
    if kind == "gelu":
        return ChainInputs("custom", kind, M, H, F, dtype, X, W1=_draw(g, (H, F), dtype),
                           b1=_draw(g, (F,), dtype), W2=_draw(g, (F, H), dtype))
    if kind == "swiglu":
        return ChainInputs("custom", kind, M, H, F, dtype, X, Wg=_draw(g, (H, F), dtype),
                           Wu=_draw(g, (H, F), dtype), W2=_draw(g, (F, H), dtype))
    if kind == "attn":
        return ChainInputs("custom", kind, M, H, F, dtype, X, Wqkv=_draw(g, (H, 3 * F), dtype),
                           Wo=_draw(g, (F, H), dtype))
    raise ValueError(kind)


def sample_rows(M: int, n: int = 64, seed: int = 1) -> list[int]:
    """Seeded row sample that always holds the first and last row of every
    128-row block, topped up with random rows to ``n`` (or all rows if M <= n)."""
    if M <= n:
        return list(range(M))
    rows = set()
    for b in range(0, M, 128):
        rows.add(b)
        rows.add(min(b + 127, M - 1))
    g = torch.Generator().manual_seed(seed)
    perm = torch.randperm(M, generator=g).tolist()
    for r in perm:
        if len(rows) >= n:
            break
        rows.add(r)
    return sorted(rows)
