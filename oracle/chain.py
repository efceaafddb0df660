"""Plain fp64 definitions of what a GEMM chain computes.

TEST INFRASTRUCTURE ONLY (see ``oracle/__init__.py``): slow, obviously correct,
evaluated in float64 from the fp16/bf16-rounded inputs.  Tile synchronisation
changes only *when* a consumer tile runs, never what it computes (CuSync
README, first paragraph: thread blocks of a producer/consumer chain are
synchronised per tile instead of per kernel).  So the oracle is the plain
composed result, with no tiling, blocking or fusion.  A library matmul
(numpy ``@`` on float64) is the only library primitive used for contractions.

Every function here is pinned by ``tests/test_oracle_pins.py`` against things
other than itself: brute-force loops, closed forms and odd-part identities,
independent library routines (torch's tanh-GeLU, SiLU and causal
scaled-dot-product attention in float64), identity chains and attention
special cases.  Nothing is "parity unpinned".

Readings of points the pages leave open:
  * "GeLU" (CuSync README, MLP paragraph) is the tanh form
        GeLU(x) = x/2 * (1 + tanh(sqrt(2/pi) * (x + 0.044715 x^3))).
  * SwiGLU (LLaMA MLP) is (SiLU(X Wg) * (X Wu)) Wd with SiLU(x) = x/(1+e^-x).
  * The attention chain is QKV = X Wqkv with columns [Q | K | V], each
    head-major (head h owns columns h*d .. h*d+d-1 of its block); per head a
    causal softmax(Q K^T / sqrt(d)) V; heads concatenated; then O Wo.
  * No bias outside GEMM1 of the GeLU MLP; the intermediate is not rounded.
"""
from __future__ import annotations

import math

import numpy as np

# GeLU tanh-form constants: sqrt(2/pi) and the cubic coefficient.
GELU_SQRT_2_OVER_PI = math.sqrt(2.0 / math.pi)
GELU_CUBIC = 0.044715


def to64(t) -> np.ndarray:
    """fp16/bf16/fp32 torch tensor or array -> float64 numpy array (exact)."""
    if hasattr(t, "detach"):
        return t.detach().to("cpu").double().numpy()
    return np.asarray(t, dtype=np.float64)


def gelu_tanh(x: np.ndarray) -> np.ndarray:
    """tanh-form GeLU, elementwise, float64."""
    x = np.asarray(x, dtype=np.float64)
    return 0.5 * x * (1.0 + np.tanh(GELU_SQRT_2_OVER_PI * (x + GELU_CUBIC * x * x * x)))


def silu(x: np.ndarray) -> np.ndarray:
    """SiLU(x) = x / (1 + exp(-x)), elementwise, float64."""
    x = np.asarray(x, dtype=np.float64)
    with np.errstate(over="ignore"):
        return x / (1.0 + np.exp(-x))


def mlp_gelu(X, W1, b1, W2, return_hidden: bool = False):
    """Y = GeLU(X @ W1 + b1) @ W2 (CuSync README: MLP with GeLU fused into the
    first GEMM).  X [M,H], W1 [H,F], b1 [F], W2 [F,H]; rows are independent,
    so a caller may pass any subset of X's rows."""
    X, W1, b1, W2 = to64(X), to64(W1), to64(b1), to64(W2)
    Hid = gelu_tanh(X @ W1 + b1[None, :])
    Y = Hid @ W2
    return (Y, Hid) if return_hidden else Y


def mlp_swiglu(X, Wg, Wu, Wd, return_hidden: bool = False):
    """Y = (SiLU(X @ Wg) * (X @ Wu)) @ Wd (LLaMA MLP shard).  X [M,H],
    Wg/Wu [H,F], Wd [F,H]; rows are independent."""
    X, Wg, Wu, Wd = to64(X), to64(Wg), to64(Wu), to64(Wd)
    Hid = silu(X @ Wg) * (X @ Wu)
    Y = Hid @ Wd
    return (Y, Hid) if return_hidden else Y


def causal_attention(Q, K, V, scale: float | None = None) -> np.ndarray:
    """One head of causal attention: softmax(Q K^T * scale, key j <= query i) V.

    Q, K, V are [S, d]; scale defaults to 1/sqrt(d).  The softmax subtracts the
    row maximum before exponentiating (mathematically the same result)."""
    Q, K, V = to64(Q), to64(K), to64(V)
    S, d = Q.shape
    if scale is None:
        scale = 1.0 / math.sqrt(d)
    logits = (Q @ K.T) * scale
    allowed = np.tril(np.ones((S, S), dtype=bool))  # key index j <= query index i
    logits = np.where(allowed, logits, -np.inf)
    logits = logits - logits.max(axis=1, keepdims=True)
    P = np.exp(logits)
    P = P / P.sum(axis=1, keepdims=True)
    return P @ V


def attention_chain(X, Wqkv, Wo, heads: int = 12, head_dim: int = 128, return_parts: bool = False):
    """QKV projection -> per-head causal attention -> output projection.

    X [M,H], Wqkv [H, 3*heads*head_dim] with columns [Q | K | V] (head-major in
    each block), Wo [heads*head_dim, H].  Sequence length = M, batch 1."""
    X, Wqkv, Wo = to64(X), to64(Wqkv), to64(Wo)
    hd = heads * head_dim
    QKV = X @ Wqkv
    O = np.empty((X.shape[0], hd), dtype=np.float64)
    for h in range(heads):
        c = slice(h * head_dim, (h + 1) * head_dim)
        Qh = QKV[:, 0 * hd:1 * hd][:, c]
        Kh = QKV[:, 1 * hd:2 * hd][:, c]
        Vh = QKV[:, 2 * hd:3 * hd][:, c]
        O[:, c] = causal_attention(Qh, Kh, Vh)
    Y = O @ Wo
    return (Y, QKV, O) if return_parts else Y


def rel_err(got, ref) -> float:
    """max|got - ref| / max|ref|, in float64 (the parity metric)."""
    got, ref = to64(got), to64(ref)
    denom = float(np.max(np.abs(ref)))
    num = float(np.max(np.abs(got - ref)))
    if denom == 0.0:
        return num
    return num / denom
