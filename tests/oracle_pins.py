"""Pins for the fp64 oracle: checks against things other than the oracle itself.

Each ``pin_*`` function raises AssertionError when the oracle disagrees with
an independent fact: a brute-force loop, a closed form or identity, an
independent library routine (torch float64), an identity chain or an
attention special case.  ``test_oracle_pins.py`` runs them on the oracle as
it is; ``test_oracle_mutants.py`` plants mistakes in the oracle and checks
that some pin catches each one.
"""
from __future__ import annotations

import math

import numpy as np
import torch
import torch.nn.functional as Fn

import oracle.chain as oc


def _rng(seed=0):
    return np.random.default_rng(seed)


def _close(a, b, tol=1e-12, what=""):
    a = np.asarray(a, dtype=np.float64)
    b = np.asarray(b, dtype=np.float64)
    scale = max(1.0, float(np.max(np.abs(b)))) if b.size else 1.0
    err = float(np.max(np.abs(a - b))) if a.size else 0.0
    assert a.shape == b.shape, f"{what}: shape {a.shape} vs {b.shape}"
    assert err <= tol * scale, f"{what}: max err {err:.3e} > {tol:.1e}"


# ---------------------------------------------------------------- activations
def pin_gelu_vs_torch_tanh_gelu():
    x = np.linspace(-8.0, 8.0, 4001)
    ref = Fn.gelu(torch.from_numpy(x), approximate="tanh").numpy()
    _close(oc.gelu_tanh(x), ref, 1e-14, "gelu vs torch tanh-gelu")


def pin_gelu_near_erf_gelu():
    # The tanh form approximates x*Phi(x); its largest deviation is a few 1e-4.
    x = np.linspace(-6.0, 6.0, 2401)
    exact = np.array([0.5 * v * (1.0 + math.erf(v / math.sqrt(2.0))) for v in x])
    err = np.max(np.abs(oc.gelu_tanh(x) - exact))
    assert err < 1e-3, f"tanh-gelu strays {err:.2e} from x*Phi(x)"


def pin_gelu_odd_identity_and_limits():
    x = np.linspace(-10.0, 10.0, 2001)
    # tanh is odd, so GeLU(x) - GeLU(-x) = x exactly in real arithmetic.
    _close(oc.gelu_tanh(x) - oc.gelu_tanh(-x), x, 1e-14, "gelu odd part")
    assert oc.gelu_tanh(np.array([0.0]))[0] == 0.0
    h = 1e-6
    slope0 = (oc.gelu_tanh(np.array([h]))[0] - oc.gelu_tanh(np.array([-h]))[0]) / (2 * h)
    assert abs(slope0 - 0.5) < 1e-9, f"gelu'(0)={slope0}"
    assert abs(oc.gelu_tanh(np.array([30.0]))[0] - 30.0) < 1e-12
    assert abs(oc.gelu_tanh(np.array([-30.0]))[0]) < 1e-12


def pin_silu():
    x = np.linspace(-20.0, 20.0, 4001)
    ref = Fn.silu(torch.from_numpy(x)).numpy()
    _close(oc.silu(x), ref, 1e-14, "silu vs torch")
    _close(oc.silu(x) - oc.silu(-x), x, 1e-13, "silu odd part")
    assert oc.silu(np.array([0.0]))[0] == 0.0


# ---------------------------------------------------------------- MLP chains
def _brute_mlp_gelu(X, W1, b1, W2):
    M, H = X.shape
    F = W1.shape[1]
    Y = np.zeros((M, W2.shape[1]))
    for m in range(M):
        hid = []
        for f in range(F):
            s = 0.0
            for k in range(H):
                s += X[m, k] * W1[k, f]
            hid.append(s + b1[f])
        hid = Fn.gelu(torch.tensor(hid, dtype=torch.float64), approximate="tanh").tolist()
        for n in range(W2.shape[1]):
            s = 0.0
            for f in range(F):
                s += hid[f] * W2[f, n]
            Y[m, n] = s
    return Y


def pin_mlp_gelu_brute_force():
    r = _rng(1)
    for (M, H, F) in [(1, 1, 1), (3, 5, 7), (4, 8, 6), (2, 7, 3)]:
        X, W1, b1, W2 = r.normal(size=(M, H)), r.normal(size=(H, F)), r.normal(size=F), r.normal(size=(F, H))
        _close(oc.mlp_gelu(X, W1, b1, W2), _brute_mlp_gelu(X, W1, b1, W2), 1e-12, f"mlp brute {M,H,F}")


def pin_mlp_gelu_vs_torch_linear():
    r = _rng(2)
    M, H, F = 37, 96, 160
    X, W1, b1, W2 = r.normal(size=(M, H)), r.normal(size=(H, F)), r.normal(size=F), r.normal(size=(F, H))
    t = lambda a: torch.from_numpy(a)  # noqa: E731
    hid = Fn.gelu(Fn.linear(t(X), t(W1).T.contiguous(), t(b1)), approximate="tanh")
    ref = Fn.linear(hid, t(W2).T.contiguous()).numpy()
    _close(oc.mlp_gelu(X, W1, b1, W2), ref, 1e-12, "mlp vs torch linear")
    Y, Hid = oc.mlp_gelu(X, W1, b1, W2, return_hidden=True)
    _close(Hid, hid.numpy(), 1e-12, "hidden vs torch")


def pin_mlp_identity_chains():
    r = _rng(3)
    X = r.normal(size=(9, 16))
    I = np.eye(16)
    _close(oc.mlp_gelu(X, I, np.zeros(16), I), oc.gelu_tanh(X), 1e-15, "W1=W2=I")
    # F > H: W1 = [I | 0], W2 = [I ; 0]
    W1 = np.concatenate([I, np.zeros((16, 8))], axis=1)
    W2 = np.concatenate([I, np.zeros((8, 16))], axis=0)
    _close(oc.mlp_gelu(X, W1, np.zeros(24), W2), oc.gelu_tanh(X), 1e-15, "[I|0] chain")
    # bias lands on the hidden column it indexes
    b = np.arange(16, dtype=np.float64) * 0.25 - 2.0
    ref = Fn.gelu(torch.from_numpy(X + b[None, :]), approximate="tanh").numpy()
    _close(oc.mlp_gelu(X, I, b, I), ref, 1e-14, "bias column")
    # rows are independent: a row subset gives the same rows
    W1r, b1r, W2r = r.normal(size=(16, 12)), r.normal(size=12), r.normal(size=(12, 16))
    full = oc.mlp_gelu(X, W1r, b1r, W2r)
    _close(oc.mlp_gelu(X[[0, 4, 8]], W1r, b1r, W2r), full[[0, 4, 8]], 1e-15, "row subset")


def pin_mlp_swiglu():
    r = _rng(4)
    M, H, F = 3, 5, 4
    X, Wg, Wu, Wd = r.normal(size=(M, H)), r.normal(size=(H, F)), r.normal(size=(H, F)), r.normal(size=(F, H))
    Y = np.zeros((M, H))
    for m in range(M):
        hid = []
        for f in range(F):
            g = sum(X[m, k] * Wg[k, f] for k in range(H))
            u = sum(X[m, k] * Wu[k, f] for k in range(H))
            hid.append(Fn.silu(torch.tensor(g, dtype=torch.float64)).item() * u)
        for n in range(H):
            Y[m, n] = sum(hid[f] * Wd[f, n] for f in range(F))
    _close(oc.mlp_swiglu(X, Wg, Wu, Wd), Y, 1e-12, "swiglu brute")
    I = np.eye(6)
    X6 = r.normal(size=(4, 6))
    _close(oc.mlp_swiglu(X6, I, I, I), Fn.silu(torch.from_numpy(X6)).numpy() * X6, 1e-14, "swiglu identity")
    # gate and up are not interchangeable: SiLU applies to the gate only
    Z = np.zeros((6, 6))
    _close(oc.mlp_swiglu(X6, Z, I, I), np.zeros_like(X6), 0.0, "zero gate")


# ---------------------------------------------------------------- attention
def pin_causal_attention_vs_sdpa():
    r = _rng(5)
    for S, d in [(1, 4), (7, 8), (33, 16), (130, 128)]:
        Q, K, V = r.normal(size=(S, d)), r.normal(size=(S, d)), r.normal(size=(S, d))
        ref = Fn.scaled_dot_product_attention(
            torch.from_numpy(Q)[None], torch.from_numpy(K)[None], torch.from_numpy(V)[None], is_causal=True
        )[0].numpy()
        _close(oc.causal_attention(Q, K, V), ref, 1e-12, f"sdpa {S},{d}")


def pin_causal_attention_special_cases():
    r = _rng(6)
    S, d = 12, 8
    Q, K, V = r.normal(size=(S, d)), r.normal(size=(S, d)), r.normal(size=(S, d))
    O = oc.causal_attention(Q, K, V)
    _close(O[0], V[0], 1e-15, "row 0 sees only key 0")
    O0 = oc.causal_attention(np.zeros((S, d)), K, V)
    prefix_mean = np.cumsum(V, axis=0) / np.arange(1, S + 1)[:, None]
    _close(O0, prefix_mean, 1e-13, "Q=0 gives the prefix mean")
    # later keys never change earlier rows
    V2 = V.copy()
    V2[-1] += 100.0
    _close(oc.causal_attention(Q, K, V2)[:-1], O[:-1], 1e-15, "causality")


def _brute_attention_chain(X, Wqkv, Wo, heads, d):
    M = X.shape[0]
    hd = heads * d
    QKV = np.array([[sum(X[m, k] * Wqkv[k, c] for k in range(X.shape[1])) for c in range(3 * hd)] for m in range(M)])
    O = np.zeros((M, hd))
    for h in range(heads):
        for i in range(M):
            logits = []
            for j in range(i + 1):
                q = QKV[i, h * d:(h + 1) * d]
                k = QKV[j, hd + h * d: hd + (h + 1) * d]
                logits.append(sum(q[t] * k[t] for t in range(d)) / math.sqrt(d))
            mx = max(logits)
            w = [math.exp(v - mx) for v in logits]
            z = sum(w)
            for t in range(d):
                O[i, h * d + t] = sum(w[j] / z * QKV[j, 2 * hd + h * d + t] for j in range(i + 1))
    return np.array([[sum(O[m, c] * Wo[c, n] for c in range(hd)) for n in range(Wo.shape[1])] for m in range(M)])


def pin_attention_chain_brute_force():
    r = _rng(7)
    M, H, heads, d = 5, 6, 2, 4
    X, Wqkv, Wo = r.normal(size=(M, H)), r.normal(size=(H, 3 * heads * d)), r.normal(size=(heads * d, H))
    got = oc.attention_chain(X, Wqkv, Wo, heads=heads, head_dim=d)
    _close(got, _brute_attention_chain(X, Wqkv, Wo, heads, d), 1e-12, "attention chain brute")


def pin_attention_chain_vs_torch():
    r = _rng(8)
    M, H, heads, d = 70, 48, 3, 16
    X, Wqkv, Wo = r.normal(size=(M, H)), r.normal(size=(H, 3 * heads * d)), r.normal(size=(heads * d, H))
    t = torch.from_numpy
    qkv = t(X) @ t(Wqkv)
    q, k, v = qkv.split(heads * d, dim=1)
    q, k, v = (z.reshape(M, heads, d).transpose(0, 1) for z in (q, k, v))
    o = Fn.scaled_dot_product_attention(q, k, v, is_causal=True).transpose(0, 1).reshape(M, heads * d)
    ref = (o @ t(Wo)).numpy()
    Y, QKV, O = oc.attention_chain(X, Wqkv, Wo, heads=heads, head_dim=d, return_parts=True)
    _close(Y, ref, 1e-12, "attention chain vs torch")
    _close(O, o.numpy(), 1e-12, "attention O vs torch")


def pin_rel_err():
    assert oc.rel_err(np.array([1.0, 2.0]), np.array([1.0, 2.0])) == 0.0
    assert abs(oc.rel_err(np.array([1.0, 2.5]), np.array([1.0, 2.0])) - 0.25) < 1e-15
    assert abs(oc.rel_err(np.array([-4.0, 0.0]), np.array([-4.0, 1.0])) - 0.25) < 1e-15


ALL_PINS = [v for k, v in sorted(globals().items()) if k.startswith("pin_")]
