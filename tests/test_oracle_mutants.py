"""Plant plausible mistakes in the oracle (on the CPU) and check that the pins
catch every one of them: a pin set that a dropped term, a wrong sign or index
or a transposed operand can slip past would not pin anything."""
from __future__ import annotations

import math

import numpy as np
import pytest

import oracle.chain as oc
from tests.oracle_pins import ALL_PINS


def _gelu_no_half(x):
    x = np.asarray(x, dtype=np.float64)
    return x * (1.0 + np.tanh(oc.GELU_SQRT_2_OVER_PI * (x + oc.GELU_CUBIC * x ** 3)))


def _gelu_square_not_cube(x):
    x = np.asarray(x, dtype=np.float64)
    return 0.5 * x * (1.0 + np.tanh(oc.GELU_SQRT_2_OVER_PI * (x + oc.GELU_CUBIC * x * x)))


def _mlp_no_bias(X, W1, b1, W2, return_hidden=False):
    X, W1, W2 = oc.to64(X), oc.to64(W1), oc.to64(W2)
    Hid = oc.gelu_tanh(X @ W1)
    return (Hid @ W2, Hid) if return_hidden else Hid @ W2


def _mlp_bias_after_act(X, W1, b1, W2, return_hidden=False):
    X, W1, b1, W2 = oc.to64(X), oc.to64(W1), oc.to64(b1), oc.to64(W2)
    Hid = oc.gelu_tanh(X @ W1) + b1[None, :]
    return (Hid @ W2, Hid) if return_hidden else Hid @ W2


def _mlp_w1_transposed(X, W1, b1, W2, return_hidden=False):
    X, W1, b1, W2 = oc.to64(X), oc.to64(W1), oc.to64(b1), oc.to64(W2)
    W1 = W1.T if W1.shape[0] == W1.shape[1] else W1[::-1, :]
    Hid = oc.gelu_tanh(X @ W1 + b1[None, :])
    return (Hid @ W2, Hid) if return_hidden else Hid @ W2


def _mlp_no_activation(X, W1, b1, W2, return_hidden=False):
    X, W1, b1, W2 = oc.to64(X), oc.to64(W1), oc.to64(b1), oc.to64(W2)
    Hid = X @ W1 + b1[None, :]
    return (Hid @ W2, Hid) if return_hidden else Hid @ W2


def _silu_wrong_sign(x):
    x = np.asarray(x, dtype=np.float64)
    with np.errstate(over="ignore"):
        return x / (1.0 + np.exp(x))


def _swiglu_act_on_up(X, Wg, Wu, Wd, return_hidden=False):
    X, Wg, Wu, Wd = oc.to64(X), oc.to64(Wg), oc.to64(Wu), oc.to64(Wd)
    Hid = (X @ Wg) * oc.silu(X @ Wu)
    return (Hid @ Wd, Hid) if return_hidden else Hid @ Wd


def _attn_variant(strict=False, nomask=False, scale_d=False, no_max=False):
    def f(Q, K, V, scale=None):
        Q, K, V = oc.to64(Q), oc.to64(K), oc.to64(V)
        S, d = Q.shape
        sc = (1.0 / d) if scale_d else (1.0 / math.sqrt(d) if scale is None else scale)
        logits = (Q @ K.T) * sc
        if not nomask:
            allowed = np.tril(np.ones((S, S), dtype=bool), k=-1 if strict else 0)
            allowed[0, 0] = True  # keep row 0 finite for the strict variant
            logits = np.where(allowed, logits, -np.inf)
        if not no_max:
            logits = logits - logits.max(axis=1, keepdims=True)
        P = np.exp(logits)
        P = P / P.sum(axis=1, keepdims=True)
        return P @ V
    return f


def _chain_kv_swapped(X, Wqkv, Wo, heads=12, head_dim=128, return_parts=False):
    X, Wqkv, Wo = oc.to64(X), oc.to64(Wqkv), oc.to64(Wo)
    hd = heads * head_dim
    QKV = X @ Wqkv
    O = np.empty((X.shape[0], hd))
    for h in range(heads):
        c = slice(h * head_dim, (h + 1) * head_dim)
        O[:, c] = oc.causal_attention(QKV[:, :hd][:, c], QKV[:, 2 * hd:][:, c], QKV[:, hd:2 * hd][:, c])
    Y = O @ Wo
    return (Y, QKV, O) if return_parts else Y


def _chain_head0_everywhere(X, Wqkv, Wo, heads=12, head_dim=128, return_parts=False):
    X, Wqkv, Wo = oc.to64(X), oc.to64(Wqkv), oc.to64(Wo)
    hd = heads * head_dim
    QKV = X @ Wqkv
    O = np.empty((X.shape[0], hd))
    c0 = slice(0, head_dim)
    for h in range(heads):
        c = slice(h * head_dim, (h + 1) * head_dim)
        O[:, c] = oc.causal_attention(QKV[:, :hd][:, c], QKV[:, hd:2 * hd][:, c0], QKV[:, 2 * hd:][:, c])
    Y = O @ Wo
    return (Y, QKV, O) if return_parts else Y


def _rel_err_mean(got, ref):
    got, ref = oc.to64(got), oc.to64(ref)
    return float(np.mean(np.abs(got - ref)) / np.max(np.abs(ref)))


MUTANTS = {
    "gelu_cubic_0.04": [("GELU_CUBIC", 0.04)],
    "gelu_sqrt_1_over_pi": [("GELU_SQRT_2_OVER_PI", math.sqrt(1.0 / math.pi))],
    "gelu_no_half": [("gelu_tanh", _gelu_no_half)],
    "gelu_square_not_cube": [("gelu_tanh", _gelu_square_not_cube)],
    "mlp_no_bias": [("mlp_gelu", _mlp_no_bias)],
    "mlp_bias_after_act": [("mlp_gelu", _mlp_bias_after_act)],
    "mlp_w1_transposed": [("mlp_gelu", _mlp_w1_transposed)],
    "mlp_no_activation": [("mlp_gelu", _mlp_no_activation)],
    "silu_wrong_sign": [("silu", _silu_wrong_sign)],
    "swiglu_act_on_up": [("mlp_swiglu", _swiglu_act_on_up)],
    "attn_strict_mask": [("causal_attention", _attn_variant(strict=True))],
    "attn_no_mask": [("causal_attention", _attn_variant(nomask=True))],
    "attn_scale_1_over_d": [("causal_attention", _attn_variant(scale_d=True))],
    "chain_k_v_swapped": [("attention_chain", _chain_kv_swapped)],
    "chain_head0_keys": [("attention_chain", _chain_head0_everywhere)],
    "rel_err_mean": [("rel_err", _rel_err_mean)],
}


@pytest.mark.parametrize("name", sorted(MUTANTS))
def test_mutant_is_caught(name, monkeypatch):
    for attr, value in MUTANTS[name]:
        monkeypatch.setattr(oc, attr, value)
    failed = []
    for pin in ALL_PINS:
        try:
            with np.errstate(all="ignore"):
                pin()
        except AssertionError:
            failed.append(pin.__name__)
    assert failed, f"mutant {name} passed every pin"
