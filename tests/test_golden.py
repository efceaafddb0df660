"""The oracle still reproduces the stored tiny-chain values (regression pin)."""
import os

import numpy as np

import cs_inputs
import oracle

HERE = os.path.join(os.path.dirname(os.path.abspath(__file__)), "golden")


def load_tiny_golden():
    rows = []
    with open(os.path.join(HERE, "tiny_chain_seed0.txt")) as f:
        for line in f:
            if line.startswith("#") or not line.strip():
                continue
            r, c, v = line.split()
            rows.append((int(r), int(c), float(v)))
    return rows


def test_tiny_golden_matches_oracle():
    inp = cs_inputs.make_inputs("tiny", seed=0)
    Y = oracle.mlp_gelu(inp.X, inp.W1, inp.b1, inp.W2)
    g = load_tiny_golden()
    assert len(g) == 54
    for r, c, v in g:
        assert abs(Y[r, c] - v) <= 1e-15 * max(1.0, abs(v)), (r, c)
    # the values are not degenerate
    assert np.std([v for _, _, v in g]) > 1e-4
