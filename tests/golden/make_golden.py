"""Writes the stored expected values under tests/golden/ from the fp64 oracle.

Run from the repository root:  python tests/golden/make_golden.py
It calls only ``oracle/`` and the seeded input module; no value here comes
from the CUDA path.
"""
from __future__ import annotations

import os
import sys

HERE = os.path.dirname(os.path.abspath(__file__))
sys.path.insert(0, os.path.dirname(os.path.dirname(HERE)))

import cs_inputs  # noqa: E402
import oracle  # noqa: E402

TINY_ROWS = (0, 1, 17, 31, 32, 63)
TINY_COLS = tuple(range(0, 256, 32)) + (255,)


def tiny_chain_lines():
    inp = cs_inputs.make_inputs("tiny", seed=0)
    Y = oracle.mlp_gelu(inp.X, inp.W1, inp.b1, inp.W2)
    lines = [
        "# Tiny MLP chain, seed 0: X[64,256] W1[256,1024] b1[1024] GeLU(tanh) W2[1024,256], fp16 inputs",
        "# (CuSync README: two dependent GEMMs with GeLU fused into the first).",
        "# Written by tests/golden/make_golden.py from the fp64 oracle.  Columns: row col Y",
    ]
    for r in TINY_ROWS:
        for c in TINY_COLS:
            lines.append(f"{r} {c} {Y[r, c]:.17e}")
    return lines


def main():
    with open(os.path.join(HERE, "tiny_chain_seed0.txt"), "w") as f:
        f.write("\n".join(tiny_chain_lines()) + "\n")


if __name__ == "__main__":
    main()
