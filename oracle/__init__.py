"""fp64 CPU oracle for tile-synchronised GEMM chains.

TEST INFRASTRUCTURE ONLY.  Only ``tests/``, ``__graft_entry__.smoke()`` and the
CPU-baseline / reference arm of ``bench.py`` may import this package.  The
library (``consumer_gemm_chain_gb300``) never imports it and shares no code
with it; the two meet only in the seeded input module ``cs_inputs``.

See ``oracle/chain.py`` for the definitions and their citations.
"""
from .chain import (  # noqa: F401
    attention_chain,
    causal_attention,
    gelu_tanh,
    mlp_gelu,
    mlp_swiglu,
    rel_err,
    silu,
    to64,
)
