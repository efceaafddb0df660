"""Tile-synchronised GEMM chains on GB300 (sm_103a).

A chain such as a transformer MLP, Y = GeLU(X W1 + b1) W2, runs as one
persistent tcgen05 kernel in which each consumer tile starts as soon as the
producer tiles it reads are finished (CuSync README, first paragraph).  The
work happens in the C-ABI library ``_lib/libcs_chain.so`` (``include/cs_chain.h``);
this package is its ctypes binding.
"""
from .chain import *  # noqa: F401,F403
from .chain import (  # noqa: F401
    CSError,
    Plan,
    cs_abi_version,
    cs_attn_chain_forward,
    cs_chain_debug_copy_intermediate,
    cs_chain_debug_poison_intermediate,
    cs_chain_debug_set_epoch,
    cs_chain_plan_info,
    cs_library_features,
    cs_chain_debug_read_sems,
    cs_chain_debug_read_trace,
    cs_chain_debug_set_delays,
    cs_chain_debug_skip_release,
    cs_chain_debug_trace,
    cs_chain_desc_init,
    cs_chain_destroy,
    cs_chain_forward_stage,
    cs_chain_host_join,
    cs_chain_plan,
    cs_chain_query,
    cs_chain_reset,
    cs_chain_status,
    cs_last_error_string,
    cs_mlp_forward,
    cs_mlp_forward_host,
    cs_mlp_forward_noalloc,
    cs_noalloc_status,
    cs_schedule_build,
    cs_tune_clear,
    cs_tune_load,
    cs_tune_match,
    cs_tune_size,
    decode_unit,
)
