"""B300 (sm_103a) Mixtral sparse mixture-of-experts feed-forward layer.

The compute lives in libmoe.so (hand-written CUDA behind the C ABI in
include/moe.h); ``binding`` is a thin ctypes layer with the same names.
Importing this package does not load the library; the first call does, and
raises if it has not been built.
"""
from .binding import (  # noqa: F401
    MoEError,
    lib,
    moe_block_forward,
    moe_block_forward_ws,
    moe_combine,
    moe_expert_down,
    moe_expert_ffn,
    moe_expert_ffn_ws,
    moe_expert_gate_up,
    moe_forward,
    moe_forward_f32,
    moe_forward_host,
    moe_workspace_bytes,
    moe_forward_ws,
    moe_get_device_status,
    moe_permute,
    moe_rmsnorm,
    moe_router_topk,
    moe_set_wait_limit_ns,
    workspace,
)
