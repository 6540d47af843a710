"""GB300-native routed mixture-of-experts hot path (router, quantized SwiGLU experts,
ordered top-k combine) behind the C ABI of include/rl_moe.h.

The functions re-exported here have the names of the C entry points and only marshal
arguments; the CUDA library `_build/librlmoe.so` does all the work and must be built first
(`quantized_moe_expert_rl_gb300.build.build()`).
"""
from ._lib import (  # noqa: F401
    RL_NO_EARLY_OUT, RlError, RlShape, load, moe_decode, moe_decode_workspace_bytes, moe_prefill_chunk,
    moe_prefill_chunk_f32, moe_prefill_workspace_bytes, rl_abi_version, rl_build_pairs,
    rl_build_pairs_workspace_bytes, rl_fill_missing, rl_fill_workspace_bytes, rl_host_device_pointer,
    rl_record_bytes, rl_resolve_slots, rl_rmsnorm, rl_route, rl_route_workspace_bytes,
)
