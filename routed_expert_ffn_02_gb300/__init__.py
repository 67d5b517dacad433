"""Routed mixture-of-experts FFN layer for NVIDIA GB300 (sm_103a).

The compute lives in libmoe.so (C ABI in include/moe.h, CUDA kernels in
csrc/); this package is its Python binding.  Importing it loads the library
and fails if the library has not been built.
"""
from .binding import (  # noqa: F401
    Shape, Workspace, MoeError, moe_route, moe_permute, moe_permute_noalloc,
    moe_expert_ffn,
    moe_combine, moe_forward, moe_forward_profiled, workspace_size, permute_workspace_size,
    expert_ffn_workspace_size, version, LIB_PATH, EXPORTED,
    PROFILE_EVENTS, PROFILE_STAGES, forward_launches, Stager, layer_weight_bytes,
    pack_layer_weights, Pipe, pipe_workspace_size, DecodeGraph, ExpertCache,
    debug_set_wait_limit,
)
