"""GB300 (sm_103a) MoE variable-size grouped GEMM with the token permutation
fused into the matmul.

The compute lives in libmgg.so (C ABI in include/mgg.h, CUDA sources in
csrc/); this package is the thin torch binding.  Build the library with
``variable_size_expert_gb300.build.build_library()``.
"""
from .ops import (  # noqa: F401
    RoutingBuffers, debug_tile_schedule, grouped_gemm, grouped_gemm_masked, moe, moe_backward,
    moe_ffn_backward, moe_ffn_forward, moe_forward, new_status, read_status, route, route_noalloc,
    tile_config,
    workspace_bytes,
    quantize_fp8, moe_forward_fp8, grouped_gemm_fp8, grouped_gemm_masked_fp8,
    quantize_fp8_cols, moe_backward_dx_fp8,
)
from . import _lib  # noqa: F401
