"""GB300-native hot path of an expert-parallel MoE layer: route -> dispatch -> SwiGLU grouped GEMM
-> combine, as hand-written sm_103a CUDA kernels behind a C ABI (include/moe.h)."""
from .moe import (Graph, GraphedMoeLayer, MoeConfig, MoeError, MoeLayer, Placement, Weights, alloc_workspace, balance,
                  combine, device_status, dispatch, dispatch_noalloc, eplb_plan, expert_ffn, forward, launch_count, load,
                  make_config, quantize_weights_fp8, quantize_weights_nvfp4, route, selftest_wait_timeout, workspace_layout,
                  workspace_size, ws_view)

__all__ = ["Graph", "GraphedMoeLayer", "MoeConfig", "MoeError", "MoeLayer", "Placement", "Weights", "alloc_workspace",
           "balance", "combine", "device_status", "dispatch", "dispatch_noalloc", "eplb_plan", "expert_ffn", "forward",
           "launch_count", "load", "make_config", "quantize_weights_fp8", "quantize_weights_nvfp4", "route",
           "selftest_wait_timeout", "workspace_layout", "workspace_size", "ws_view"]
