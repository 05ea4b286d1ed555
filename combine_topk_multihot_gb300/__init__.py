"""Single-GPU MoE dispatch / experts / combine for GB300 (sm_103a).

The compute path is the CUDA library ``_lib/libmoe.so`` (C ABI in
``include/moe.h``); this package is its Python binding.  Importing it fails
loudly if the library has not been built -- there is no CPU fallback.
``ops`` registers every step as a PyTorch custom operator (``torch.ops.moe_gb300``)
and ``moe_layer`` is the differentiable layer built from them.
"""
from .moe import (Layout, MoEError, ForwardResult, worst_case_rows, moe_router_topk,
                  moe_router_topk_backward, moe_route_to_multihot,
                  moe_dispatch, moe_dispatch_topk, moe_dispatch_fp8, moe_dispatch_topk_fp8, moe_quantize_fp8,
                  moe_grouped_experts_fp8,
                  moe_dispatch_layout, moe_grouped_experts_gather,
                  moe_grouped_experts, moe_combine, moe_combine_backward,
                  moe_dispatch_backward, moe_route_to_multihot_backward, moe_layer_forward,
                  moe_grouped_experts_backward)
from . import _native
from . import ops
from .ops import moe_layer, moe_layer_from_logits

__all__ = [
    "Layout", "MoEError", "ForwardResult", "worst_case_rows", "moe_router_topk",
    "moe_router_topk_backward", "moe_route_to_multihot",
    "moe_dispatch", "moe_dispatch_topk", "moe_dispatch_fp8", "moe_dispatch_topk_fp8", "moe_quantize_fp8",
    "moe_grouped_experts_fp8",
    "moe_dispatch_layout", "moe_grouped_experts_gather",
    "moe_grouped_experts", "moe_combine", "moe_combine_backward",
    "moe_dispatch_backward", "moe_route_to_multihot_backward", "moe_layer_forward",
    "moe_grouped_experts_backward", "_native", "ops", "moe_layer", "moe_layer_from_logits",
]
