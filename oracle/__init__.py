"""CPU oracle for the MoE dispatch / experts / combine layer.

TEST INFRASTRUCTURE ONLY.  Nothing on the product path may import, call or
execute anything in this package: only the test suite, the smoke check in
``__graft_entry__`` and the CPU-baseline leg of ``bench.py`` use it.  It shares
no code with the CUDA library (no kernels, headers, helpers, tables or
constants); the only thing both sides share is the seeded input generator in
``synthetic``, which holds none of the method's arithmetic.

It is a plain, slow, obviously-correct restatement of what the pages define
(and, in ``router.py``, of the router step in front of the path; in ``fp8.py``,
of the FP8 dispatch and gate/up GEMM):

* "feat: add hybridep (NVIDIA-NeMo/Automodel #1333)" -- the preprocessing
  that maps top-k indices to a multihot ``routing_map`` with fp32 ``probs``
  (Changelog; review of ``dispatch()``: fp32 probs, ``tokens_per_expert``,
  ``pad_multiple``, the permuted-row total as the sum of the counts; the
  review's list of multihot test cases: basic, topk=1, all -1, partial -1,
  single token, a token naming one expert twice).
* "Add the deepep expert-parallel implementation (huggingface/transformers
  #49638)" -- What this adds: Expanded layout (every (token, expert) pair gets
  its own row, rows are grouped per expert and carry the pair's weight; the
  weight is applied inside the experts and the combine just adds rows up);
  Eager vs captured (either the exact row count read back to the host, or a
  buffer big enough for any routing whose unused rows are zero and belong to
  a sentinel expert that no expert computes); Training (the combine's gradient
  is a dispatch along the same layout, and the routing weights get gradients
  through the combine); Benchmarks (the experts are bf16 grouped GEMMs).

Floating point: expert math in fp64 from the exact bf16 values, with the
roundings the layer itself has (h and y to bf16); combine sums in fp32 in a
fixed order and rounds once to bf16.  The expert backward is the chain rule
of that forward in fp64 with no rounding at all (its bf16 outputs are
rounded once at the end); the test suite holds a bf16 implementation of it
to an element-wise forward-error bound around this exact value.

Every function is pinned by ``tests/test_oracle_*.py`` against something other
than itself (hand-written cases, library routines, closed forms, brute force,
finite differences).  No function here is "parity unpinned".
"""
from .bf16 import (bf16_bits_to_f64, bf16_bits_to_f32, f64_to_bf16_bits,
                   f32_to_bf16_bits, bf16_round_f64)
from .moe_oracle import (OracleIndexError, OracleCapacityError, sentinel_expert,
                         route_to_multihot, counts_and_offsets, build_layout,
                         dispatch, expert_forward_f64, grouped_experts, combine,
                         combine_backward, routing_weight_grad,
                         expert_backward_f64, expert_backward_steps,
                         grouped_experts_backward,
                         backward_scale, backward_gate_up, backward_swiglu,
                         backward_gemms,
                         dispatch_backward, route_to_multihot_backward,
                         layer_forward, layer_backward, worst_case_capacity)
from .router import router_topk, router_topk_f64, router_topk_backward
from .fp8 import (e4m3_round, e4m3_to_bits, e4m3_bits_to_f64, quantize_rows, dispatch_fp8,
                  expert_gate_up_fp8, grouped_experts_fp8)

__all__ = [
    "bf16_bits_to_f64", "bf16_bits_to_f32", "f64_to_bf16_bits", "f32_to_bf16_bits",
    "bf16_round_f64", "OracleIndexError", "OracleCapacityError", "sentinel_expert",
    "route_to_multihot", "counts_and_offsets", "build_layout", "dispatch",
    "expert_forward_f64", "grouped_experts", "combine", "combine_backward",
    "routing_weight_grad", "expert_backward_f64", "expert_backward_steps",
    "grouped_experts_backward",
    "backward_scale", "backward_gate_up", "backward_swiglu", "backward_gemms",
    "dispatch_backward", "route_to_multihot_backward", "layer_forward",
    "layer_backward", "worst_case_capacity", "router_topk", "router_topk_f64",
    "router_topk_backward", "e4m3_round", "e4m3_to_bits", "e4m3_bits_to_f64", "quantize_rows",
    "dispatch_fp8", "expert_gate_up_fp8", "grouped_experts_fp8",
]
