"""The MoE layer as PyTorch custom operators, with autograd.

Page cited: "Add the deepep expert-parallel implementation
(huggingface/transformers #49638)", What this adds, Custom ops.  There the
dispatch, the combine and the combine's backward become torch.library
operators, each with a shape-only ("fake") implementation for tracing and an
autograd rule, and the dispatch handle, which no operator can carry, travels
between them as its component tensors and is put back together on the far
side.  Here every step of the layer is such an operator: the router (with
its gradient registered on the operator), multihot, dispatch, grouped
experts, combine, and the four backward steps.

Every operator takes the sync-free route: the expanded buffers are sized for
the worst case (T*K + E*(pad_multiple - 1) rows), nothing is read back to the
host, and each output's shape is a function of the input shapes alone -- so the
layer can be captured in a CUDA graph and traced by torch.compile with
fullgraph=True.  The operators are registered for CUDA only (a CPU tensor gets
PyTorch's "no kernel" error) and only marshal arguments to the C library; all
arithmetic runs in its CUDA kernels.
"""
from __future__ import annotations

from typing import List, Tuple

import torch
from torch import Tensor

from . import moe as _m

NS = "moe_gb300"


def _capacity(T, E, K, P):
    return T * K + E * (P - 1)


def _layout(T: int, E: int, K: int, P: int, lay: List[Tensor]) -> _m.Layout:
    return _m.Layout.from_tensors(T, E, K, P, lay)


def _layout_fake(T, E, K, P, device) -> Tuple[Tensor, ...]:
    """Shapes and dtypes of Layout.tensors()."""
    C = _capacity(T, E, K, P)
    i32 = dict(dtype=torch.int32, device=device)
    return (torch.empty(E, **i32), torch.empty(E + 1, **i32), torch.empty(2, **i32),
            torch.empty(C, **i32), torch.empty(C, **i32),
            torch.empty(C, dtype=torch.float32, device=device), torch.empty(T * K, **i32),
            torch.empty(1, **i32))


# ------------------------------------------------------------------ router
@torch.library.custom_op(f"{NS}::router_topk", mutates_args=(), device_types="cuda")
def router_topk(logits: Tensor, top_k: int) -> Tuple[Tensor, Tensor]:
    """(topk_idx int64 [T, K], topk_probs fp32 [T, K]): softmax, top-k, renormalise."""
    return _m.moe_router_topk(logits.contiguous(), top_k)


@router_topk.register_fake
def _(logits, top_k):
    T = logits.shape[0]
    return (torch.empty(T, top_k, dtype=torch.int64, device=logits.device),
            torch.empty(T, top_k, dtype=torch.float32, device=logits.device))


@torch.library.custom_op(f"{NS}::router_topk_backward", mutates_args=(), device_types="cuda")
def router_topk_backward(grad_topk_probs: Tensor, topk_probs: Tensor, topk_idx: Tensor,
                         num_experts: int) -> Tensor:
    """grad_logits fp32 [T, E]."""
    return _m.moe_router_topk_backward(grad_topk_probs.contiguous(), topk_probs, topk_idx, num_experts)


@router_topk_backward.register_fake
def _(grad_topk_probs, topk_probs, topk_idx, num_experts):
    return torch.empty(topk_idx.shape[0], num_experts, dtype=torch.float32, device=topk_idx.device)


def _router_setup(ctx, inputs, output):
    logits, _ = inputs
    idx, w = output
    ctx.save_for_backward(idx, w)
    ctx.num_experts = logits.shape[1]
    ctx.mark_non_differentiable(idx)


def _router_backward(ctx, grad_idx, grad_w):
    idx, w = ctx.saved_tensors
    if grad_w is None:
        return None, None
    return torch.ops.moe_gb300.router_topk_backward(grad_w, w, idx, ctx.num_experts), None


torch.library.register_autograd(f"{NS}::router_topk", _router_backward, setup_context=_router_setup)


# ------------------------------------------------------------------ forward
@torch.library.custom_op(f"{NS}::route_to_multihot", mutates_args=(), device_types="cuda")
def route_to_multihot(topk_idx: Tensor, topk_probs: Tensor,
                      num_experts: int) -> Tuple[Tensor, Tensor, Tensor, Tensor]:
    """(routing_map uint8 [T, E], probs fp32 [T, E], winner_slot int8 [T, E], status int32 [1])."""
    status = torch.zeros(1, dtype=torch.int32, device=topk_idx.device)
    rmap, probs, win = _m.moe_route_to_multihot(topk_idx.contiguous(), topk_probs.contiguous(),
                                                num_experts, status)
    return rmap, probs, win, status


@route_to_multihot.register_fake
def _(topk_idx, topk_probs, num_experts):
    T, d = topk_idx.shape[0], topk_idx.device
    return (torch.empty(T, num_experts, dtype=torch.uint8, device=d),
            torch.empty(T, num_experts, dtype=torch.float32, device=d),
            torch.empty(T, num_experts, dtype=torch.int8, device=d),
            torch.empty(1, dtype=torch.int32, device=d))


@torch.library.custom_op(f"{NS}::dispatch", mutates_args=(), device_types="cuda")
def dispatch(x: Tensor, routing_map: Tensor, probs: Tensor, status: Tensor, top_k: int,
             pad_multiple: int) -> Tuple[Tensor, Tensor, Tensor, Tensor, Tensor, Tensor, Tensor,
                                         Tensor, Tensor]:
    """Sync-free dispatch: (x_disp [C, H], *Layout.tensors()).  ``status``
    carries the multihot step's device error bits; the layout gets a copy."""
    T, H = x.shape
    E = routing_map.shape[1]
    lay = _m.Layout(T, E, top_k, pad_multiple, _capacity(T, E, top_k, pad_multiple),
                    device=x.device, status=status.clone())
    x_disp, _ = _m.moe_dispatch(x.contiguous(), routing_map, probs, lay, host_sync=False)
    return (x_disp,) + lay.tensors()


@dispatch.register_fake
def _(x, routing_map, probs, status, top_k, pad_multiple):
    T, H = x.shape
    E = routing_map.shape[1]
    C = _capacity(T, E, top_k, pad_multiple)
    return (x.new_empty(C, H),) + _layout_fake(T, E, top_k, pad_multiple, x.device)


@torch.library.custom_op(f"{NS}::grouped_experts", mutates_args=(), device_types="cuda")
def grouped_experts(x_disp: Tensor, W1: Tensor, W2: Tensor, lay: List[Tensor], T: int, top_k: int,
                    pad_multiple: int, save_for_backward: bool) -> Tuple[Tensor, Tensor, Tensor, Tensor]:
    """(y [C, H], h [C, I], o [C, H], gu [C, 2I]); o and gu have no rows unless saving."""
    L = _layout(T, W1.shape[0], top_k, pad_multiple, lay)
    r = _m.moe_grouped_experts(x_disp, L, W1.contiguous(), W2.contiguous(), save_o=save_for_backward,
                               save_gu=save_for_backward)
    if save_for_backward:
        return r["y"], r["h"], r["o"], r["gu"]
    return r["y"], r["h"], x_disp.new_empty(0, x_disp.shape[1]), x_disp.new_empty(0, W1.shape[1])


@grouped_experts.register_fake
def _(x_disp, W1, W2, lay, T, top_k, pad_multiple, save_for_backward):
    C, H = x_disp.shape
    twoI = W1.shape[1]
    S = C if save_for_backward else 0
    return x_disp.new_empty(C, H), x_disp.new_empty(C, twoI // 2), x_disp.new_empty(S, H), \
        x_disp.new_empty(S, twoI)


@torch.library.custom_op(f"{NS}::combine", mutates_args=(), device_types="cuda")
def combine(y: Tensor, lay: List[Tensor], T: int, top_k: int, pad_multiple: int,
            num_experts: int) -> Tensor:
    """out [T, H]: the sum of each token's expert rows."""
    return _m.moe_combine(y, _layout(T, num_experts, top_k, pad_multiple, lay))


@combine.register_fake
def _(y, lay, T, top_k, pad_multiple, num_experts):
    return y.new_empty(T, y.shape[1])


# ------------------------------------------------------------------ backward
@torch.library.custom_op(f"{NS}::combine_backward", mutates_args=(), device_types="cuda")
def combine_backward(grad_out: Tensor, o_save: Tensor, lay: List[Tensor], T: int, top_k: int,
                     pad_multiple: int, num_experts: int) -> Tuple[Tensor, Tensor]:
    """(G_o [C, H], grad_w fp32 [C]): grad_out sent along the forward's layout
    with each row's routing weight applied (G_o = w * grad_y, the gradient of
    the experts' pre-weight output), and each row's routing-weight gradient."""
    L = _layout(T, num_experts, top_k, pad_multiple, lay)
    return _m.moe_combine_backward(grad_out.contiguous(), L, o_save=o_save, scaled=True)


@combine_backward.register_fake
def _(grad_out, o_save, lay, T, top_k, pad_multiple, num_experts):
    C = lay[3].shape[0]
    return grad_out.new_empty(C, grad_out.shape[1]), \
        torch.empty(C, dtype=torch.float32, device=grad_out.device)


@torch.library.custom_op(f"{NS}::experts_backward", mutates_args=(), device_types="cuda")
def experts_backward(g_o: Tensor, x_disp: Tensor, h: Tensor, gu_save: Tensor, W1: Tensor,
                     W2: Tensor, lay: List[Tensor], T: int, top_k: int,
                     pad_multiple: int) -> Tuple[Tensor, Tensor, Tensor]:
    """(grad_x_disp [C, H] bf16, dW1 fp32 [E, 2I, H], dW2 fp32 [E, H, I]) from
    combine_backward's G_o."""
    L = _layout(T, W1.shape[0], top_k, pad_multiple, lay)
    return _m.moe_grouped_experts_backward(g_o, x_disp, h, gu_save, L, W1.contiguous(),
                                           W2.contiguous(), scaled=True)


@experts_backward.register_fake
def _(g_o, x_disp, h, gu_save, W1, W2, lay, T, top_k, pad_multiple):
    return (x_disp.new_empty(x_disp.shape),
            torch.empty(W1.shape, dtype=torch.float32, device=W1.device),
            torch.empty(W2.shape, dtype=torch.float32, device=W2.device))


@torch.library.custom_op(f"{NS}::dispatch_backward", mutates_args=(), device_types="cuda")
def dispatch_backward(grad_x_disp: Tensor, grad_w: Tensor, lay: List[Tensor], T: int, top_k: int,
                      pad_multiple: int, num_experts: int) -> Tuple[Tensor, Tensor]:
    """(grad_x [T, H], grad_probs fp32 [T, E])."""
    L = _layout(T, num_experts, top_k, pad_multiple, lay)
    return _m.moe_dispatch_backward(grad_x_disp, L, grad_w=grad_w)


@dispatch_backward.register_fake
def _(grad_x_disp, grad_w, lay, T, top_k, pad_multiple, num_experts):
    return (grad_x_disp.new_empty(T, grad_x_disp.shape[1]),
            torch.empty(T, num_experts, dtype=torch.float32, device=grad_x_disp.device))


@torch.library.custom_op(f"{NS}::route_to_multihot_backward", mutates_args=(), device_types="cuda")
def route_to_multihot_backward(grad_probs: Tensor, topk_idx: Tensor, winner_slot: Tensor) -> Tensor:
    """grad_topk_probs fp32 [T, K]."""
    return _m.moe_route_to_multihot_backward(grad_probs.contiguous(), topk_idx.contiguous(),
                                             winner_slot)


@route_to_multihot_backward.register_fake
def _(grad_probs, topk_idx, winner_slot):
    return torch.empty(topk_idx.shape, dtype=torch.float32, device=topk_idx.device)


# ------------------------------------------------------------------ the layer
_ops = torch.ops.moe_gb300


class MoELayerFunction(torch.autograd.Function):
    """out = combine(experts(dispatch(x, multihot(topk_idx, topk_probs)), W1, W2)).

    The backward gives gradients for x, topk_probs, W1 and W2.  The kernels
    accumulate the weight gradients in fp32; autograd wants them in the
    weights' own dtype, so they are cast on the way out."""

    @staticmethod
    def forward(ctx, x, topk_idx, topk_probs, W1, W2, pad_multiple: int):
        T, K = topk_idx.shape
        E = W1.shape[0]
        rmap, probs, win, status = _ops.route_to_multihot(topk_idx, topk_probs, E)
        x_disp, *lay = _ops.dispatch(x, rmap, probs, status, K, pad_multiple)
        y, h, o, gu = _ops.grouped_experts(x_disp, W1, W2, lay, T, K, pad_multiple, True)
        out = _ops.combine(y, lay, T, K, pad_multiple, E)
        ctx.save_for_backward(topk_idx, win, x_disp, h, o, gu, W1, W2, *lay)
        ctx.meta = (T, K, E, pad_multiple)
        status = lay[-1]
        ctx.mark_non_differentiable(status)
        ctx.set_materialize_grads(False)   # no zero gradient is made for status
        return out, status

    @staticmethod
    def backward(ctx, grad_out, _grad_status):
        topk_idx, win, x_disp, h, o, gu, W1, W2, *lay = ctx.saved_tensors
        T, K, E, P = ctx.meta
        g_o, grad_w = _ops.combine_backward(grad_out, o, lay, T, K, P, E)
        gxd, dW1, dW2 = _ops.experts_backward(g_o, x_disp, h, gu, W1, W2, lay, T, K, P)
        grad_x, grad_probs = _ops.dispatch_backward(gxd, grad_w, lay, T, K, P, E)
        grad_topk = _ops.route_to_multihot_backward(grad_probs, topk_idx, win)
        return grad_x, None, grad_topk, dW1.to(W1.dtype), dW2.to(W2.dtype), None


def moe_layer(x: Tensor, topk_idx: Tensor, topk_probs: Tensor, W1: Tensor, W2: Tensor,
              pad_multiple: int = 1, return_status: bool = False):
    """The whole layer (a1..a6 forward, a7..a10 backward) as one differentiable
    call on the sync-free route.  Under torch.no_grad() the gate/up values and
    the pre-weight outputs are not saved.  With ``return_status`` it returns
    (out, status): status is the device's error word (MOE_DEVERR_* bits; 1 = an
    expert index outside [-1, E) was seen and dropped), left on the device so
    that reading it is the caller's choice of synchronisation point."""
    if torch.is_grad_enabled() and any(t.requires_grad for t in (x, topk_probs, W1, W2)):
        out, status = MoELayerFunction.apply(x, topk_idx, topk_probs, W1, W2, pad_multiple)
    else:
        T, K = topk_idx.shape
        E = W1.shape[0]
        rmap, probs, win, status = _ops.route_to_multihot(topk_idx, topk_probs, E)
        x_disp, *lay = _ops.dispatch(x, rmap, probs, status, K, pad_multiple)
        y, h, o, gu = _ops.grouped_experts(x_disp, W1, W2, lay, T, K, pad_multiple, False)
        out = _ops.combine(y, lay, T, K, pad_multiple, E)
        status = lay[-1]
    return (out, status) if return_status else out


def moe_layer_from_logits(x: Tensor, router_logits: Tensor, top_k: int, W1: Tensor, W2: Tensor,
                          pad_multiple: int = 1, return_status: bool = False):
    """The router (softmax, top-k, renormalise) and the layer; gradients also
    reach the router logits."""
    topk_idx, topk_probs = torch.ops.moe_gb300.router_topk(router_logits, top_k)
    return moe_layer(x, topk_idx, topk_probs, W1, W2, pad_multiple, return_status)
