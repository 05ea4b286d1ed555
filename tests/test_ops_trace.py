"""The custom-operator layer without a GPU: shape-only ("fake") implementations,
the autograd wiring, symbolic tracing and fullgraph compilation on meta
tensors, and the loud failure on CPU tensors (there is no CPU kernel).

Page: "Add the deepep expert-parallel implementation (huggingface/transformers
#49638)", What this adds, Custom ops.
"""
import pytest
import torch
from torch.fx.experimental.proxy_tensor import make_fx

from combine_topk_multihot_gb300 import ops

T, H, E, K, I, P = 64, 256, 8, 2, 128, 16
C = T * K + E * (P - 1)
ALL_OPS = {"route_to_multihot", "dispatch", "grouped_experts", "combine", "combine_backward",
           "experts_backward", "dispatch_backward", "route_to_multihot_backward"}
ROUTER_OPS = {"router_topk", "router_topk_backward"}


def _inputs(device, grad=True):
    mk = lambda *s, dt=torch.bfloat16: torch.zeros(*s, dtype=dt, device=device)
    x, W1, W2 = mk(T, H), mk(E, 2 * I, H), mk(E, H, I)
    idx = torch.zeros(T, K, dtype=torch.int64, device=device)
    p = torch.zeros(T, K, dtype=torch.float32, device=device)
    if grad:
        for t in (x, p, W1, W2):
            t.requires_grad_(True)
    return x, idx, p, W1, W2


def test_fake_shapes_forward_and_backward():
    x, idx, p, W1, W2 = _inputs("meta")
    out = ops.moe_layer(x, idx, p, W1, W2, P)
    assert out.shape == (T, H) and out.dtype == torch.bfloat16
    out.float().sum().backward()
    assert x.grad.shape == (T, H) and x.grad.dtype == torch.bfloat16
    assert p.grad.shape == (T, K) and p.grad.dtype == torch.float32
    assert W1.grad.shape == W1.shape and W1.grad.dtype == torch.bfloat16
    assert W2.grad.shape == W2.shape and W2.grad.dtype == torch.bfloat16


def test_fake_layout_is_worst_case_sized():
    x, idx, p, W1, W2 = _inputs("meta", grad=False)
    rmap, probs, win, status = torch.ops.moe_gb300.route_to_multihot(idx, p, E)
    assert (rmap.shape, probs.shape, win.shape) == ((T, E),) * 3
    x_disp, *lay = torch.ops.moe_gb300.dispatch(x, rmap, probs, status, K, P)
    assert x_disp.shape == (C, H)
    assert [tuple(t.shape) for t in lay] == [(E,), (E + 1,), (2,), (C,), (C,), (C,), (T * K,), (1,)]
    y, h, o, gu = torch.ops.moe_gb300.grouped_experts(x_disp, W1, W2, lay, T, K, P, False)
    assert (y.shape, h.shape, o.shape, gu.shape) == ((C, H), (C, I), (0, H), (0, 2 * I))
    y, h, o, gu = torch.ops.moe_gb300.grouped_experts(x_disp, W1, W2, lay, T, K, P, True)
    assert (o.shape, gu.shape) == ((C, H), (C, 2 * I))


def _ops_in(graph_module):
    return {str(n.target).split(".")[1] for n in graph_module.graph.nodes
            if n.op == "call_function" and str(n.target).startswith("moe_gb300.")}


def test_symbolic_trace_of_forward_and_backward_uses_only_the_library_ops():
    """Forward and backward traced with symbolic sizes: every step of the
    layer is one of the library's operators; what remains is the cast of the
    weight gradients to the weights' dtype and shape bookkeeping."""
    def step(x, idx, p, W1, W2, g):
        out = ops.moe_layer(x, idx, p, W1, W2, P)
        return (out,) + torch.autograd.grad(out, (x, p, W1, W2), g)

    x, idx, p, W1, W2 = _inputs("cpu")
    g = torch.zeros(T, H, dtype=torch.bfloat16)
    gm = make_fx(step, tracing_mode="symbolic")(x, idx, p, W1, W2, g)
    assert _ops_in(gm) == ALL_OPS
    compute = {str(n.target) for n in gm.graph.nodes if n.op == "call_function"
               and not str(n.target).startswith("moe_gb300.")}
    assert compute <= {"aten.sym_size.int", "aten._to_copy.default", "<built-in function getitem>"}, compute


def test_inference_trace_skips_the_saved_operands_and_the_backward():
    x, idx, p, W1, W2 = _inputs("cpu", grad=False)
    gm = make_fx(lambda *a: ops.moe_layer(*a, P), tracing_mode="symbolic")(x, idx, p, W1, W2)
    assert _ops_in(gm) == {"route_to_multihot", "dispatch", "grouped_experts", "combine"}
    ge = [n for n in gm.graph.nodes if str(n.target).startswith("moe_gb300.grouped_experts")]
    assert ge[0].args[-1] is False


def test_compile_fullgraph_on_meta():
    x, idx, p, W1, W2 = _inputs("meta")
    f = torch.compile(lambda *a: ops.moe_layer(*a, P), fullgraph=True, backend="aot_eager")
    out = f(x, idx, p, W1, W2)
    out.float().sum().backward()
    assert out.shape == (T, H) and W1.grad.shape == W1.shape and p.grad.shape == (T, K)


def test_cpu_tensors_fail_loudly():
    x, idx, p, W1, W2 = _inputs("cpu", grad=False)
    with pytest.raises(NotImplementedError, match="CPU"):
        ops.moe_layer(x, idx, p, W1, W2, P)


def test_layer_from_logits_fake_shapes_and_trace():
    """The router in front of the layer: gradients reach the logits, and the
    traced forward + backward consists of the library's operators."""
    x, idx, p, W1, W2 = _inputs("meta")
    lg = torch.zeros(T, E, dtype=torch.float32, device="meta", requires_grad=True)
    out = ops.moe_layer_from_logits(x, lg, K, W1, W2, P)
    out.float().sum().backward()
    assert lg.grad.shape == (T, E) and lg.grad.dtype == torch.float32

    def step(x, lg, W1, W2, g):
        out = ops.moe_layer_from_logits(x, lg, K, W1, W2, P)
        return (out,) + torch.autograd.grad(out, (x, lg, W1, W2), g)

    x, _, _, W1, W2 = _inputs("cpu")
    lg = torch.zeros(T, E, dtype=torch.float32, requires_grad=True)
    gm = make_fx(step, tracing_mode="symbolic")(x, lg, W1, W2, torch.zeros(T, H, dtype=torch.bfloat16))
    assert _ops_in(gm) == ALL_OPS | ROUTER_OPS
