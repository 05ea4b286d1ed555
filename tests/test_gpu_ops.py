"""The custom-operator layer on the GPU.

Page: "Add the deepep expert-parallel implementation (huggingface/transformers
#49638)", What this adds, Custom ops, and its test list (the capture-and-compile
test): the layer trains through autograd, a CUDA graph captured after an eager
warm-up replays like eager, and torch.compile(fullgraph=True) matches eager.

* the operators' forward and backward equal, bit for bit, the same steps called
  through the binding directly (sync-free, worst-case rows);
* end to end against the fp64 oracle's layer forward and backward;
* torch.library.opcheck of every operator (schema, fake tensors, autograd
  registration);
* CUDA graph replay of forward + backward == eager, bit for bit;
* torch.compile(fullgraph=True) of the layer (the aot_eager backend: the
  trace and the autograd split, with no generated kernels) == eager, bit for bit;
* a bad expert index is reported in the returned device status word;
* the router in front (moe_layer_from_logits) == router then layer, with the
  logits' gradient from the router backward.
"""
import numpy as np
import pytest
import torch

import oracle as O
import synthetic
from tests._bounds import (SAFETY, U_B, U_F, acc, check_within, expert_backward_bound,
                           expert_forward_h_bound)
from tests._util import GEMM_REL_L2, assert_gemm_close, bits, random_routing

pytestmark = pytest.mark.gpu
DEV = "cuda"
BF = torch.bfloat16


@pytest.fixture(scope="module")
def moe():
    assert torch.cuda.is_available(), "GPU tests need a GPU"
    import combine_topk_multihot_gb300 as m
    return m


def _inputs(T, H, E, K, I, seed, drop=0.0, dup=0.0):
    idx, p = random_routing(T, E, K, seed=seed, drop=drop, dup=dup)
    gen = torch.Generator().manual_seed(seed)
    x = torch.randn(T, H, generator=gen).to(BF)
    W1 = (torch.randn(E, 2 * I, H, generator=gen) * 0.02).to(BF)
    W2 = (torch.randn(E, H, I, generator=gen) * 0.02).to(BF)
    g = torch.randn(T, H, generator=gen).to(BF)
    return [t.to(DEV) for t in (x, idx, p, W1, W2, g)]


def _layer(fn, x, idx, p, W1, W2, g):
    """Forward + backward through autograd; returns (out, dx, dp, dW1, dW2)."""
    leaves = [t.detach().clone().requires_grad_(True) for t in (x, p, W1, W2)]
    xs, ps, W1s, W2s = leaves
    out = fn(xs, idx, ps, W1s, W2s)
    out.backward(g)
    return [out.detach()] + [t.grad for t in leaves]


def _direct(moe, x, idx, p, W1, W2, g, P):
    """The same steps called through the binding (no operators, no autograd)."""
    fwd = moe.moe_layer_forward(x, idx, p, W1, W2, P, host_sync=False, save_for_backward=True)
    grad_y, grad_w = moe.moe_combine_backward(g, fwd.layout, o_save=fwd.o)
    gxd, dW1, dW2 = moe.moe_grouped_experts_backward(grad_y, fwd.x_disp, fwd.h, fwd.gu, fwd.layout,
                                                     W1, W2)
    grad_x, grad_probs = moe.moe_dispatch_backward(gxd, fwd.layout, grad_w=grad_w)
    g_topk = moe.moe_route_to_multihot_backward(grad_probs, idx, fwd.winner_slot)
    return [fwd.out, grad_x, g_topk, dW1.to(BF), dW2.to(BF)]


def _same(a, b, what):
    for name, u, v in zip(("out", "grad_x", "grad_topk_probs", "dW1", "dW2"), a, b):
        assert u.dtype == v.dtype and u.shape == v.shape, f"{what} {name}"
        assert torch.equal(u.view(torch.int8), v.view(torch.int8)) if u.dtype != torch.float32 \
            else torch.equal(u, v), f"{what} {name} differs"


CASES = [  # T, H, E, K, I, P, drop, dup
    (64, 256, 8, 2, 128, 16, 0.0, 0.0),
    (300, 512, 8, 2, 256, 16, 0.1, 0.1),
    (20, 512, 12, 1, 384, 1, 0.0, 0.0),
    (260, 768, 12, 3, 256, 128, 0.2, 0.0),
]


@pytest.mark.parametrize("T,H,E,K,I,P,drop,dup", CASES)
def test_ops_equal_the_direct_calls(moe, T, H, E, K, I, P, drop, dup):
    x, idx, p, W1, W2, g = _inputs(T, H, E, K, I, seed=T + H, drop=drop, dup=dup)
    got = _layer(lambda *a: moe.moe_layer(*a, pad_multiple=P), x, idx, p, W1, W2, g)
    ref = _direct(moe, x, idx, p, W1, W2, g, P)
    torch.cuda.synchronize()
    _same(got, ref, "ops vs direct")


def _layer_grad_bounds(fwd, g_bits, W1b, W2b, I):
    """The exact gradients of the layer (the oracle's layout, forward h and
    fp64 chain rule, rounding nothing) and element-wise bounds on a bf16
    implementation's: dW1, dW2 (cast to bf16 by autograd), grad_x (the
    combine of the bf16 grad_x_disp rows) and the routing-weight gradient
    per row (<grad_y, o> with o = h W2^T, which the implementation computes
    from its own h and rounds to bf16)."""
    f = O.bf16_bits_to_f64
    L = fwd["layout"]
    E = W1b.shape[0]
    T, H = g_bits.shape
    K = L["token_row"].shape[1]
    C = L["row_token"].shape[0]
    GYall = f(O.combine_backward(g_bits, L["row_token"]))
    dX = np.zeros((C, H))
    bX = np.zeros((C, H))
    gw = np.zeros(C)
    bgw = np.zeros(C)
    dW1 = np.zeros((E, 2 * I, H))
    dW2 = np.zeros((E, H, I))
    bW1 = np.zeros_like(dW1)
    bW2 = np.zeros_like(dW2)
    for e in range(E):
        R = np.flatnonzero(L["row_expert"] == e)
        if R.size == 0:
            continue
        X, h, GY = f(fwd["x_disp"][R]), f(fwd["h"][R]), GYall[R]
        W1e, W2e = f(W1b[e]), f(W2b[e])
        hf = expert_forward_h_bound(X, W1e, I)
        st, b = expert_backward_bound(X, h, GY, L["row_weight"][R], W1e, W2e, I, h_flips=hf,
                                      dW_bf16=True)
        dX[R], bX[R] = st["dX"], b["dX"]
        dW1[e], dW2[e], bW1[e], bW2[e] = st["dW1"], st["dW2"], b["dW1"], b["dW2"]
        o = h @ W2e.T
        b_o = hf @ np.abs(W2e).T + acc(I) * (np.abs(h) @ np.abs(W2e).T) + U_B * np.abs(o)
        gw[R] = np.sum(GY * o, axis=1)
        bgw[R] = SAFETY * (np.sum(np.abs(GY) * b_o, axis=1) + acc(H) * np.sum(np.abs(GY * o), axis=1))
    tr = L["token_row"]
    gx = np.zeros((T, H))
    bgx = np.zeros((T, H))
    absum = np.zeros((T, H))
    for j in range(K):
        r = tr[:, j]
        ok = r >= 0
        gx[ok] += dX[r[ok]]
        bgx[ok] += bX[r[ok]]
        absum[ok] += np.abs(dX[r[ok]]) + bX[r[ok]]
    bgx += SAFETY * (K * U_F * absum + U_B * np.abs(gx))
    return dict(dW1=dW1, dW2=dW2, bW1=bW1, bW2=bW2, gx=gx, bgx=bgx, gw=gw, bgw=bgw)


@pytest.mark.parametrize("T,H,E,K,I,P,drop,dup", CASES[:2])
def test_ops_match_the_oracle_end_to_end(moe, T, H, E, K, I, P, drop, dup):
    """Forward output within the GEMM tolerance; every gradient element-wise
    within its error bound around the exact chain rule of the oracle's
    forward (tests/_bounds.py), and within rel L2 5e-3 of it."""
    x, idx, p, W1, W2, g = _inputs(T, H, E, K, I, seed=7 * T + H, drop=drop, dup=dup)
    out, dx, dp, dW1, dW2 = _layer(lambda *a: moe.moe_layer(*a, pad_multiple=P), x, idx, p, W1, W2, g)
    torch.cuda.synchronize()
    idx_np = idx.cpu().numpy()
    W1b, W2b = bits(W1), bits(W2)
    C = O.worst_case_capacity(T, E, K, P)
    fwd = O.layer_forward(bits(x), idx_np, p.cpu().numpy(), W1b, W2b, I, P, capacity=C)
    assert_gemm_close(bits(out), fwd["out"], "out")
    ref = _layer_grad_bounds(fwd, bits(g), W1b, W2b, I)

    def rel(gpu, exact, what):
        gpu, exact = np.asarray(gpu, np.float64), np.asarray(exact, np.float64)
        r = np.linalg.norm(gpu - exact) / max(np.linalg.norm(exact), 1e-30)
        assert np.isfinite(gpu).all() and r <= GEMM_REL_L2, f"{what}: rel_l2={r:.3g}"

    gx = O.bf16_bits_to_f64(bits(dx))
    check_within(gx, ref["gx"], ref["bgx"], "grad_x")
    rel(gx, ref["gx"], "grad_x")
    for name, got in (("dW1", dW1), ("dW2", dW2)):
        got = got.float().cpu().numpy()
        check_within(got, ref[name], ref["b" + name[1:]], name)
        rel(got, ref[name], name)
    # grad_topk_probs: the routing-weight gradient of each slot's row (the
    # winner slot of each (token, expert) pair; 0 for dropped and losing slots)
    L = fwd["layout"]
    exact = np.zeros((T, E))
    bound = np.zeros((T, E))
    ok = L["row_token"] >= 0
    exact[L["row_token"][ok], L["row_expert"][ok]] = ref["gw"][ok]
    bound[L["row_token"][ok], L["row_expert"][ok]] = ref["bgw"][ok]
    win = fwd["winner_slot"]
    ex_k = np.zeros((T, K))
    b_k = np.zeros((T, K))
    for t in range(T):
        for k in range(K):
            e = idx_np[t, k]
            if e >= 0 and win[t, e] == k:
                ex_k[t, k], b_k[t, k] = exact[t, e], bound[t, e]
    gp = dp.cpu().numpy().astype(np.float64)
    check_within(gp, ex_k, b_k, "grad_topk_probs")
    rel(gp, ex_k, "grad_topk_probs")


def test_opcheck_every_operator(moe):
    T, H, E, K, I, P = 64, 256, 8, 2, 128, 16
    x, idx, p, W1, W2, g = _inputs(T, H, E, K, I, seed=11, drop=0.1)
    ops = torch.ops.moe_gb300
    utils = ("test_schema", "test_autograd_registration", "test_faketensor")
    rmap, probs, win, status = ops.route_to_multihot(idx, p, E)
    x_disp, *lay = ops.dispatch(x, rmap, probs, status, K, P)
    y, h, o, gu = ops.grouped_experts(x_disp, W1, W2, lay, T, K, P, True)
    grad_y, grad_w = ops.combine_backward(g, o, lay, T, K, P, E)
    gxd, dW1, dW2 = ops.experts_backward(grad_y, x_disp, h, gu, W1, W2, lay, T, K, P)
    grad_x, grad_probs = ops.dispatch_backward(gxd, grad_w, lay, T, K, P, E)
    calls = [
        (ops.route_to_multihot.default, (idx, p, E)),
        (ops.dispatch.default, (x, rmap, probs, status, K, P)),
        (ops.grouped_experts.default, (x_disp, W1, W2, lay, T, K, P, True)),
        (ops.grouped_experts.default, (x_disp, W1, W2, lay, T, K, P, False)),
        (ops.combine.default, (y, lay, T, K, P, E)),
        (ops.combine_backward.default, (g, o, lay, T, K, P, E)),
        (ops.experts_backward.default, (grad_y, x_disp, h, gu, W1, W2, lay, T, K, P)),
        (ops.dispatch_backward.default, (gxd, grad_w, lay, T, K, P, E)),
        (ops.route_to_multihot_backward.default, (grad_probs, idx, win)),
    ]
    for op, args in calls:
        torch.library.opcheck(op, args, test_utils=utils)


@pytest.mark.parametrize("T,H,E,K,I,P", [
    (256, 512, 8, 2, 256, 16),    # one-CTA expert tiles
    (1500, 512, 40, 8, 512, 16),  # CTA-pair expert tiles; eager with per-chunk readiness, captured without
])
def test_cuda_graph_replay_equals_eager(moe, T, H, E, K, I, P):
    """Forward + backward captured once after an eager warm-up, replayed on
    new inputs copied into the static ones: replay == eager, bit for bit."""
    W1, W2 = synthetic.make_weights(E, H, I, 4, device=DEV)
    W1.requires_grad_(True)
    W2.requires_grad_(True)
    sx = torch.zeros(T, H, dtype=BF, device=DEV, requires_grad=True)
    sp = torch.zeros(T, K, dtype=torch.float32, device=DEV, requires_grad=True)
    sidx = torch.zeros(T, K, dtype=torch.int64, device=DEV)
    sg = torch.zeros(T, H, dtype=BF, device=DEV)
    sets = [_inputs(T, H, E, K, I, seed=100 + k, drop=0.05 * k) for k in range(3)]

    def load(s):
        with torch.no_grad():
            sx.copy_(s[0]); sidx.copy_(s[1]); sp.copy_(s[2]); sg.copy_(s[5])

    def step():
        out = moe.moe_layer(sx, sidx, sp, W1, W2, pad_multiple=P)
        return (out,) + torch.autograd.grad(out, (sx, sp, W1, W2), sg)

    side = torch.cuda.Stream()
    side.wait_stream(torch.cuda.current_stream())
    eager = []
    with torch.cuda.stream(side):
        for s in sets:
            load(s)
            eager.append([t.clone() for t in step()])
    torch.cuda.current_stream().wait_stream(side)
    graph = torch.cuda.CUDAGraph()
    with torch.cuda.graph(graph):
        static_out = step()
    for s, ref in zip(reversed(sets), reversed(eager)):
        load(s)
        graph.replay()
        torch.cuda.synchronize()
        _same(list(static_out), ref, "graph replay vs eager")


def test_compile_fullgraph_equals_eager(moe):
    T, H, E, K, I, P = 300, 512, 8, 2, 256, 16
    x, idx, p, W1, W2, g = _inputs(T, H, E, K, I, seed=23, drop=0.1)
    fn = lambda *a: moe.moe_layer(*a, pad_multiple=P)
    compiled = torch.compile(fn, fullgraph=True, backend="aot_eager")
    ref = _layer(fn, x, idx, p, W1, W2, g)
    for _ in range(2):
        got = _layer(compiled, x, idx, p, W1, W2, g)
        torch.cuda.synchronize()
        _same(got, ref, "compiled vs eager")


def test_bad_index_is_reported_in_the_status_word(moe):
    T, H, E, K, I, P = 64, 256, 8, 2, 128, 16
    x, idx, p, W1, W2, g = _inputs(T, H, E, K, I, seed=5)
    idx = idx.clone()
    idx[3, 1] = E          # outside [-1, E): dropped and flagged
    out, status = moe.moe_layer(x, idx, p, W1, W2, pad_multiple=P, return_status=True)
    torch.cuda.synchronize()
    assert int(status.item()) & moe._native.MOE_DEVERR_BAD_INDEX
    # through autograd too: the bad slot gets no gradient
    ps = p.clone().requires_grad_(True)
    out, status = moe.moe_layer(x, idx, ps, W1, W2, pad_multiple=P, return_status=True)
    out.backward(g)
    torch.cuda.synchronize()
    assert int(status.item()) & moe._native.MOE_DEVERR_BAD_INDEX
    assert float(ps.grad[3, 1]) == 0.0 and torch.isfinite(ps.grad).all()
    out, status = moe.moe_layer(x, idx.clamp(max=E - 1), p, W1, W2, pad_multiple=P,
                                return_status=True)
    torch.cuda.synchronize()
    assert int(status.item()) == 0


def test_layer_from_logits_equals_router_then_layer(moe):
    """moe_layer_from_logits == the router's top-k fed to moe_layer, forward
    and backward, bit for bit; the logits' gradient is the router backward of
    the layer's top-k gradient; the router op passes opcheck; compiled == eager."""
    T, H, E, K, I, P = 300, 512, 8, 2, 256, 16
    x, _, _, W1, W2, g = _inputs(T, H, E, K, I, seed=31)
    logits = synthetic.make_logits(T, E, seed=31).to(DEV)

    def run(fn):
        xs = x.detach().clone().requires_grad_(True)
        ls = logits.detach().clone().requires_grad_(True)
        W1s = W1.detach().clone().requires_grad_(True)
        W2s = W2.detach().clone().requires_grad_(True)
        out = fn(xs, ls, W1s, W2s)
        out.backward(g)
        return out.detach(), xs.grad, ls.grad, W1s.grad, W2s.grad

    fused = lambda xs, ls, a, b: moe.moe_layer_from_logits(xs, ls, K, a, b, pad_multiple=P)
    got = run(fused)
    idx, w = moe.moe_router_topk(logits, K)
    ref = _layer(lambda *a: moe.moe_layer(*a, pad_multiple=P), x, idx, w, W1, W2, g)
    torch.cuda.synchronize()
    assert torch.equal(got[0].view(torch.int16), ref[0].view(torch.int16))
    assert torch.equal(got[1].view(torch.int16), ref[1].view(torch.int16))
    assert torch.equal(got[3].view(torch.int16), ref[3].view(torch.int16))
    assert torch.equal(got[4].view(torch.int16), ref[4].view(torch.int16))
    assert torch.equal(got[2], moe.moe_router_topk_backward(ref[2], w, idx, E))
    torch.library.opcheck(torch.ops.moe_gb300.router_topk.default, (logits, K),
                          test_utils=("test_schema", "test_faketensor"))
    torch.library.opcheck(torch.ops.moe_gb300.router_topk_backward.default, (ref[2], w, idx, E),
                          test_utils=("test_schema", "test_autograd_registration", "test_faketensor"))
    compiled = torch.compile(fused, fullgraph=True, backend="aot_eager")
    for _ in range(2):
        c = run(compiled)
        torch.cuda.synchronize()
        for u, v in zip(c, got):
            assert torch.equal(u.view(torch.int8), v.view(torch.int8))
