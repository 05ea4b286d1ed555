"""Pins for the oracle's SwiGLU experts and the whole backward (CPU only).

* E = 1 with every token on expert 0 reduces the grouped experts to a dense
  SwiGLU MLP, computed here with torch's own fp64 ops (a library routine
  independent of the oracle's numpy code); gate/up order, the bf16 rounding of
  h and of w*o are all visible there.
* A pure-Python brute force of the same formulas on a tiny shape.
* The fp64 backward equals torch autograd of the same real-valued layer, and
  central finite differences of the oracle's own forward.
"""
import numpy as np
import pytest
import torch
import torch.nn.functional as F

import oracle as O


def _bf(a):
    return O.f64_to_bf16_bits(np.asarray(a, dtype=np.float64))


def _f(bits):
    return O.bf16_bits_to_f64(bits)


def _ulp(v):
    return np.ldexp(1.0, np.frexp(np.abs(v))[1] - 8)


@pytest.mark.parametrize("n,H,I", [(1, 16, 8), (37, 64, 32), (130, 256, 128)])
def test_single_expert_is_dense_swiglu(n, H, I):
    rng = np.random.default_rng(n)
    x = _bf(rng.standard_normal((n, H)))
    W1 = _bf(rng.standard_normal((1, 2 * I, H)) * 0.05)
    W2 = _bf(rng.standard_normal((1, H, I)) * 0.05)
    w = rng.random(n).astype(np.float32)
    y, h, o = O.grouped_experts(x, np.zeros(n, np.int32), w, W1, W2, I)

    X = torch.from_numpy(_f(x))
    Wg = torch.from_numpy(_f(W1[0, :I]))
    Wu = torch.from_numpy(_f(W1[0, I:]))
    Wd = torch.from_numpy(_f(W2[0]))
    h_ref = F.silu(X @ Wg.T) * (X @ Wu.T)
    # h is the real value rounded once to bf16: within half a bf16 ulp (one ulp
    # of slack for the different fp64 summation order near a rounding boundary)
    assert np.all(np.abs(_f(h) - h_ref.numpy()) <= _ulp(h_ref.numpy()) + 1e-300)
    # feed the oracle's own rounded h to the down projection so y is comparable
    o_ref = torch.from_numpy(_f(h)) @ Wd.T
    y_ref = torch.from_numpy(w.astype(np.float64))[:, None] * o_ref
    assert np.all(np.abs(_f(y) - y_ref.numpy()) <= _ulp(y_ref.numpy()) / 2 + 1e-300)
    assert np.all(np.abs(_f(o) - o_ref.numpy()) <= _ulp(o_ref.numpy()) / 2 + 1e-300)


def test_brute_force_tiny_expert():
    rng = np.random.default_rng(7)
    n, H, I = 3, 4, 2
    X = _f(_bf(rng.standard_normal((n, H))))
    W1 = _f(_bf(rng.standard_normal((2 * I, H))))
    W2 = _f(_bf(rng.standard_normal((H, I))))
    w = np.array([0.5, 1.0, 0.25])
    ident = lambda a: np.asarray(a, dtype=np.float64)
    y, h, o = O.expert_forward_f64(X, W1, W2, w, I, rnd=ident)
    for r in range(n):
        for i in range(I):
            g = sum(X[r, k] * W1[i, k] for k in range(H))
            u = sum(X[r, k] * W1[I + i, k] for k in range(H))
            hh = g / (1.0 + np.exp(-g)) * u
            assert abs(h[r, i] - hh) <= 1e-12 * (1 + abs(hh))
        for j in range(H):
            oo = sum(h[r, i] * W2[j, i] for i in range(I))
            assert abs(o[r, j] - oo) <= 1e-12 * (1 + abs(oo))
            assert abs(y[r, j] - w[r] * oo) <= 1e-12 * (1 + abs(oo))


def test_rows_go_to_their_own_expert():
    """Interleaved rows of three experts give, row by row, what each expert
    alone gives; sentinel rows stay zero."""
    rng = np.random.default_rng(8)
    E, H, I, C = 3, 32, 16, 20
    x = _bf(rng.standard_normal((C, H)))
    W1 = _bf(rng.standard_normal((E, 2 * I, H)) * 0.1)
    W2 = _bf(rng.standard_normal((E, H, I)) * 0.1)
    re = rng.integers(0, E + 1, size=C).astype(np.int32)  # E = sentinel
    w = rng.random(C).astype(np.float32)
    y, h, o = O.grouped_experts(x, re, w, W1, W2, I)
    for r in range(C):
        if re[r] == E:
            assert not y[r].any() and not h[r].any()
            continue
        ye, he, _ = O.expert_forward_f64(_f(x[r:r + 1]), _f(W1[re[r]]), _f(W2[re[r]]), w[r:r + 1], I)
        assert np.array_equal(y[r], _bf(ye[0])) and np.array_equal(h[r], _bf(he[0]))


# ---------------------------------------------------------------- backward

def _layer_f64(x, idx, p, W1, W2, I, P=4):
    """The layer as a real-valued function (no roundings), built from the
    oracle's layout and fp64 expert forward."""
    E = W1.shape[0]
    m, probs, win = O.route_to_multihot(idx, p, E)
    L = O.build_layout(m, probs, idx.shape[1], P)
    ident = lambda a: np.asarray(a, dtype=np.float64)
    T, H = x.shape
    out = np.zeros((T, H))
    for r in range(L["capacity"]):
        t, e = L["row_token"][r], L["row_expert"][r]
        if t < 0:
            continue
        y, _, _ = O.expert_forward_f64(x[t:t + 1], W1[e], W2[e], np.array([probs[t, e]], np.float64), I, rnd=ident)
        out[t] += y[0]
    return out, L, win


def _oracle_grads_f64(x, idx, p, W1, W2, I, G, P=4):
    """The oracle's backward, in fp64 with no roundings."""
    E = W1.shape[0]
    T, H = x.shape
    out, L, win = _layer_f64(x, idx, p, W1, W2, I, P)
    ident = lambda a: np.asarray(a, dtype=np.float64)
    gx = np.zeros_like(x)
    gW1 = np.zeros_like(W1)
    gW2 = np.zeros_like(W2)
    C = L["capacity"]
    gw = np.zeros(C)
    for e in range(E):
        R = np.flatnonzero(L["row_expert"] == e)
        if R.size == 0:
            continue
        toks = L["row_token"][R]
        X = x[toks]
        w = L["row_weight"][R].astype(np.float64)
        _, h, o = O.expert_forward_f64(X, W1[e], W2[e], w, I, rnd=ident)
        GY = G[toks]                      # combine backward: a dispatch of G
        gw[R] = np.sum(GY * o, axis=1)    # routing-weight gradient
        dX, d1, d2 = O.expert_backward_f64(X, h, GY, w, W1[e], W2[e], I)
        gW1[e] += d1
        gW2[e] += d2
        np.add.at(gx, toks, dX)           # dispatch backward: sum per token
    gprobs = np.zeros((T, E))
    ok = L["row_token"] >= 0
    gprobs[L["row_token"][ok], L["row_expert"][ok]] = gw[ok]
    gtopk = O.route_to_multihot_backward(gprobs.astype(np.float32), idx, win)
    return out, gx, gW1, gW2, gprobs, gtopk


def _tiny_problem(seed, T=6, H=8, E=3, K=2, I=4, dup=True):
    rng = np.random.default_rng(seed)
    x = rng.standard_normal((T, H))
    idx = np.stack([rng.permutation(E)[:K] for _ in range(T)]).astype(np.int64)
    idx[1, 1] = -1
    if dup:
        idx[2, 1] = idx[2, 0]
    p = rng.random((T, K)).astype(np.float32).astype(np.float64)
    W1 = rng.standard_normal((E, 2 * I, H)) * 0.5
    W2 = rng.standard_normal((E, H, I)) * 0.5
    G = rng.standard_normal((T, H))
    return x, idx, p, W1, W2, I, G


def test_backward_matches_torch_autograd():
    x, idx, p, W1, W2, I, G = _tiny_problem(11)
    out, gx, gW1, gW2, gprobs, gtopk = _oracle_grads_f64(x, idx, p, W1, W2, I, G)
    T, K = idx.shape
    E = W1.shape[0]
    X = torch.tensor(x, requires_grad=True)
    Pp = torch.tensor(p, requires_grad=True)
    A = torch.tensor(W1, requires_grad=True)
    B = torch.tensor(W2, requires_grad=True)
    outs = []
    for t in range(T):
        # the multihot: each distinct expert once, weighted by its last slot
        last = {}
        for k in range(K):
            if idx[t, k] >= 0:
                last[int(idx[t, k])] = k
        acc = torch.zeros(X.shape[1], dtype=torch.float64)
        for e, k in sorted(last.items()):
            g = A[e, :I] @ X[t]
            u = A[e, I:] @ X[t]
            acc = acc + Pp[t, k] * (B[e] @ (F.silu(g) * u))
        outs.append(acc)
    OUT = torch.stack(outs)
    assert np.allclose(OUT.detach().numpy(), out, rtol=1e-12, atol=1e-12)
    (OUT * torch.tensor(G)).sum().backward()
    assert np.allclose(X.grad.numpy(), gx, rtol=1e-10, atol=1e-12)
    assert np.allclose(A.grad.numpy(), gW1, rtol=1e-10, atol=1e-12)
    assert np.allclose(B.grad.numpy(), gW2, rtol=1e-10, atol=1e-12)
    assert np.allclose(Pp.grad.numpy(), gtopk, rtol=1e-6, atol=1e-7)  # gtopk is fp32


def test_backward_matches_finite_differences():
    x, idx, p, W1, W2, I, G = _tiny_problem(12, T=5, H=6, E=4, K=3, I=3)
    _, gx, gW1, gW2, gprobs, gtopk = _oracle_grads_f64(x, idx, p, W1, W2, I, G)
    loss = lambda x_, p_, a_, b_: float(np.sum(_layer_f64(x_, idx, p_, a_, b_, I)[0] * G))
    eps = 1e-6
    rng = np.random.default_rng(0)
    for _ in range(6):
        t, h = rng.integers(0, x.shape[0]), rng.integers(0, x.shape[1])
        d = np.zeros_like(x); d[t, h] = eps
        fd = (loss(x + d, p, W1, W2) - loss(x - d, p, W1, W2)) / (2 * eps)
        assert abs(fd - gx[t, h]) <= 1e-6 * (1 + abs(fd))
        e, i, h = rng.integers(0, W1.shape[0]), rng.integers(0, W1.shape[1]), rng.integers(0, W1.shape[2])
        d = np.zeros_like(W1); d[e, i, h] = eps
        fd = (loss(x, p, W1 + d, W2) - loss(x, p, W1 - d, W2)) / (2 * eps)
        assert abs(fd - gW1[e, i, h]) <= 1e-6 * (1 + abs(fd))
        e, h, i = rng.integers(0, W2.shape[0]), rng.integers(0, W2.shape[1]), rng.integers(0, W2.shape[2])
        d = np.zeros_like(W2); d[e, h, i] = eps
        fd = (loss(x, p, W1, W2 + d) - loss(x, p, W1, W2 - d)) / (2 * eps)
        assert abs(fd - gW2[e, h, i]) <= 1e-6 * (1 + abs(fd))
    # the layer is linear in the routing weights, which travel as fp32, so a
    # large step is exact up to the fp32 rounding of p + d
    for t in range(idx.shape[0]):
        for k in range(idx.shape[1]):
            d = np.zeros_like(p); d[t, k] = 2.0**-6
            fd = (loss(x, p + d, W1, W2) - loss(x, p - d, W1, W2)) / (2 * 2.0**-6)
            assert abs(fd - gtopk[t, k]) <= 1e-5 * (1 + abs(fd)), (t, k)


def test_bits_backward_wrappers_route_rows():
    """The bit-level wrappers give, row by row and expert by expert, what the
    fp64 core gives on the same (bf16-valued) inputs."""
    rng = np.random.default_rng(13)
    E, H, I, C = 3, 16, 8, 14
    xd = _bf(rng.standard_normal((C, H)))
    gy = _bf(rng.standard_normal((C, H)))
    hb = _bf(rng.standard_normal((C, I)))
    ob = _bf(rng.standard_normal((C, H)))
    W1 = _bf(rng.standard_normal((E, 2 * I, H)) * 0.1)
    W2 = _bf(rng.standard_normal((E, H, I)) * 0.1)
    re = rng.integers(0, E + 1, size=C).astype(np.int32)
    w = rng.random(C).astype(np.float32)
    gx, dW1, dW2 = O.grouped_experts_backward(gy, xd, hb, re, w, W1, W2, I)
    gw = O.routing_weight_grad(gy, ob, re, E)
    for e in range(E):
        R = np.flatnonzero(re == e)
        dX, d1, d2 = O.expert_backward_f64(_f(xd[R]), _f(hb[R]), _f(gy[R]), w[R], _f(W1[e]), _f(W2[e]), I)
        assert np.array_equal(gx[R], _bf(dX))
        assert np.array_equal(dW1[e], d1.astype(np.float32))
        assert np.array_equal(dW2[e], d2.astype(np.float32))
    for r in range(C):
        if re[r] == E:
            assert gw[r] == 0 and not gx[r].any()
        else:
            assert gw[r] == np.float32(np.dot(_f(gy[r]), _f(ob[r])))


def test_multihot_backward_winner_slots():
    idx = np.array([[2, 2, 0], [1, -1, 1], [-1, -1, -1]])
    p = np.ones((3, 3), np.float32)
    _, _, win = O.route_to_multihot(idx, p, 4)
    gp = np.arange(12, dtype=np.float32).reshape(3, 4) + 1
    g = O.route_to_multihot_backward(gp, idx, win)
    # token 0: slot 1 is the winner for expert 2, slot 0 (a losing duplicate) gets 0
    assert g.tolist() == [[0.0, 3.0, 1.0], [0.0, 0.0, 6.0], [0.0, 0.0, 0.0]]


def test_backward_has_no_rounding():
    """The chain rule is exact fp64 with no bf16 rounding anywhere: scaling
    grad_y by a power of two (exact in fp64) scales every gradient exactly,
    and a grad_y holding values that no bf16 can hold goes through unchanged
    (a rounding of G_o to bf16 would lose those bits)."""
    rng = np.random.default_rng(21)
    n, H, I = 9, 16, 8
    X = rng.standard_normal((n, H))
    W1 = rng.standard_normal((2 * I, H)) * 0.3
    W2 = rng.standard_normal((H, I)) * 0.3
    h = rng.standard_normal((n, I))
    GY = rng.standard_normal((n, H))
    w = rng.random(n)
    a = O.expert_backward_f64(X, h, GY, w, W1, W2, I)
    b = O.expert_backward_f64(X, h, GY * 2.0**-20, w, W1, W2, I)
    for u, v in zip(a, b):
        assert np.array_equal(u * 2.0**-20, v)
    # h = I_n (n = I) and w = 1: dW2 = G_o^T is grad_y itself, bit for bit
    n = I
    h = np.eye(n)
    X = rng.standard_normal((n, H))
    GY = rng.standard_normal((n, H))
    dW2 = O.expert_backward_f64(X, h, GY, np.ones(n), W1, W2, I)[2]
    assert np.array_equal(dW2, GY.T)
    assert not np.array_equal(dW2, O.bf16_round_f64(dW2))
