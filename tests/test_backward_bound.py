"""Pins for the expert-backward error bound (tests/_bounds.py), on the CPU.

The GPU tests hold the library's a9 outputs to an element-wise bound around
the oracle's exact fp64 chain rule.  Here the bound itself is checked from
both sides, on inputs drawn like the layers' (x ~ N(0,1) and grad ~ N(0,1)
in bf16, routing weights in (0, 1), bf16 weights whose spread gives gate
values like the layers' N(0, 0.02) weights at H = 2048), plus a case with
large gate values where silu saturates, and experts with one and three rows:

* sufficient: a bf16 implementation emulated in numpy -- every intermediate
  a plain bf16 chain rule would round (G_o, G_h, g, u, G_g, G_u) rounded to
  bf16, every GEMM an fp32 product -- stays inside the bound, with margin;
* tight enough: the same emulation with a planted mistake (silu' without its
  second factor, G_u taken with silu' instead of silu, the routing weight
  dropped, the gate and up halves of the weight gradient swapped, h read from
  the neighbouring row, a sign flip in G_g) falls outside it.
"""
import numpy as np
import pytest

import oracle as O
from tests._bounds import expert_backward_bound, expert_forward_h_bound


def _bf(a):
    return O.bf16_round_f64(np.asarray(a, dtype=np.float64))


def _mm(a, b):
    """fp32 GEMM (numpy's sgemm), returned as fp64."""
    return (np.asarray(a, np.float32) @ np.asarray(b, np.float32)).astype(np.float64)


def _emulated_bf16_backward(X, h, GY, w, W1e, W2e, I, mistake=None):
    f32 = lambda a: np.asarray(a, np.float32)
    G_o = _bf(f32(w)[:, None] * f32(GY))
    if mistake == "no_weight":
        G_o = _bf(GY)
    G_h = _bf(_mm(G_o, W2e))
    g = _bf(_mm(X, W1e[:I].T))
    u = _bf(_mm(X, W1e[I:].T))
    s = (1.0 / (1.0 + np.exp(-f32(g)))).astype(np.float64)
    silu = g * s
    dsilu = s * (1.0 + g * (1.0 - s))
    if mistake == "dsilu_is_sigmoid":
        dsilu = s
    G_g = _bf(G_h * u * dsilu)
    G_u = _bf(G_h * (dsilu if mistake == "gu_with_dsilu" else silu))
    if mistake == "sign":
        G_g = -G_g
    G_gu = np.concatenate([G_g, G_u], axis=1)
    dX = _bf(_mm(G_gu, W1e))
    dW1 = _mm(G_gu.T, X)
    if mistake == "swap_halves":
        dW1 = np.concatenate([dW1[I:], dW1[:I]], axis=0)
    hh = np.roll(h, 1, axis=0) if mistake == "h_row_shift" else h
    dW2 = _mm(G_o.T, hh)
    return dX, dW1, dW2


def _problem(seed, n, H, I, wstd=0.02):
    rng = np.random.default_rng(seed)
    X = _bf(rng.standard_normal((n, H)))
    W1 = _bf(rng.standard_normal((2 * I, H)) * wstd)
    W2 = _bf(rng.standard_normal((H, I)) * wstd)
    GY = _bf(rng.standard_normal((n, H)))
    w = rng.random(n).astype(np.float32).astype(np.float64)
    g, u = O.backward_gate_up(X, W1, I)
    h = _bf(g / (1 + np.exp(-g)) * u)
    return X, h, GY, w, W1, W2


CASES = [(0, 200, 256, 128, 0.06), (1, 64, 512, 256, 0.045), (2, 130, 256, 128, 0.2),
         (3, 400, 2048, 256, 0.02), (4, 1, 256, 128, 0.06), (5, 3, 512, 128, 0.03)]


def _ratios(got, st, bound):
    names = ("dX", "dW1", "dW2")
    return {k: np.abs(np.asarray(v) - st[k]) / np.maximum(bound[k], 1e-300) for k, v in zip(names, got)}


@pytest.mark.parametrize("seed,n,H,I,wstd", CASES)
def test_bf16_emulation_is_inside_the_bound(seed, n, H, I, wstd):
    X, h, GY, w, W1, W2 = _problem(seed, n, H, I, wstd)
    st, bound = expert_backward_bound(X, h, GY, w, W1, W2, I)
    r = _ratios(_emulated_bf16_backward(X, h, GY, w, W1, W2, I), st, bound)
    # the emulation's rounding of G_o is one of the bound's own terms, taken
    # twice (SAFETY): at most half the bound, up to the fp32 accumulation
    for k, v in r.items():
        assert v.max() <= 0.55, f"{k}: worst error is {v.max():.3g} of the bound"


@pytest.mark.parametrize("mistake,out", [
    ("dsilu_is_sigmoid", "dW1"), ("gu_with_dsilu", "dW1"), ("no_weight", "dW2"),
    ("swap_halves", "dW1"), ("h_row_shift", "dW2"), ("sign", "dX"),
])
@pytest.mark.parametrize("seed,n,H,I,wstd", CASES[:4])
def test_planted_mistakes_leave_the_bound(mistake, out, seed, n, H, I, wstd):
    X, h, GY, w, W1, W2 = _problem(seed, n, H, I, wstd)
    st, bound = expert_backward_bound(X, h, GY, w, W1, W2, I)
    r = _ratios(_emulated_bf16_backward(X, h, GY, w, W1, W2, I, mistake), st, bound)[out]
    # well outside, on a share of the elements (silu' without its second
    # factor differs from it by g (1 - s) s, small where g is small)
    assert r.max() > 2 and (r > 1).mean() > 0.02, f"{mistake}: max ratio {r.max():.3g}, " \
                                                   f"share outside {(r > 1).mean():.3g}"


def test_the_exact_chain_rule_needs_no_room():
    """Pins the comparison itself: the oracle against itself is exact, and a
    single element moved by half its own magnitude is caught."""
    X, h, GY, w, W1, W2 = _problem(5, 96, 256, 128)
    st, bound = expert_backward_bound(X, h, GY, w, W1, W2, 128)
    for k in ("dX", "dW1", "dW2"):
        assert (np.abs(st[k] - st[k]) <= bound[k]).all()
    i = np.unravel_index(np.argmax(np.abs(st["dW1"])), st["dW1"].shape)
    bad = st["dW1"].copy()
    bad[i] *= 1.5
    assert np.abs(bad - st["dW1"])[i] > bound["dW1"][i]


def test_forward_h_bound_covers_an_fp32_forward():
    """h computed with fp32 GEMMs and an fp32 SwiGLU, then rounded once, stays
    within expert_forward_h_bound of the oracle's h."""
    X, h, GY, w, W1, W2 = _problem(3, 150, 512, 256, 0.05)
    g32 = np.asarray(X, np.float32) @ np.asarray(W1[:256].T, np.float32)
    u32 = np.asarray(X, np.float32) @ np.asarray(W1[256:].T, np.float32)
    h32 = _bf(g32 / (np.float32(1) + np.exp(-g32)) * u32)
    b = expert_forward_h_bound(X, W1, 256)
    assert (np.abs(h32 - h) <= b).all()
