"""Element-wise error bounds for a bf16 implementation of the expert backward
(a9) around the oracle's exact fp64 chain rule.

The experts are bf16 grouped GEMMs ("Add the deepep expert-parallel
implementation (huggingface/transformers #49638)", Benchmarks), so an
implementation of their backward ("What this adds", Training) feeds its GEMMs
bf16 operands and accumulates in fp32.  It may round to bf16 any of the
chain rule's intermediates -- G_o = w * grad_y, the gate and up values g and
u, G_h = G_o W2, G_g and G_u -- and must round the bf16 output grad_x_disp.
The bound allows every one of those roundings, so it does not depend on
which ones a given implementation makes.

Terms (all computed in fp64 from the exact intermediates of
oracle.expert_backward_steps):

 1. Rounding effects, exact and signed.  For each intermediate p, the change
    of the outputs when p alone is rounded to the nearest bf16 value and
    everything else stays exact; the bound takes the sum of their absolute
    values (first order: the effect of several roundings is the sum of their
    effects).  A rounding of p made from an upstream value that is already
    off absorbs the upstream error unless the two round to different
    neighbours, so this also covers an implementation that rounds several
    points in a row.
 2. Flips.  Where p lies within its incoming error of a rounding midpoint, an
    implementation may round to the other neighbour; such elements get two
    bf16 ulps of p, carried to the outputs through absolute values.
 3. fp32 accumulation.  Each dot product of n terms is held to
    LAMBDA * sqrt(n) * U_F * sum_k |a_k b_k| (the probabilistic bound of
    Higham and Mary, "A new approach to probabilistic rounding error
    analysis", SIAM J. Sci. Comput. 41(5), 2019, with the unit roundoff
    doubled, U_F = 2^-23, for additions that do not round to nearest; with
    LAMBDA = 6 a single dot product exceeds it with probability below
    2 exp(-18)), carried on through absolute values.
 4. The fp32 evaluation of sigmoid-based silu and silu': FN_ABS (1 + |g|)
    absolute, and four fp32 roundings of each product.
The sum is multiplied by SAFETY = 2 for the second-order terms.  A plausible
mistake (a dropped or wrong term, a wrong index, a swapped or transposed
operand, a sign) moves the result by a sizeable fraction of its magnitude
and leaves the bound; tests/test_backward_bound.py checks both directions on
the CPU.
"""
from __future__ import annotations

import numpy as np

import oracle as O

U_B = 2.0 ** -8       # one bf16 ulp, relative
U_F = 2.0 ** -23      # fp32 rounding, doubled
LAMBDA = 6.0
MAX_DSILU = 1.1       # max |silu'(z)| = 1.0998 near z = 2.40
MAX_D2SILU = 0.5      # max |silu''(z)| = 0.5 at z = 0
FN_ABS = 2.0 ** -16
SAFETY = 2.0


def acc(n: int) -> float:
    """Relative bound of an fp32 dot product of n terms (term 3)."""
    return LAMBDA * np.sqrt(max(n, 1)) * U_F


def bf16_ulp(v):
    """Spacing of bf16 values at |v| (the subnormal spacing at 0)."""
    v = np.abs(np.asarray(v, dtype=np.float64))
    e = np.frexp(v)[1]
    return np.ldexp(1.0, np.maximum(e - 8, -133))


def rne_err(v):
    """Signed error of rounding v to the nearest bf16 value."""
    return O.bf16_round_f64(v) - v


def flips(v, e_in):
    """Two bf16 ulps of v where v is within e_in of a rounding midpoint (a
    value within e_in of v may round to the other neighbour), else 0."""
    ulp = bf16_ulp(v)
    to_mid = ulp / 2 - np.abs(rne_err(v))
    return np.where(to_mid <= e_in, 2 * ulp, 0.0)


def _sig(z):
    return 1.0 / (1.0 + np.exp(-np.clip(z, -700.0, 700.0)))


def expert_forward_h_bound(X, W1e, I):
    """How far an implementation's bf16 h = bf16(silu(g) u) (fp32 GEMMs and
    SwiGLU, one rounding) can be from the oracle's bf16 h, element-wise: zero
    except where the exact value is within the fp32 error of a rounding
    midpoint, where the two may round to neighbouring values."""
    aX = np.abs(X)
    g, u = O.backward_gate_up(X, W1e, I)
    H = X.shape[1]
    eg = acc(H) * (aX @ np.abs(W1e[:I]).T)
    eu = acc(H) * (aX @ np.abs(W1e[I:]).T)
    s = _sig(g)
    silu = g * s
    pre = silu * u
    e_pre = np.abs(silu) * eu + np.abs(u) * MAX_DSILU * eg + np.abs(u) * FN_ABS * (1 + np.abs(g)) \
        + 4 * U_F * np.abs(pre)
    return flips(pre, e_pre)


def expert_backward_bound(X, h, GY, w, W1e, W2e, I, h_flips=None, dW_bf16=False):
    """The oracle's exact chain rule for one expert's rows, and element-wise
    bounds on how far a bf16 implementation can be from it.

    X [n, H], h [n, I], GY [n, H] (bf16 values, as fp64), w [n], W1e [2I, H],
    W2e [H, I].  ``h_flips`` [n, I], if given, bounds how far the h the
    implementation uses can be from ``h`` (its forward rounded its own h;
    see expert_forward_h_bound).  ``dW_bf16``: the weight gradients are
    rounded to bf16 at the end.
    Returns (steps, bound): steps = oracle.expert_backward_steps(...), bound a
    dict of "dX" [n, H], "dW1" [2I, H], "dW2" [H, I].
    """
    st = O.expert_backward_steps(X, h, GY, w, W1e, W2e, I)
    n, H = X.shape
    G_o, G_h, g, u = st["G_o"], st["G_h"], st["g"], st["u"]
    D, S, G_gu = st["dsilu"], st["silu"], st["G_gu"]
    aX, aW1, aW2, ah = np.abs(X), np.abs(W1e), np.abs(W2e), np.abs(h)
    aGo, aGh, au = np.abs(G_o), np.abs(G_h), np.abs(u)

    bX = np.zeros_like(st["dX"])
    bW1 = np.zeros_like(st["dW1"])
    bW2 = np.zeros_like(st["dW2"])

    def carry(dGgu):
        """Add the outputs' change for a signed change of [G_g | G_u]."""
        nonlocal bX, bW1
        bX = bX + np.abs(dGgu @ W1e)
        bW1 = bW1 + np.abs(dGgu.T @ X)

    # 1. rounding effects
    r_o = rne_err(G_o)
    bW2 = bW2 + np.abs(r_o.T @ h)
    dGh_o = r_o @ W2e
    up = [np.concatenate([dGh_o * u * D, dGh_o * S], axis=1)]
    g2 = O.bf16_round_f64(g)
    s2 = _sig(g2)
    up.append(np.concatenate([G_h * u * (s2 * (1 + g2 * (1 - s2)) - D), G_h * (g2 * s2 - S)], axis=1))
    up.append(np.concatenate([G_h * rne_err(u) * D, np.zeros_like(u)], axis=1))
    r_h = rne_err(G_h)
    up.append(np.concatenate([r_h * u * D, r_h * S], axis=1))
    for d in up:
        carry(d)
    r_gu = rne_err(G_gu)
    carry(r_gu)

    # 3. fp32 accumulation of G_h, g, u; 2. flips of G_o, g, u, G_h
    f_o = flips(G_o, 2 * U_F * aGo)
    e_h = acc(H) * (aGo @ aW2)
    e_g = acc(H) * (aX @ aW1[:I].T)
    e_u = acc(H) * (aX @ aW1[I:].T)
    fo_h = f_o @ aW2
    f_h = flips(G_h, e_h + np.abs(dGh_o) + fo_h)
    Bh = e_h + fo_h + f_h
    Bg = e_g + flips(g, e_g)
    Bu = e_u + flips(u, e_u)
    fn = FN_ABS * (1.0 + np.abs(g))
    G_g, G_u = G_gu[:, :I], G_gu[:, I:]
    B_gu = np.concatenate([
        Bh * au * np.abs(D) + aGh * Bu * np.abs(D) + aGh * au * (MAX_D2SILU * Bg + fn) + 4 * U_F * np.abs(G_g),
        Bh * np.abs(S) + aGh * (MAX_DSILU * Bg + fn) + 4 * U_F * np.abs(G_u)], axis=1)
    B_gu = B_gu + flips(G_gu, B_gu + sum(np.abs(d) for d in up))
    aGgu = np.abs(G_gu)
    bX = bX + B_gu @ aW1 + acc(2 * I) * (aGgu @ aW1) + U_B * np.abs(st["dX"])
    bW1 = bW1 + B_gu.T @ aX + acc(n) * (aGgu.T @ aX)
    bW2 = bW2 + f_o.T @ ah + acc(n) * (aGo.T @ ah)
    if h_flips is not None:
        bW2 = bW2 + aGo.T @ h_flips
    if dW_bf16:
        bW1 = bW1 + U_B * np.abs(st["dW1"])
        bW2 = bW2 + U_B * np.abs(st["dW2"])
    return st, {"dX": SAFETY * bX, "dW1": SAFETY * bW1, "dW2": SAFETY * bW2}


def check_within(got, ref, bound, what):
    """Every element of ``got`` within ``bound`` of ``ref``; the message names
    the worst element and its ratio to the bound.  Returns the worst ratio."""
    got = np.asarray(got, dtype=np.float64)
    ref = np.asarray(ref, dtype=np.float64)
    assert got.shape == ref.shape == bound.shape, what
    assert np.isfinite(got).all(), f"{what}: non-finite values"
    err = np.abs(got - ref)
    if not err.size:
        return 0.0
    ratio = err / np.maximum(bound, 1e-300)
    worst = np.unravel_index(int(np.argmax(ratio)), ratio.shape)
    assert (err <= bound).all(), (
        f"{what}: {int((err > bound).sum())} of {err.size} elements outside the bound; worst at "
        f"{worst}: got {got[worst]:.6g}, exact {ref[worst]:.6g}, err {err[worst]:.3g} > bound "
        f"{bound[worst]:.3g}")
    return float(ratio.max())
