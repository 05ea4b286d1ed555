"""Pins of the router oracle (softmax -> top-k -> renormalise) to things other
than itself: hand-worked cases, brute force over subsets, library softmax and
autograd, closed forms, finite differences."""
import itertools
import json
import os

import numpy as np
import pytest
import scipy.special
import torch

import oracle as O

GOLDEN = os.path.join(os.path.dirname(__file__), "golden", "router_cases.json")


def _cases():
    with open(GOLDEN) as f:
        return json.load(f)["cases"]


@pytest.mark.parametrize("case", _cases(), ids=lambda c: c["name"])
def test_hand_worked_cases(case):
    logits = np.log(np.asarray(case["logits_ln"], dtype=np.float64)).astype(np.float32)
    idx, w = O.router_topk(logits, case["K"])
    assert np.array_equal(idx, np.asarray(case["topk_idx"]))
    den = np.asarray(case["topk_probs_den"], dtype=np.float64).reshape(-1, 1)
    want = np.asarray(case["topk_probs_num"], dtype=np.float64) / den
    np.testing.assert_allclose(w, want, rtol=1e-6, atol=0)


def test_brute_force_subsets_small_E():
    """The chosen set is the unique K-subset whose every probability is at
    least every probability outside it (no ties in random logits)."""
    rng = np.random.default_rng(0)
    for E in (2, 3, 5, 6):
        for K in range(1, E + 1):
            logits = rng.standard_normal((20, E)).astype(np.float32)
            idx, w = O.router_topk(logits, K)
            p = scipy.special.softmax(logits.astype(np.float64), axis=1)
            for t in range(20):
                best = [S for S in itertools.combinations(range(E), K)
                        if min(p[t, list(S)]) >= max([p[t, j] for j in range(E) if j not in S],
                                                     default=-1.0)]
                assert len(best) == 1
                assert sorted(idx[t].tolist()) == list(best[0])
                # descending order inside the selection
                assert all(p[t, idx[t, k]] >= p[t, idx[t, k + 1]] for k in range(K - 1))
                np.testing.assert_allclose(w[t], p[t, idx[t]] / p[t, idx[t]].sum(), rtol=1e-6)


def test_k_equals_e_is_the_full_softmax_sorted():
    rng = np.random.default_rng(1)
    logits = rng.standard_normal((50, 16)).astype(np.float32)
    idx, w = O.router_topk(logits, 16)
    p = scipy.special.softmax(logits.astype(np.float64), axis=1)
    np.testing.assert_allclose(w, np.take_along_axis(p, idx, axis=1), rtol=1e-6)
    assert np.all(np.diff(np.take_along_axis(p, idx, axis=1), axis=1) <= 0)


def test_top1_is_argmax_with_weight_one():
    rng = np.random.default_rng(2)
    logits = rng.standard_normal((100, 32)).astype(np.float32)
    idx, w = O.router_topk(logits, 1)
    assert np.array_equal(idx[:, 0], np.argmax(logits, axis=1))
    assert np.all(w == 1.0)


def test_renormalised_topk_is_softmax_of_selected_logits_and_shift_invariant():
    rng = np.random.default_rng(3)
    logits = (rng.standard_normal((64, 128)) - 1.2 * np.log(np.arange(1, 129))).astype(np.float32)
    idx, w = O.router_topk(logits, 8)
    sel = np.take_along_axis(logits.astype(np.float64), idx, axis=1)
    np.testing.assert_allclose(w, scipy.special.softmax(sel, axis=1), rtol=1e-6)
    idx2, w2 = O.router_topk(logits + np.float32(7.0), 8)
    assert np.array_equal(idx, idx2)
    np.testing.assert_allclose(w2, w, rtol=1e-5)
    np.testing.assert_allclose(w.sum(axis=1), 1.0, rtol=1e-6)
    assert all(len(set(r)) == 8 for r in idx.tolist())


def test_backward_matches_torch_autograd_with_the_selection_fixed():
    rng = np.random.default_rng(4)
    T, E, K = 16, 32, 6
    logits = rng.standard_normal((T, E)).astype(np.float32)
    idx, w = O.router_topk(logits, K)
    g = rng.standard_normal((T, K)).astype(np.float32)
    lt = torch.tensor(logits, dtype=torch.float64, requires_grad=True)
    sel = torch.gather(torch.softmax(lt, dim=1), 1, torch.from_numpy(idx))
    wt = sel / sel.sum(dim=1, keepdim=True)
    (wt * torch.from_numpy(g).double()).sum().backward()
    got = O.router_topk_backward(g, w, idx, E)
    np.testing.assert_allclose(got, lt.grad.numpy(), rtol=1e-5, atol=1e-7)
    # no gradient outside the selection
    mask = np.ones((T, E), bool)
    np.put_along_axis(mask, idx, False, axis=1)
    assert np.all(got[mask] == 0)


def test_backward_central_finite_differences():
    rng = np.random.default_rng(5)
    T, E, K = 4, 10, 3
    logits = rng.standard_normal((T, E))
    idx, w = O.router_topk_f64(logits, K)
    g = rng.standard_normal((T, K))
    got = O.router_topk_backward(g, w, idx, E).astype(np.float64)
    h = 1e-6
    for t in range(T):
        for j in range(E):
            lp, lm = logits.copy(), logits.copy()
            lp[t, j] += h
            lm[t, j] -= h
            ip, wp = O.router_topk_f64(lp, K)
            im, wm = O.router_topk_f64(lm, K)
            assert np.array_equal(ip, idx) and np.array_equal(im, idx)  # away from a tie
            fd = ((wp[t] - wm[t]) * g[t]).sum() / (2 * h)
            assert abs(fd - got[t, j]) < 1e-6, (t, j, fd, got[t, j])
