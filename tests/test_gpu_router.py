"""GPU parity of the router (softmax -> top-k -> renormalise), alone and fused
with the multihot step, and of its backward, against the fp64 router oracle.

Tolerances.  The expert indices must match exactly: the kernel compares the
fp32 logits, the oracle the fp64 softmax of the same fp32 values, and the
softmax is strictly increasing, so both order the experts identically (equal
logits by index in both).  A weight is exp(l_k - l_0) / sum_j exp(l_j - l_0)
in fp32: the subtraction, the exponential (2 ulp), K - 1 additions and one
division give a relative error below (K + 24) * 2^-24, the bound used here.
The backward adds one dot product of K terms and a subtraction; it is held to
(2K + 32) * 2^-24 relative to max |w_j| * (|g_j| + sum_k |w_k g_k|).
"""
import numpy as np
import pytest
import torch

import oracle as O
import synthetic

pytestmark = pytest.mark.gpu
DEV = "cuda"


@pytest.fixture(scope="module")
def moe():
    assert torch.cuda.is_available(), "GPU tests need a GPU"
    import combine_topk_multihot_gb300 as m
    return m


def _check_forward(idx, w, logits, K):
    ref_idx, ref_w = O.router_topk_f64(logits.numpy(), K)
    assert np.array_equal(idx.cpu().numpy(), ref_idx)
    got = w.cpu().numpy().astype(np.float64)
    tol = (K + 24) * 2.0 ** -24
    rel = np.abs(got - ref_w) / ref_w
    assert rel.max(initial=0.0) <= tol, f"max rel err {rel.max():.3g} > {tol:.3g}"


CASES = [  # T, E, K, zipf
    (64, 8, 2, 0.0),        # the tiny layer
    (1, 128, 8, 0.0),       # one token
    (333, 128, 8, 1.2),     # log-Zipf bias: skewed experts
    (100, 1024, 127, 0.0),  # largest E and K
    (50, 12, 12, 0.0),      # K = E
    (77, 36, 1, 0.0),       # top-1, E not a multiple of 32
    (0, 8, 2, 0.0),         # no tokens
]


@pytest.mark.parametrize("T,E,K,zipf", CASES)
def test_router_matches_oracle(moe, T, E, K, zipf):
    logits = synthetic.make_logits(T, E, seed=T + E, zipf_s=zipf)
    idx, w = moe.moe_router_topk(logits.to(DEV), K)
    torch.cuda.synchronize()
    _check_forward(idx, w, logits, K)


def test_router_ties_go_to_the_lower_index(moe):
    """Integer-valued logits make many exact ties."""
    g = torch.Generator().manual_seed(9)
    logits = torch.randint(0, 4, (500, 64), generator=g).to(torch.float32)
    idx, w = moe.moe_router_topk(logits.to(DEV), 8)
    torch.cuda.synchronize()
    _check_forward(idx, w, logits, 8)


@pytest.mark.parametrize("T,E,K,zipf", [(64, 8, 2, 0.0), (333, 128, 8, 1.2), (100, 1024, 127, 0.0)])
def test_router_fused_multihot_equals_the_two_steps(moe, T, E, K, zipf):
    """The fused kernel's multihot outputs are bit-identical to moe_route_to_multihot
    on the router's own top-k, and to the oracle's multihot of it."""
    logits = synthetic.make_logits(T, E, seed=3 * T + E, zipf_s=zipf).to(DEV)
    idx, w, rmap, probs, win = moe.moe_router_topk(logits, K, multihot=True)
    idx2, w2 = moe.moe_router_topk(logits, K)
    status = torch.zeros(1, dtype=torch.int32, device=DEV)
    rmap2, probs2, win2 = moe.moe_route_to_multihot(idx2, w2, E, status)
    torch.cuda.synchronize()
    assert torch.equal(idx, idx2) and torch.equal(w, w2)
    assert torch.equal(rmap, rmap2) and torch.equal(probs, probs2) and torch.equal(win, win2)
    rm, pr, wn = O.route_to_multihot(idx.cpu().numpy(), w.cpu().numpy(), E)
    assert np.array_equal(rmap.cpu().numpy(), rm)
    assert np.array_equal(probs.cpu().numpy(), pr)
    assert np.array_equal(win.cpu().numpy(), wn)
    assert int(status.item()) == 0


@pytest.mark.parametrize("T,E,K", [(64, 8, 2), (333, 128, 8), (100, 1024, 127), (20, 12, 12)])
def test_router_backward_matches_oracle(moe, T, E, K):
    logits = synthetic.make_logits(T, E, seed=5 * T + E)
    idx, w = moe.moe_router_topk(logits.to(DEV), K)
    gen = torch.Generator().manual_seed(T)
    g = torch.randn(T, K, generator=gen)
    grad = moe.moe_router_topk_backward(g.to(DEV), w, idx, E)
    torch.cuda.synchronize()
    wn = w.cpu().numpy().astype(np.float64)
    gn = g.numpy().astype(np.float64)
    ref = O.router_topk_backward(gn, wn, idx.cpu().numpy(), E).astype(np.float64)
    # exact bound from the arithmetic, per token
    scale = (np.abs(wn).max(axis=1, keepdims=True) *
             (np.abs(gn).max(axis=1, keepdims=True) + np.abs(wn * gn).sum(axis=1, keepdims=True)))
    err = np.abs(grad.cpu().numpy().astype(np.float64) - ref)
    assert np.all(err <= (2 * K + 32) * 2.0 ** -24 * scale + 1e-30)
    # exactly zero away from the chosen experts
    mask = np.ones((T, E), bool)
    np.put_along_axis(mask, idx.cpu().numpy(), False, axis=1)
    assert np.all(grad.cpu().numpy()[mask] == 0)


def test_router_full_size_qwen_layer(moe):
    """T 4096, E 128, top-8 (the Qwen3-30B-A3B layer's router), every token."""
    cfg = synthetic.CONFIGS["qwen3_30b_a3b"]
    logits = synthetic.make_logits(cfg.T, cfg.E, cfg.seed)
    idx, w = moe.moe_router_topk(logits.to(DEV), cfg.K)
    torch.cuda.synchronize()
    _check_forward(idx, w, logits, cfg.K)
