"""The router step in front of the path, on the CPU.  Test infrastructure only.

The pages start the path at the router's output (top-k expert indices and
fp32 weights): "feat: add hybridep (NVIDIA-NeMo/Automodel #1333)", Changelog,
turns top-k indices into multihot routing data.  The router itself is the
plain reading of the synthetic workload's recipe: fp32 logits [T, E], a softmax
over the experts, the K most probable experts, and their probabilities
renormalised to sum to one.

Readings taken (each pinned by tests/test_oracle_router.py):
  * the K experts come out in descending probability; equal probabilities
    are ordered by ascending expert index;
  * softmax, selection and renormalisation are computed in fp64 from the fp32
    logits and the weights returned as fp32;
  * the gradient with respect to the logits follows from the chain rule
    through the softmax and the renormalisation; the selection itself is
    piecewise constant and passes no gradient (an expert outside the top-k
    gets zero).
"""
from __future__ import annotations

import numpy as np


def router_topk(logits, K: int):
    """softmax over E -> top-K -> renormalise.

    logits: [T, E] (float32 or float64).  Returns (topk_idx int64 [T, K],
    topk_probs float32 [T, K]); slot 0 holds the most probable expert.
    """
    lg = np.asarray(logits, dtype=np.float64)
    T, E = lg.shape
    if not 1 <= K <= E:
        raise ValueError("need 1 <= K <= E")
    # softmax over the experts (shifted by the row maximum for range)
    z = np.exp(lg - lg.max(axis=1, keepdims=True))
    p = z / z.sum(axis=1, keepdims=True)
    # descending probability; a stable sort of -p keeps equal ones in index order
    order = np.argsort(-p, axis=1, kind="stable")
    idx = order[:, :K]
    sel = np.take_along_axis(p, idx, axis=1)
    w = sel / sel.sum(axis=1, keepdims=True)
    return idx.astype(np.int64), w.astype(np.float32)


def router_topk_f64(logits, K: int):
    """As router_topk, with the weights left in fp64 (for tolerance checks)."""
    lg = np.asarray(logits, dtype=np.float64)
    z = np.exp(lg - lg.max(axis=1, keepdims=True))
    p = z / z.sum(axis=1, keepdims=True)
    idx = np.argsort(-p, axis=1, kind="stable")[:, :K]
    sel = np.take_along_axis(p, idx, axis=1)
    return idx.astype(np.int64), sel / sel.sum(axis=1, keepdims=True)


def router_topk_backward(grad_topk_probs, topk_probs, topk_idx, E: int):
    """dL/dlogits [T, E] (fp64 -> fp32) given dL/dw [T, K].

    With s_j = p_j / sum_{i in top-k} p_i over the selected experts, the full
    softmax's normaliser cancels, so w = softmax of the selected logits alone
    and dw_k/dl_j = w_k (delta_kj - w_j).  Hence
    dL/dl_j = w_j (g_j - sum_k w_k g_k) for j in the top-k, and 0 elsewhere.
    """
    g = np.asarray(grad_topk_probs, dtype=np.float64)
    w = np.asarray(topk_probs, dtype=np.float64)
    idx = np.asarray(topk_idx, dtype=np.int64)
    T, K = idx.shape
    out = np.zeros((T, E), dtype=np.float64)
    dot = (w * g).sum(axis=1, keepdims=True)
    np.put_along_axis(out, idx, w * (g - dot), axis=1)
    return out.astype(np.float32)
