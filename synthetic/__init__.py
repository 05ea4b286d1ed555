"""Seeded synthetic workloads for the MoE dispatch / experts / combine layer.

This module only *draws inputs*: token activations, router top-k choices and
expert weights.  It holds none of the layer's own arithmetic (no multihot, no
counts, no layout, no expert math, no combine), so both the CUDA path and the
CPU oracle can take their inputs from here without sharing any of the method.

The router that produces top-k choices is the step *before* the path
(softmax over router logits, top-k, renormalise), as in the MoE layers that
"feat: add hybridep (NVIDIA-NeMo/Automodel #1333)" wires up: the path starts at
the top-k expert indices and their fp32 probabilities.  make_routing applies
that recipe with torch's CPU softmax and top-k to draw the inputs of the path
itself.  The library's own router kernel is checked against the separate
router oracle on logits from make_logits, never against make_routing.

Shapes follow the layer shapes of "Add the deepep expert-parallel
implementation (huggingface/transformers #49638)", Benchmarks: "30b" is the
Qwen3-30B-A3B expert layer (E=128, H=2048, I=768, top-8) and "h4096" is
E=128, H=4096, I=1536, top-8.
"""
from __future__ import annotations

import dataclasses
from typing import Optional

import torch


@dataclasses.dataclass(frozen=True)
class LayerConfig:
    name: str
    T: int            # tokens
    H: int            # hidden size
    E: int            # experts
    K: int            # top-k
    I: int            # SwiGLU intermediate size
    P: int            # pad_multiple
    seed: int
    zipf_s: float = 0.0      # log-Zipf router bias exponent (0 = none)
    drop: float = 0.0        # probability that a (token, slot) index is set to -1
    sync_free: bool = False  # worst-case capacity, no host sync
    backward: bool = False   # forward plus backward


# The workloads.  The tiny layer's seed 0 is part of its description; the
# other seeds are fixed, arbitrary choices.
CONFIGS = {
    "tiny": LayerConfig("tiny", T=64, H=256, E=8, K=2, I=128, P=16, seed=0),
    "qwen3_30b_a3b": LayerConfig("qwen3_30b_a3b", T=4096, H=2048, E=128, K=8, I=768, P=128, seed=1),
    "qwen3_30b_a3b_16k": LayerConfig("qwen3_30b_a3b_16k", T=16384, H=2048, E=128, K=8, I=768, P=128, seed=1),
    "h4096": LayerConfig("h4096", T=16384, H=4096, E=128, K=8, I=1536, P=128, seed=2, backward=True),
    "skewed": LayerConfig("skewed", T=16384, H=2048, E=128, K=8, I=768, P=128, seed=3, zipf_s=1.2, drop=0.05),
    # the h4096 expert shape (about 1024 rows per expert) on 16 experts: a few
    # GB on the device, small enough for detailed profiler captures
    "h4096_small": LayerConfig("h4096_small", T=2048, H=4096, E=16, K=8, I=1536, P=128, seed=2, backward=True),
    "decode_1": LayerConfig("decode_1", T=1, H=2048, E=128, K=8, I=768, P=1, seed=5, sync_free=True),
    "decode_256": LayerConfig("decode_256", T=256, H=2048, E=128, K=8, I=768, P=1, seed=260, sync_free=True),
    "decode_1024": LayerConfig("decode_1024", T=1024, H=2048, E=128, K=8, I=768, P=1, seed=1028, sync_free=True),
}


def _gen(seed: int, device="cpu") -> torch.Generator:
    g = torch.Generator(device=device)
    g.manual_seed(seed)
    return g


def make_tokens(T: int, H: int, seed: int, device="cpu") -> torch.Tensor:
    """x ~ N(0, 1), stored as bf16, shape [T, H]."""
    g = _gen(seed * 1000 + 1, device)
    return torch.randn(T, H, generator=g, device=device, dtype=torch.float32).to(torch.bfloat16)


def _draw_logits(g, T: int, E: int, zipf_s: float):
    logits = torch.randn(T, E, generator=g, dtype=torch.float32)
    if zipf_s:
        bias = -zipf_s * torch.log(torch.arange(1, E + 1, dtype=torch.float32))
        logits = logits + bias
    return logits


def make_logits(T: int, E: int, seed: int, zipf_s: float = 0.0) -> torch.Tensor:
    """Router logits fp32 [T, E] ~ N(0,1) [+ log-Zipf bias], on the CPU: the
    same draw make_routing starts from, as input for the router step."""
    return _draw_logits(_gen(seed * 1000 + 2), T, E, zipf_s).contiguous()


def make_routing(T: int, E: int, K: int, seed: int, zipf_s: float = 0.0, drop: float = 0.0):
    """Router choices: fp32 logits ~ N(0,1) [+ log-Zipf bias], softmax, top-k, renormalise.

    With ``zipf_s > 0`` expert e's logit gets ``-zipf_s * ln(e + 1)``, which
    multiplies its softmax odds by (e + 1) ** -zipf_s.  With ``drop > 0`` each
    (token, slot) index is independently replaced by -1 after renormalising (the
    dropped weight is not redistributed).  Returns (topk_idx int64 [T, K],
    topk_probs fp32 [T, K]), on the CPU.
    """
    g = _gen(seed * 1000 + 2)
    logits = _draw_logits(g, T, E, zipf_s)
    p = torch.softmax(logits, dim=-1)
    vals, idx = torch.topk(p, K, dim=-1)
    vals = vals / vals.sum(dim=-1, keepdim=True)
    idx = idx.to(torch.int64)
    if drop:
        u = torch.rand(T, K, generator=g)
        idx = torch.where(u < drop, torch.full_like(idx, -1), idx)
    return idx.contiguous(), vals.to(torch.float32).contiguous()


def make_weights(E: int, H: int, I: int, seed: int, device="cpu", std: float = 0.02):
    """Expert weights ~ N(0, std) in bf16.

    W1 [E, 2I, H]: rows 0..I-1 of each expert are the gate projection, rows
    I..2I-1 the up projection.  W2 [E, H, I]: the down projection.  Both are
    "out x in" with the contraction dimension contiguous.
    """
    g = _gen(seed * 1000 + 3, device)
    W1 = torch.empty(E, 2 * I, H, dtype=torch.bfloat16, device=device)
    W2 = torch.empty(E, H, I, dtype=torch.bfloat16, device=device)
    for e in range(E):  # per expert, to bound the fp32 temporary
        W1[e] = (torch.randn(2 * I, H, generator=g, device=device) * std).to(torch.bfloat16)
        W2[e] = (torch.randn(H, I, generator=g, device=device) * std).to(torch.bfloat16)
    return W1, W2


def make_layer_inputs(cfg: LayerConfig, device="cpu", with_weights: bool = True, layer: int = 0):
    """All inputs of one layer.  ``layer`` selects one of several distinct
    weight/token sets of the same shape (used to cycle layers so the working
    set does not sit in L2)."""
    s = cfg.seed + 7919 * layer
    x = make_tokens(cfg.T, cfg.H, s, device=device)
    idx, probs = make_routing(cfg.T, cfg.E, cfg.K, s, cfg.zipf_s, cfg.drop)
    out = {"x": x, "topk_idx": idx.to(device), "topk_probs": probs.to(device)}
    if with_weights:
        out["W1"], out["W2"] = make_weights(cfg.E, cfg.H, cfg.I, s, device=device)
    return out


def make_grad_out(T: int, H: int, seed: int, device="cpu") -> torch.Tensor:
    """Upstream gradient of the layer output, ~ N(0, 1) in bf16."""
    g = _gen(seed * 1000 + 4, device)
    return torch.randn(T, H, generator=g, device=device, dtype=torch.float32).to(torch.bfloat16)


__all__ = [
    "LayerConfig", "CONFIGS", "make_tokens", "make_logits", "make_routing", "make_weights",
    "make_layer_inputs", "make_grad_out",
]
