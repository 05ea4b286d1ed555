"""Helpers shared by the GPU tests: bit views and the parity tolerances."""
import numpy as np
import torch

import oracle as O

# Tolerances for the bf16 expert GEMM outputs (max |err| and relative L2),
# compared with the fp64 oracle on the same inputs.
GEMM_MAX_ABS = 2e-2
GEMM_REL_L2 = 5e-3


def bits(t: torch.Tensor) -> np.ndarray:
    """bf16 tensor -> numpy uint16 bit patterns (on the CPU)."""
    return t.detach().cpu().contiguous().view(torch.int16).numpy().view(np.uint16)


def from_bits(b: np.ndarray, device="cpu") -> torch.Tensor:
    return torch.from_numpy(np.ascontiguousarray(b).view(np.int16)).view(torch.bfloat16).to(device)


def assert_gemm_close(gpu_bits: np.ndarray, ref_bits: np.ndarray, what: str,
                      intermediate: bool = False):
    """The expert outputs (y, o and the layer output) must satisfy
    max |err| <= 2e-2 and rel L2 <= 5e-3.  For the intermediates (h and the
    saved gate/up pre-activations), whose values exceed 4 where one bf16 ulp
    is already 2^-5 > 2e-2, the max-error bound scales with the magnitude:
    |err| <= 2e-2 * max(1, |ref|); the rel L2 bound is the same."""
    g = O.bf16_bits_to_f64(gpu_bits)
    r = O.bf16_bits_to_f64(ref_bits)
    assert np.isfinite(g).all(), f"{what}: non-finite GPU values"
    d = np.abs(g - r)
    if intermediate:
        d = d / np.maximum(1.0, np.abs(r))
    err = d.max() if g.size else 0.0
    den = np.linalg.norm(r)
    rel = np.linalg.norm(g - r) / den if den > 0 else np.linalg.norm(g - r)
    assert err <= GEMM_MAX_ABS and rel <= GEMM_REL_L2, f"{what}: max|err|={err:.3g} rel_l2={rel:.3g}"
    return err, rel


def random_routing(T, E, K, seed, drop=0.0, dup=0.0):
    """Top-k choices with optional dropped (-1) and duplicated slots."""
    rng = np.random.default_rng(seed)
    idx = np.stack([rng.permutation(E)[:K] for _ in range(T)]) if T else np.zeros((0, K), np.int64)
    if drop:
        idx[rng.random((T, K)) < drop] = -1
    if dup and K > 1:
        d = rng.random(T) < dup
        idx[d, K - 1] = idx[d, 0]
    p = rng.random((T, K)).astype(np.float32)
    return torch.from_numpy(idx.astype(np.int64)), torch.from_numpy(p)
