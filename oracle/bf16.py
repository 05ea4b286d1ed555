"""bfloat16 as bit patterns, for the oracle.  Test infrastructure only.

bf16 is the top half of an IEEE binary32: 1 sign bit, 8 exponent bits, 7
stored significand bits.  Tensors travel through the oracle as ``uint16`` bit
patterns, exactly as they sit in device memory, and are widened exactly.

Rounding to bf16 is round-to-nearest, ties-to-even, done *once* from the exact
fp64 (or fp32) value: no intermediate rounding through fp32.
"""
from __future__ import annotations

import numpy as np

_MIN_NORMAL_EXP = -125   # frexp exponent of 2**-126, the smallest normal bf16
_SIG_BITS = 8            # significant bits of a normal bf16 (1 implicit + 7)
_SUBNORMAL_QUANTUM_EXP = -133  # 2**-133 = spacing of bf16 subnormals


def bf16_bits_to_f32(bits: np.ndarray) -> np.ndarray:
    """Exact widening of bf16 bit patterns to float32."""
    b = np.asarray(bits, dtype=np.uint16)
    return (b.astype(np.uint32) << np.uint32(16)).view(np.float32)


def bf16_bits_to_f64(bits: np.ndarray) -> np.ndarray:
    """Exact widening of bf16 bit patterns to float64."""
    return bf16_bits_to_f32(bits).astype(np.float64)


def bf16_round_f64(v: np.ndarray) -> np.ndarray:
    """Round fp64 values to the nearest bf16 value (ties to even); result in fp64.

    For |v| = m * 2**e with 0.5 <= m < 1, a normal bf16 keeps 8 significant
    bits, so its spacing is 2**(e - 8); below the smallest normal the spacing
    is fixed at 2**-133.  Scaling by a power of two is exact, and ``np.rint``
    rounds half to even.  Results at or beyond 2**128 overflow to infinity.
    """
    v = np.asarray(v, dtype=np.float64)
    out = np.array(v, dtype=np.float64, copy=True)
    fin = np.isfinite(v) & (v != 0.0)
    a = np.abs(v[fin])
    _, e = np.frexp(a)
    qe = np.maximum(e - _SIG_BITS, _SUBNORMAL_QUANTUM_EXP)
    r = np.rint(np.ldexp(a, -qe))
    mag = np.ldexp(r, qe)
    mag = np.where(mag >= 2.0 ** 128, np.inf, mag)
    out[fin] = np.copysign(mag, v[fin])
    return out


def f64_to_bf16_bits(v: np.ndarray) -> np.ndarray:
    """fp64 -> bf16 bit patterns with a single round-to-nearest-even.

    NaN maps to the quiet NaN 0x7FC0 (sign kept); signed zeros and infinities
    are kept.
    """
    v = np.asarray(v, dtype=np.float64)
    with np.errstate(invalid="ignore", over="ignore"):
        r = bf16_round_f64(v)
    # every finite r is a bf16 value, hence exactly a float32 whose low 16 bits are 0
    with np.errstate(invalid="ignore", over="ignore"):
        bits = (r.astype(np.float32).view(np.uint32) >> np.uint32(16)).astype(np.uint16)
    nan = np.isnan(v)
    if nan.any():
        sign = (np.signbit(v[nan]).astype(np.uint16) << np.uint16(15))
        bits[nan] = np.uint16(0x7FC0) | sign
    return bits


def f32_to_bf16_bits(v: np.ndarray) -> np.ndarray:
    """float32 -> bf16 bit patterns, round-to-nearest-even (exact via fp64)."""
    with np.errstate(invalid="ignore"):   # signalling-NaN payloads warn on widening
        wide = np.asarray(v, dtype=np.float32).astype(np.float64)
    return f64_to_bf16_bits(wide)
