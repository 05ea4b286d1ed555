"""Pins for the oracle's bf16 conversions (CPU only).

The round-to-nearest-even rule is checked against two things the oracle does
not use: torch's float32 -> bfloat16 cast (a library routine), and exact
rational arithmetic on the two bf16 neighbours of each value (brute force).
"""
from fractions import Fraction

import numpy as np
import pytest
import torch

from oracle import bf16_bits_to_f32, f32_to_bf16_bits, f64_to_bf16_bits


def _torch_bits(f32: np.ndarray) -> np.ndarray:
    t = torch.from_numpy(f32.copy()).to(torch.bfloat16)
    return t.view(torch.int16).numpy().view(np.uint16)


def test_widen_all_patterns_roundtrip():
    bits = np.arange(65536, dtype=np.uint32).astype(np.uint16)
    f = bf16_bits_to_f32(bits)
    back = f32_to_bf16_bits(f)
    nan = np.isnan(f)
    assert np.array_equal(back[~nan], bits[~nan])
    assert np.isnan(bf16_bits_to_f32(back[nan])).all()
    # widening is the top-half embedding
    assert np.array_equal(f.view(np.uint32) >> 16, bits.astype(np.uint32))


def test_f32_rounding_matches_torch_cast():
    rng = np.random.default_rng(0)
    raw = rng.integers(0, 2**32, size=1_000_000, dtype=np.uint64).astype(np.uint32)
    f = raw.view(np.float32)
    special = np.array([0.0, -0.0, np.inf, -np.inf, 1.0, 1.0 + 2**-8, 1.0 + 3 * 2**-8,
                        3.3895313892515355e38, 3.4028234663852886e38, 1e-45, -1e-45,
                        2**-126, 2**-127 + 2**-134, 2**-133 * 1.5], dtype=np.float32)
    f = np.concatenate([f, special])
    ok = ~np.isnan(f)
    assert np.array_equal(f32_to_bf16_bits(f[ok]), _torch_bits(f[ok]))
    assert np.isnan(bf16_bits_to_f32(f32_to_bf16_bits(f[~ok]))).all()


def test_ties_go_to_even():
    # 1 + 2^-8 is halfway between 1 and 1 + 2^-7: even significand is 1.0
    assert f64_to_bf16_bits(np.array([1.0 + 2**-8]))[0] == 0x3F80
    # 1 + 3*2^-8 is halfway between 1+2^-7 (odd) and 1+2^-6 (even)
    assert f64_to_bf16_bits(np.array([1.0 + 3 * 2**-8]))[0] == 0x3F82
    # just above the tie rounds up
    assert f64_to_bf16_bits(np.array([1.0 + 2**-8 + 2**-40]))[0] == 0x3F81


def _all_bf16_values():
    bits = np.arange(0, 0x7F81, dtype=np.uint32).astype(np.uint16)  # +0 .. +inf
    return bf16_bits_to_f32(bits).astype(np.float64)


def test_f64_rounding_brute_force_exact():
    """Nearest bf16 by exact rational comparison with its two neighbours."""
    vals = _all_bf16_values()
    finite = vals[np.isfinite(vals)]
    rng = np.random.default_rng(1)
    xs = list(np.ldexp(rng.random(3000) + 0.5, rng.integers(-140, 130, size=3000)))
    # exact midpoints (ties) and near-midpoints, including subnormal and overflow edges
    for i in rng.integers(0, finite.size - 1, size=600):
        lo, hi = finite[i], finite[i + 1]
        mid = (lo + hi) / 2
        xs += [mid, np.nextafter(mid, np.inf), np.nextafter(mid, -np.inf)]
    xs += [finite[-1] + (finite[-1] - finite[-2]) / 2, 2**-134, 2**-135, 3 * 2**-135]
    xs = np.array(xs, dtype=np.float64)
    got = bf16_bits_to_f32(f64_to_bf16_bits(xs)).astype(np.float64)
    for x, g in zip(xs, got):
        j = np.searchsorted(finite, x)
        if j >= finite.size:  # beyond the largest finite bf16
            lo, hi = finite[-1], np.inf
        else:
            lo = finite[j - 1] if finite[j] > x else finite[j]
            hi = finite[j]
        if lo == x:
            assert g == x
            continue
        if np.isinf(hi):
            # the overflow threshold is the midpoint to the next (virtual) binade value 2^128
            thr = Fraction(lo) + (Fraction(2**128) - Fraction(lo)) / 2
            exp = np.inf if Fraction(x) >= thr else lo
            assert g == exp, (x, g, exp)
            continue
        dlo, dhi = Fraction(x) - Fraction(lo), Fraction(hi) - Fraction(x)
        if dlo < dhi:
            exp = lo
        elif dhi < dlo:
            exp = hi
        else:
            lo_bits = int(f64_to_bf16_bits(np.array([lo]))[0])
            exp = lo if lo_bits % 2 == 0 else hi
        assert g == exp, (x, g, exp)


def test_negative_values_mirror():
    rng = np.random.default_rng(2)
    x = rng.standard_normal(10000) * 10.0 ** rng.integers(-30, 30, size=10000)
    a = f64_to_bf16_bits(x)
    b = f64_to_bf16_bits(-x)
    assert np.array_equal(a ^ np.uint16(0x8000), b)
