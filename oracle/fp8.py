"""FP8 (e4m3) dispatch and the FP8 gate/up GEMM, on the CPU.  Test infrastructure only.

"Add the deepep expert-parallel implementation (huggingface/transformers
#49638)", What this adds, scope note: FP8 dispatch -- half the dispatch bytes
for FP8 recipes -- is named as the follow-up.  The page fixes no format, so
the plainest reading is taken (each pinned by tests/test_oracle_fp8.py):

  * values are float8 e4m3 (1 sign, 4 exponent bits with bias 7, 3 mantissa
    bits, no infinities, largest finite 448, subnormals down to 2^-9);
    conversion rounds to nearest, ties to even, and saturates at +-448;
  * one fp32 scale per row (a dispatched token row; an output channel of the
    gate/up weight): scale = amax(|row|) / 448 computed in fp32, or 1 for an
    all-zero row; the code is e4m3(v / scale) with the division in fp32, so
    the row's largest element maps to +-448;
  * the gate/up GEMM multiplies the e4m3 codes exactly and applies
    scale_row * scale_channel to the fp32 accumulator before the SwiGLU; the
    down projection stays bf16.
"""
from __future__ import annotations

import numpy as np

from .bf16 import bf16_bits_to_f32, bf16_bits_to_f64, bf16_round_f64, f64_to_bf16_bits
from .moe_oracle import _silu

E4M3_MAX = 448.0


def e4m3_round(v) -> np.ndarray:
    """Round float values to the nearest e4m3 value (ties to even), saturating
    at +-448.  Returns float64 holding exact e4m3 values (NaN stays NaN)."""
    x = np.asarray(v, dtype=np.float64)
    out = np.zeros_like(x)
    a = np.abs(x)
    finite = np.isfinite(x)
    nz = finite & (a > 0)
    # exponent of the value's binade, clamped below at the subnormal range
    e = np.floor(np.log2(np.where(nz, a, 1.0)))
    # correct log2 rounding at binade edges
    e = np.where(nz & (2.0 ** e > a), e - 1, e)
    e = np.where(nz & (2.0 ** (e + 1) <= a), e + 1, e)
    e = np.maximum(e, -6.0)           # normals reach 2^-6; below, the quantum stays 2^-9
    q = 2.0 ** (e - 3)                # spacing: 3 mantissa bits
    r = np.rint(a / q) * q            # rint: ties to even
    r = np.minimum(r, E4M3_MAX)
    out = np.copysign(np.where(nz, r, 0.0), x)      # keeps the sign of zeros and underflows
    out = np.where(finite, out, np.where(np.isnan(x), np.nan, np.sign(x) * E4M3_MAX))
    return out


def e4m3_to_bits(v) -> np.ndarray:
    """Exact e4m3 values (as from e4m3_round) -> uint8 codes."""
    x = np.asarray(v, dtype=np.float64)
    sign = (np.signbit(x)).astype(np.uint8) << 7
    a = np.abs(x)
    code = np.zeros(x.shape, dtype=np.uint8)
    sub = (a > 0) & (a < 2.0 ** -6)
    code = np.where(sub, np.rint(a / 2.0 ** -9), code)           # subnormal: mantissa only
    nrm = a >= 2.0 ** -6
    e = np.floor(np.log2(np.where(nrm, a, 1.0)))
    m = np.rint((np.where(nrm, a, 1.0) / 2.0 ** e - 1.0) * 8.0)
    code = np.where(nrm, (e + 7) * 8 + m, code)
    return (code.astype(np.uint8) | sign).astype(np.uint8)


def e4m3_bits_to_f64(b) -> np.ndarray:
    """uint8 e4m3 codes -> float64 values (0x7f / 0xff are NaN)."""
    c = np.asarray(b, dtype=np.uint8).astype(np.int64)
    s = np.where(c & 0x80, -1.0, 1.0)
    ex = (c >> 3) & 0xF
    mt = c & 7
    val = np.where(ex == 0, mt * 2.0 ** -9, (1.0 + mt / 8.0) * 2.0 ** (ex - 7.0))
    val = np.where((c & 0x7F) == 0x7F, np.nan, val)
    return s * val


def quantize_rows(v_f32) -> tuple:
    """Rowwise e4m3: returns (codes uint8 [n, m], scale fp32 [n]).  scale =
    amax/448 in fp32 (1 for an all-zero row); code = e4m3(v / scale), the
    division in fp32."""
    v = np.asarray(v_f32, dtype=np.float32)
    amax = np.abs(v).max(axis=1) if v.shape[1] else np.zeros(v.shape[0], np.float32)
    scale = np.where(amax > 0, amax / np.float32(E4M3_MAX), np.float32(1.0)).astype(np.float32)
    scaled = (v / scale[:, None]).astype(np.float32)
    return e4m3_to_bits(e4m3_round(scaled)), scale


def dispatch_fp8(x_bits, row_token):
    """FP8 dispatch: each valid row r gets the e4m3 codes and scale of token
    row_token[r] (quantized once per token); pad and spare rows are zero codes
    with scale 0."""
    x = bf16_bits_to_f32(np.asarray(x_bits, dtype=np.uint16))
    codes, scale = quantize_rows(x)
    rt = np.asarray(row_token)
    C = rt.shape[0]
    q = np.zeros((C, x.shape[1]), dtype=np.uint8)
    s = np.zeros(C, dtype=np.float32)
    ok = rt >= 0
    q[ok] = codes[rt[ok]]
    s[ok] = scale[rt[ok]]
    return q, s


def expert_gate_up_fp8(qx, sx, qw1e, sw1e, I, rnd=bf16_round_f64):
    """h = bf16(silu(g) * u) with [g | u] = (qx qw1e^T) * sx[:, None] * sw1e[None, :],
    exact in fp64 from the e4m3 codes."""
    a = e4m3_bits_to_f64(qx)
    b = e4m3_bits_to_f64(qw1e)
    acc = a @ b.T
    gu = acc * np.asarray(sx, np.float64)[:, None] * np.asarray(sw1e, np.float64)[None, :]
    g, u = gu[:, :I], gu[:, I:]
    return rnd(_silu(g) * u)


def grouped_experts_fp8(qx_disp, sx_disp, row_expert, row_weight, qW1, sW1, W2_bits, I,
                        experts=None):
    """The experts with the FP8 gate/up GEMM.  Returns (y bits [C, H], h bits
    [C, I]); h from expert_gate_up_fp8, o = h W2^T and y = bf16(w o) as in the
    bf16 experts; sentinel rows stay zero.  qW1[e], sW1[e], W2_bits[e] are read
    only for the experts computed: all that have rows, or those in ``experts``."""
    re = np.asarray(row_expert)
    C, H = np.asarray(qx_disp).shape
    todo = sorted(set(int(e) for e in np.unique(re) if 0 <= e < len(W2_bits)) if experts is None
                  else set(experts))
    h_bits = np.zeros((C, I), dtype=np.uint16)
    y_bits = np.zeros((C, H), dtype=np.uint16)
    for e in todo:
        R = np.flatnonzero(re == e)
        if R.size == 0:
            continue
        h = expert_gate_up_fp8(qx_disp[R], np.asarray(sx_disp)[R], qW1[e], sW1[e], I)
        o = h @ bf16_bits_to_f64(W2_bits[e]).T
        y = bf16_round_f64(np.asarray(row_weight, np.float64)[R, None] * o)
        h_bits[R] = f64_to_bf16_bits(h)
        y_bits[R] = f64_to_bf16_bits(y)
    return y_bits, h_bits
