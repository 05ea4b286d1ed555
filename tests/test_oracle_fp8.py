"""Pins of the FP8 oracle: e4m3 rounding and codes against torch's float8_e4m3fn
(a library routine) and hand-worked values; rowwise quantization by its
defining properties; the FP8 gate/up GEMM against torch fp64 on the decoded
values, and against the bf16 expert oracle where the two must agree exactly."""
import numpy as np
import pytest
import torch

import oracle as O
from tests._util import random_routing


def test_e4m3_round_and_codes_match_torch_within_range():
    rng = np.random.default_rng(0)
    x = np.concatenate([
        rng.standard_normal(200000).astype(np.float32) * 50,
        rng.standard_normal(50000).astype(np.float32) * 1e-2,       # subnormals and small normals
        np.float32([0.0, -0.0, 448.0, -448.0, 2 ** -9, 2 ** -10, 3 * 2 ** -11, 2 ** -6, 1.0625,
                    1.1875, 0.001953125, 240.0, 232.0, 464.0 - 1e-3]),
    ]).astype(np.float32)
    x = x[np.abs(x) < 464]                       # torch does not saturate past the rounding edge
    t = torch.from_numpy(x).to(torch.float8_e4m3fn)
    np.testing.assert_array_equal(O.e4m3_round(x), t.to(torch.float64).numpy())
    np.testing.assert_array_equal(O.e4m3_to_bits(O.e4m3_round(x)), t.view(torch.uint8).numpy())


def test_e4m3_decode_all_codes_matches_torch():
    codes = np.arange(256, dtype=np.uint8)
    got = O.e4m3_bits_to_f64(codes)
    ref = torch.from_numpy(codes).view(torch.float8_e4m3fn).to(torch.float64).numpy()
    assert np.all((got == ref) | (np.isnan(got) & np.isnan(ref)))


@pytest.mark.parametrize("v,code,value", [
    (1.0, 0x38, 1.0), (448.0, 0x7E, 448.0), (-448.0, 0xFE, -448.0), (2.0 ** -9, 0x01, 2.0 ** -9),
    (1.0625, 0x38, 1.0),      # halfway between 1 and 1.125: ties to the even mantissa (1.0)
    (1.1875, 0x3A, 1.25),     # halfway between 1.125 and 1.25: ties to even (1.25)
    (500.0, 0x7E, 448.0),     # saturates
    (-1e6, 0xFE, -448.0),
    (0.0, 0x00, 0.0),
])
def test_e4m3_hand_worked(v, code, value):
    r = O.e4m3_round(np.float32([v]))
    assert r[0] == value
    assert O.e4m3_to_bits(r)[0] == code


def test_quantize_rows_properties():
    rng = np.random.default_rng(1)
    v = (rng.standard_normal((64, 256)) * rng.uniform(0.01, 100, (64, 1))).astype(np.float32)
    v[5] = 0.0
    codes, scale = O.quantize_rows(v)
    deq = O.e4m3_bits_to_f64(codes) * scale[:, None].astype(np.float64)
    # the largest element of every non-zero row maps to +-448
    j = np.abs(v).argmax(axis=1)
    top = np.abs(O.e4m3_bits_to_f64(codes[np.arange(64), j]))
    assert np.all(top[np.arange(64) != 5] == 448.0)
    assert scale[5] == 1.0 and not codes[5].any()
    # rounding error: at most half an e4m3 spacing (relative 2^-4) of the scaled value,
    # or half the subnormal quantum
    err = np.abs(deq - v)
    bound = np.maximum(np.abs(v) * 2.0 ** -4, 2.0 ** -10 * scale[:, None]) * (1 + 1e-6)
    assert np.all(err <= bound)
    np.testing.assert_array_equal(scale, np.where(np.abs(v).max(1) > 0,
                                                  np.abs(v).max(1) / np.float32(448), 1).astype(np.float32))


def test_dispatch_fp8_rows():
    T, H, E, K, P = 40, 256, 8, 2, 4
    idx, p = random_routing(T, E, K, seed=2, drop=0.2)
    rm, pr, _ = O.route_to_multihot(idx.numpy(), p.numpy(), E)
    L = O.build_layout(rm, pr, K, P, O.worst_case_capacity(T, E, K, P))
    x = torch.randn(T, H, generator=torch.Generator().manual_seed(2)).to(torch.bfloat16)
    xb = x.view(torch.int16).numpy().view(np.uint16)
    q, s = O.dispatch_fp8(xb, L["row_token"])
    codes, scale = O.quantize_rows(x.float().numpy())
    rt = L["row_token"]
    for r in range(rt.shape[0]):
        if rt[r] >= 0:
            assert np.array_equal(q[r], codes[rt[r]]) and s[r] == scale[rt[r]]
        else:
            assert not q[r].any() and s[r] == 0


def test_gate_up_fp8_matches_torch_on_decoded_values():
    rng = np.random.default_rng(3)
    n, H, I = 17, 256, 64
    x = rng.standard_normal((n, H)).astype(np.float32)
    w = (rng.standard_normal((2 * I, H)) * 0.02).astype(np.float32)
    qx, sx = O.quantize_rows(x)
    qw, sw = O.quantize_rows(w)
    got = O.expert_gate_up_fp8(qx, sx, qw, sw, I, rnd=lambda z: z)
    a = torch.from_numpy(qx).view(torch.float8_e4m3fn).to(torch.float64) * torch.from_numpy(sx).double()[:, None]
    b = torch.from_numpy(qw).view(torch.float8_e4m3fn).to(torch.float64) * torch.from_numpy(sw).double()[:, None]
    gu = a @ b.T
    ref = torch.nn.functional.silu(gu[:, :I]) * gu[:, I:]
    np.testing.assert_allclose(got, ref.numpy(), rtol=1e-12, atol=1e-15)


def test_fp8_experts_equal_bf16_experts_when_values_are_exact_e4m3():
    """Rows whose values are e4m3 numbers with amax 448 quantize with scale 1
    and no rounding, so the FP8 experts equal the (separately pinned) bf16
    experts on the same values, bit for bit."""
    rng = np.random.default_rng(4)
    T, H, E, K, I, P = 24, 256, 4, 2, 64, 1
    grid = O.e4m3_bits_to_f64(np.arange(0, 0x7F, dtype=np.uint8))      # non-negative e4m3 values
    grid = np.concatenate([grid, -grid])
    x = rng.choice(grid, (T, H)).astype(np.float32)
    x[:, 0] = 448.0
    W1 = rng.choice(grid, (E, 2 * I, H)).astype(np.float32)
    W1[:, :, 0] = 448.0
    W2 = (rng.standard_normal((E, H, I)) * 0.02).astype(np.float32)
    to_bits = lambda a: torch.from_numpy(a).to(torch.bfloat16).view(torch.int16).numpy().view(np.uint16)
    xb, W1b, W2b = to_bits(x), to_bits(W1), to_bits(W2)          # e4m3 values are exact in bf16
    idx, p = random_routing(T, E, K, seed=4)
    rm, pr, _ = O.route_to_multihot(idx.numpy(), p.numpy(), E)
    L = O.build_layout(rm, pr, K, P, O.worst_case_capacity(T, E, K, P))
    qx, sx = O.dispatch_fp8(xb, L["row_token"])
    assert np.all(sx[L["row_token"] >= 0] == 1.0)
    qW1 = np.stack([O.quantize_rows(W1[e])[0] for e in range(E)])
    sW1 = np.stack([O.quantize_rows(W1[e])[1] for e in range(E)])
    assert np.all(sW1 == 1.0)
    y8, h8 = O.grouped_experts_fp8(qx, sx, L["row_expert"], L["row_weight"], qW1, sW1, W2b, I)
    y16, h16, _ = O.grouped_experts(O.dispatch(xb, L["row_token"]), L["row_expert"], L["row_weight"],
                                    W1b, W2b, I)
    assert np.array_equal(h8, h16) and np.array_equal(y8, y16)
