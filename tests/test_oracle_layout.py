"""Pins for the oracle's multihot, counts/offsets, layout, dispatch and combine.

Multihot cases are hand-worked (tests/golden/multihot_cases.json); the layout
is checked against a hand-worked example and against Python's stable
``sorted`` of the (expert, token) pairs; counts against a brute-force set
count; dispatch + identity experts + combine against closed forms.
"""
import json
import os

import numpy as np
import pytest

import torch

import oracle as O
import synthetic

GOLDEN = os.path.join(os.path.dirname(__file__), "golden", "multihot_cases.json")


def _cases():
    with open(GOLDEN) as f:
        return json.load(f)


@pytest.mark.parametrize("case", _cases()["cases"], ids=lambda c: c["name"])
def test_multihot_golden(case):
    idx = np.array(case["idx"], dtype=np.int64)
    p = np.array(case["p"], dtype=np.float32)
    m, probs, win = O.route_to_multihot(idx, p, case["E"])
    assert np.array_equal(m, np.array(case["map"], dtype=np.uint8))
    assert np.array_equal(probs, np.array(case["probs"], dtype=np.float32))
    assert np.array_equal(win, np.array(case["winner"], dtype=np.int8))


@pytest.mark.parametrize("bad", [-2, 4, 100])
def test_multihot_rejects_out_of_range(bad):
    idx = np.array([[0, bad]], dtype=np.int64)
    with pytest.raises(O.OracleIndexError):
        O.route_to_multihot(idx, np.ones((1, 2), np.float32), 4)


def test_layout_golden():
    g = _cases()
    L0 = g["layout"]
    case = [c for c in g["cases"] if c["name"] == L0["case"]][0]
    m, probs, _ = O.route_to_multihot(np.array(case["idx"]), np.array(case["p"], np.float32), case["E"])
    L = O.build_layout(m, probs, L0["K"], L0["P"])
    for key in ("tokens_per_expert", "offsets", "row_token", "row_expert", "token_row"):
        assert np.array_equal(np.asarray(L[key]), np.array(L0[key])), key
    assert np.array_equal(L["row_weight"], np.array(L0["row_weight"], np.float32))
    assert L["rows_used"] == 8 and L["rows_valid"] == 6


def _random_routing(T, E, K, seed, drop=0.1, dup=0.1):
    rng = np.random.default_rng(seed)
    idx = rng.integers(0, E, size=(T, K))
    idx[rng.random((T, K)) < drop] = -1
    # occasional duplicates: copy slot 0 into another slot
    d = rng.random(T) < dup
    if K > 1:
        idx[d, K - 1] = idx[d, 0]
    p = rng.random((T, K)).astype(np.float32)
    return idx.astype(np.int64), p


@pytest.mark.parametrize("T,E,K,P", [(1, 4, 1, 1), (37, 8, 2, 16), (200, 16, 4, 8),
                                     (513, 32, 8, 128), (64, 8, 8, 3)])
def test_layout_against_sorted_pairs(T, E, K, P):
    idx, p = _random_routing(T, E, K, seed=T * 31 + E)
    m, probs, win = O.route_to_multihot(idx, p, E)
    # brute-force: the set of distinct valid (t, e) pairs
    pairs = {(t, int(e)) for t in range(T) for e in idx[t] if e >= 0}
    L = O.build_layout(m, probs, K, P)
    counts, offsets = L["tokens_per_expert"], L["offsets"]
    assert counts.sum() == len(pairs) == L["rows_valid"]
    for e in range(E):
        assert counts[e] == sum(1 for (_, ee) in pairs if ee == e)
        pad = offsets[e + 1] - offsets[e]
        assert pad % P == 0 and 0 <= pad - counts[e] < P
        if counts[e] == 0:
            assert pad == 0
    assert np.all(np.diff(offsets) >= 0) and offsets[0] == 0
    # the valid rows, read in row order, are the stable sort of (e, t) pairs
    valid = L["row_token"] >= 0
    got = list(zip(L["row_token"][valid].tolist(), L["row_expert"][valid].tolist()))
    assert got == sorted(pairs, key=lambda pr: (pr[1], pr[0]))
    # each valid row is inside its expert's range; pad rows are sentinel rows
    SENT = O.sentinel_expert(E)
    for r in range(L["capacity"]):
        e = L["row_expert"][r]
        if L["row_token"][r] >= 0:
            assert offsets[e] <= r < offsets[e] + counts[e]
            assert L["row_weight"][r] == probs[L["row_token"][r], e]
        else:
            assert e == SENT and L["row_weight"][r] == 0.0
    # token_row: brute force per token
    for t in range(T):
        es = sorted({int(e) for e in idx[t] if e >= 0})
        rows = [r for r in range(L["capacity"]) if L["row_token"][r] == t]
        assert [L["row_expert"][r] for r in rows] == es
        assert L["token_row"][t].tolist() == rows + [-1] * (K - len(rows))


def test_layout_capacity_and_spare_rows():
    idx, p = _random_routing(50, 8, 2, seed=5)
    m, probs, _ = O.route_to_multihot(idx, p, 8)
    C = O.worst_case_capacity(50, 8, 2, 4)
    L = O.build_layout(m, probs, 2, 4, capacity=C)
    R = L["rows_used"]
    assert L["capacity"] == C and R <= C
    assert np.all(L["row_token"][R:] == -1) and np.all(L["row_expert"][R:] == 8)
    assert np.all(L["row_weight"][R:] == 0)
    with pytest.raises(O.OracleCapacityError):
        O.build_layout(m, probs, 2, 4, capacity=R - 1)


def test_worst_case_capacity_is_reached():
    # every slot valid and distinct, every expert one row past a multiple of P
    T, E, K, P = 9, 3, 2, 4
    idx = np.array([[t % E, (t + 1) % E] for t in range(T)])
    m, probs, _ = O.route_to_multihot(idx, np.ones((T, K), np.float32), E)
    L = O.build_layout(m, probs, K, P)
    assert L["rows_valid"] == T * K
    # counts are 6 each -> padded to 8 each: 24 <= 18 + 3*3 = 27
    assert L["rows_used"] <= O.worst_case_capacity(T, E, K, P)


def test_dispatch_bitwise_and_zero_rows():
    cfg = synthetic.CONFIGS["tiny"]
    inp = synthetic.make_layer_inputs(cfg, with_weights=False)
    x = inp["x"].view(torch.int16).numpy().view(np.uint16)
    m, probs, _ = O.route_to_multihot(inp["topk_idx"].numpy(), inp["topk_probs"].numpy(), cfg.E)
    L = O.build_layout(m, probs, cfg.K, cfg.P, capacity=O.worst_case_capacity(cfg.T, cfg.E, cfg.K, cfg.P))
    xd = O.dispatch(x, L["row_token"])
    for r in range(L["capacity"]):
        t = L["row_token"][r]
        if t >= 0:
            assert np.array_equal(xd[r], x[t])
        else:
            assert not xd[r].any()


def _identity_experts(x_disp_bits, row_weight, row_expert, E):
    """y = bf16(w * x): the expert replaced by the identity."""
    y = O.f64_to_bf16_bits(row_weight.astype(np.float64)[:, None] * O.bf16_bits_to_f64(x_disp_bits))
    y[row_expert >= E] = 0
    return y


def _bits(a):
    return O.f64_to_bf16_bits(np.asarray(a, dtype=np.float64))


def test_identity_topk1_returns_x_bitwise():
    rng = np.random.default_rng(3)
    T, E, H = 40, 5, 16
    x = _bits(rng.standard_normal((T, H)))
    idx = rng.integers(0, E, size=(T, 1))
    m, probs, _ = O.route_to_multihot(idx, np.ones((T, 1), np.float32), E)
    L = O.build_layout(m, probs, 1, 4)
    y = _identity_experts(O.dispatch(x, L["row_token"]), L["row_weight"], L["row_expert"], E)
    assert np.array_equal(O.combine(y, L["token_row"]), x)


def test_identity_two_rows_unit_weight_is_2x():
    rng = np.random.default_rng(4)
    T, E, H = 30, 6, 8
    x = _bits(rng.standard_normal((T, H)))
    idx = np.stack([rng.permutation(E)[:2] for _ in range(T)])
    m, probs, _ = O.route_to_multihot(idx, np.ones((T, 2), np.float32), E)
    L = O.build_layout(m, probs, 2, 2)
    y = _identity_experts(O.dispatch(x, L["row_token"]), L["row_weight"], L["row_expert"], E)
    out = O.combine(y, L["token_row"])
    assert np.array_equal(O.bf16_bits_to_f64(out), 2.0 * O.bf16_bits_to_f64(x))


def test_identity_general_weights_scale_x():
    """out ~= x * (sum of the token's weights), within 2 bf16 ulp."""
    rng = np.random.default_rng(5)
    T, E, K, H = 64, 8, 4, 32
    x = _bits(rng.standard_normal((T, H)))
    idx = np.stack([rng.permutation(E)[:K] for _ in range(T)])
    idx[rng.random((T, K)) < 0.2] = -1
    p = rng.random((T, K)).astype(np.float32)
    m, probs, _ = O.route_to_multihot(idx, p, E)
    L = O.build_layout(m, probs, K, 8)
    y = _identity_experts(O.dispatch(x, L["row_token"]), L["row_weight"], L["row_expert"], E)
    out = O.bf16_bits_to_f64(O.combine(y, L["token_row"]))
    wsum = probs.astype(np.float64).sum(axis=1)
    ref = O.bf16_bits_to_f64(x) * wsum[:, None]
    ulp = np.ldexp(1.0, np.frexp(np.abs(ref))[1] - 8)
    assert np.all(np.abs(out - ref) <= 2 * ulp + 1e-30)


def test_all_invalid_gives_zero_and_no_rows():
    T, E, K, H = 7, 4, 3, 8
    idx = -np.ones((T, K), dtype=np.int64)
    m, probs, _ = O.route_to_multihot(idx, np.ones((T, K), np.float32), E)
    L = O.build_layout(m, probs, K, 16, capacity=O.worst_case_capacity(T, E, K, 16))
    assert L["rows_used"] == 0 and L["rows_valid"] == 0
    y = np.zeros((L["capacity"], H), np.uint16)
    out = O.combine(y, L["token_row"])
    assert np.array_equal(out, np.zeros((T, H), np.uint16))   # +0.0, not -0.0


def test_sentinel_rows_poisoned_with_nan_do_not_reach_out():
    rng = np.random.default_rng(6)
    T, E, K, H = 33, 6, 2, 16
    x = _bits(rng.standard_normal((T, H)))
    idx = np.stack([rng.permutation(E)[:K] for _ in range(T)])
    idx[::5, 1] = -1
    m, probs, _ = O.route_to_multihot(idx, rng.random((T, K)).astype(np.float32), E)
    L = O.build_layout(m, probs, K, 8, capacity=O.worst_case_capacity(T, E, K, 8))
    y = _identity_experts(O.dispatch(x, L["row_token"]), L["row_weight"], L["row_expert"], E)
    ref = O.combine(y, L["token_row"])
    y2 = y.copy()
    y2[L["row_token"] < 0] = 0x7FC0     # NaN on every pad / spare row
    assert np.array_equal(O.combine(y2, L["token_row"]), ref)


def test_combine_order_is_fixed_fp32():
    """Rows 1, 2^-8, 2^-25, 2^-25, 2^-25.  In row order each 2^-25 is a quarter
    of an fp32 ulp of 1 + 2^-8 and vanishes, leaving the bf16 tie 1 + 2^-8,
    which rounds to 1.  Summed small-first, the three add up to 3/4 ulp and
    push the sum past the tie, so it rounds to 1 + 2^-7.  An fp64 accumulator
    would also give 1 + 2^-7 in row order."""
    y = _bits(np.array([[1.0], [2.0**-8], [2.0**-25], [2.0**-25], [2.0**-25]]))
    fwd = O.combine(y, np.array([[0, 1, 2, 3, 4]]))
    rev = O.combine(y, np.array([[2, 3, 4, 1, 0]]))
    assert O.bf16_bits_to_f64(fwd)[0, 0] == 1.0
    assert O.bf16_bits_to_f64(rev)[0, 0] == 1.0 + 2.0**-7
