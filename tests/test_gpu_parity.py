"""GPU parity: the CUDA path, called through the C ABI, against the CPU oracle.

Bit-exact: multihot, counts, offsets, the layout, the dispatched rows, the
combine (given the same expert outputs), the backward gathers and scatters.
Within the bf16 GEMM tolerance (max |err| <= 2e-2, rel L2 <= 5e-3): the
expert outputs y and o and the layer output; the intermediates h and the
gate/up pre-activations use the same bound scaled by max(1, |ref|).
"""
import ctypes

import numpy as np
import pytest
import torch

import oracle as O
import synthetic
from tests._util import (assert_gemm_close, bits, from_bits, random_routing)

pytestmark = pytest.mark.gpu


@pytest.fixture(scope="module")
def moe():
    assert torch.cuda.is_available(), "GPU tests need a GPU"
    import combine_topk_multihot_gb300 as m
    assert m._native.lib.moe_device_check() == 0, m._native.last_error()
    return m


DEV = "cuda"


def _layout_case(moe, idx, p, E, P, capacity, host_sync, H=256, x=None):
    T, K = idx.shape
    status = torch.zeros(1, dtype=torch.int32, device=DEV)
    rmap, probs, win = moe.moe_route_to_multihot(idx.to(DEV), p.to(DEV), E, status)
    L = moe.Layout(T, E, K, P, capacity, device=DEV, status=status)
    if x is None:
        x = torch.randn(T, H, generator=torch.Generator().manual_seed(T + E)).to(torch.bfloat16)
    x_disp, rows = moe.moe_dispatch(x.to(DEV), rmap, probs, L, host_sync=host_sync)
    torch.cuda.synchronize()
    return dict(rmap=rmap, probs=probs, win=win, L=L, x=x, x_disp=x_disp, rows=rows, status=status)


def _check_layout(g, idx, p, E, P, capacity):
    T, K = idx.shape
    rm, pr, wn = O.route_to_multihot(idx.numpy(), p.numpy(), E)
    assert np.array_equal(g["rmap"].cpu().numpy(), rm)
    assert np.array_equal(g["probs"].cpu().numpy(), pr)
    assert np.array_equal(g["win"].cpu().numpy(), wn)
    Lr = O.build_layout(rm, pr, K, P, capacity)
    L = g["L"]
    assert np.array_equal(L.tokens_per_expert.cpu().numpy(), Lr["tokens_per_expert"])
    assert np.array_equal(L.offsets.cpu().numpy(), Lr["offsets"])
    assert L.totals.cpu().tolist() == [Lr["rows_used"], Lr["rows_valid"]]
    assert np.array_equal(L.row_token.cpu().numpy(), Lr["row_token"])
    assert np.array_equal(L.row_expert.cpu().numpy(), Lr["row_expert"])
    assert np.array_equal(L.row_weight.cpu().numpy(), Lr["row_weight"])
    assert np.array_equal(L.token_row.cpu().numpy().reshape(T, K), Lr["token_row"])
    assert np.array_equal(bits(g["x_disp"]), O.dispatch(bits(g["x"]), Lr["row_token"]))
    if g["rows"] is not None:
        assert g["rows"] == (Lr["rows_used"], Lr["rows_valid"])
    assert int(g["status"].item()) == 0
    return Lr


# ----------------------------------------------------------------- a1-a4

@pytest.mark.parametrize("T,E,K,P,drop,dup", [
    (64, 8, 2, 16, 0.0, 0.0),       # the tiny layer's shape
    (1, 8, 2, 16, 0.0, 0.0),        # single token
    (77, 12, 3, 5, 0.2, 0.2),       # ragged chunk tail, drops, duplicates
    (513, 32, 8, 128, 0.1, 0.1),    # several chunks, ragged tail
    (300, 1024, 4, 1, 0.0, 0.0),    # the largest E
    (40, 8, 1, 3, 0.0, 0.0),        # topk = 1
    (33, 4, 4, 2, 0.0, 0.0),        # K = E
    (0, 8, 2, 16, 0.0, 0.0),        # no tokens
    (65, 64, 4, 8, 0.1, 0.1),       # 3 chunks: one CTA per chunk, each counting all of them
    (256, 128, 8, 1, 0.05, 0.05),   # 8 chunks: the largest layer laid out without a grid barrier
    (257, 128, 8, 16, 0.0, 0.0),    # 9 chunks: the cooperative layout kernel
    (1024, 128, 8, 1, 0.05, 0.05),  # 32 chunks
    (40000, 128, 8, 4, 0.05, 0.0),  # 1250 chunks: more than the layout kernel's resident CTAs
])
@pytest.mark.parametrize("host_sync", [True, False])
def test_multihot_and_layout(moe, T, E, K, P, drop, dup, host_sync):
    idx, p = random_routing(T, E, K, seed=T * 7 + E, drop=drop, dup=dup)
    C = O.worst_case_capacity(T, E, K, P)
    g = _layout_case(moe, idx, p, E, P, C, host_sync)
    _check_layout(g, idx, p, E, P, C)


@pytest.mark.parametrize("T,E,K,P,drop,dup", [
    (1, 128, 8, 1, 0.0, 0.0),       # the decode T = 1 layer
    (4, 16, 4, 1, 0.2, 0.2),        # drops and duplicates
    (3, 8, 2, 4, 0.0, 0.0),         # pad rows
    (8, 8, 7, 1, 0.0, 0.0),         # 64 items: the largest row pass the layout CTA takes
    (9, 8, 7, 1, 0.0, 0.0),         # 72 items: a separate row pass
    (0, 8, 2, 8, 0.0, 0.0),         # no tokens: spare rows only
])
@pytest.mark.parametrize("layout_only", [False, True])
def test_single_cta_row_pass(moe, T, E, K, P, drop, dup, layout_only):
    """Sync-free layers of a few rows: the one-CTA layout kernel also copies
    the rows and writes the pad and spare rows.  Every output buffer starts
    out poisoned, so each row must have been written."""
    idx, p = random_routing(T, E, K, seed=T * 11 + E, drop=drop, dup=dup)
    H = 512
    C = O.worst_case_capacity(T, E, K, P)
    status = torch.zeros(1, dtype=torch.int32, device=DEV)
    rmap, probs, _ = moe.moe_route_to_multihot(idx.to(DEV), p.to(DEV), E, status)
    L = moe.Layout(T, E, K, P, C, device=DEV, status=status)
    L.row_token.fill_(12345)
    L.row_expert.fill_(-7)
    L.row_weight.fill_(float("nan"))
    L.token_row.fill_(999)
    x = torch.randn(T, H, generator=torch.Generator().manual_seed(T + 1)).to(torch.bfloat16)
    x_disp = torch.full((C, H), float("nan"), dtype=torch.bfloat16, device=DEV)
    if layout_only:
        moe.moe_dispatch_layout(rmap, probs, L, host_sync=False)
    else:
        moe.moe_dispatch(x.to(DEV), rmap, probs, L, host_sync=False, x_disp=x_disp)
    torch.cuda.synchronize()
    assert int(status.item()) == 0
    rm, pr, _ = O.route_to_multihot(idx.numpy(), p.numpy(), E)
    Lr = O.build_layout(rm, pr, K, P, C)
    assert L.totals.cpu().tolist() == [Lr["rows_used"], Lr["rows_valid"]]
    for f in ("row_token", "row_expert", "row_weight"):
        assert np.array_equal(getattr(L, f).cpu().numpy(), Lr[f]), f
    assert np.array_equal(L.token_row.cpu().numpy().reshape(T, K), Lr["token_row"])
    if not layout_only:
        assert np.array_equal(bits(x_disp), O.dispatch(bits(x), Lr["row_token"]))


LAYOUT_CASES = [
    (1, 8, 2, 16, 0.0, 0.0),        # single token
    (77, 12, 3, 5, 0.2, 0.2),       # ragged chunk tail, drops, duplicates
    (256, 128, 8, 1, 0.05, 0.05),   # 8 chunks: the multihot kernel, then the barrier-free layout
    (257, 128, 8, 16, 0.0, 0.0),    # 9 chunks: one cooperative kernel for all of it
    (513, 32, 8, 128, 0.1, 0.1),    # several chunks, ragged tail, drops, duplicates
    (700, 1024, 4, 1, 0.0, 0.0),    # the largest E (8 stripes of 128 experts per token row)
    (300, 16, 16, 3, 0.1, 0.3),     # K = E, duplicates
    (333, 64, 40, 2, 0.2, 0.2),     # K > 32: slots in two registers per lane
    (4096, 128, 8, 128, 0.0, 0.0),  # the Qwen3-30B-A3B routing shape
    (40000, 128, 8, 4, 0.05, 0.0),  # more chunks than resident CTAs
    (0, 8, 2, 16, 0.0, 0.0),        # no tokens
]


@pytest.mark.parametrize("T,E,K,P,drop,dup", LAYOUT_CASES)
@pytest.mark.parametrize("host_sync", [True, False])
def test_dispatch_topk_matches_oracle(moe, T, E, K, P, drop, dup, host_sync):
    """moe_dispatch_topk (the multihot step fused into the dispatch): the
    multihot outputs, the layout and the rows bit for bit against the oracle,
    with every row buffer poisoned first so each entry must be written."""
    idx, p = random_routing(T, E, K, seed=T * 5 + E + K, drop=drop, dup=dup)
    H = 512 if T < 5000 else 256
    C = O.worst_case_capacity(T, E, K, P)
    status = torch.zeros(1, dtype=torch.int32, device=DEV)
    L = moe.Layout(T, E, K, P, C, device=DEV, status=status)
    L.row_token.fill_(12345)
    L.row_expert.fill_(-7)
    L.row_weight.fill_(float("nan"))
    L.token_row.fill_(999)
    x = torch.randn(T, H, generator=torch.Generator().manual_seed(T + 3)).to(torch.bfloat16)
    x_disp = torch.full((C, H), float("nan"), dtype=torch.bfloat16, device=DEV)
    mh = (torch.full((T, E), 7, dtype=torch.uint8, device=DEV),
          torch.full((T, E), float("nan"), dtype=torch.float32, device=DEV),
          torch.full((T, E), 5, dtype=torch.int8, device=DEV))
    _, mh, rows = moe.moe_dispatch_topk(x.to(DEV), idx.to(DEV), p.to(DEV), L, host_sync=host_sync,
                                        x_disp=x_disp, multihot=mh)
    torch.cuda.synchronize()
    g = dict(rmap=mh[0], probs=mh[1], win=mh[2], L=L, x=x, x_disp=x_disp, rows=rows, status=status)
    _check_layout(g, idx, p, E, P, C)


@pytest.mark.parametrize("T,E,K,P", [(257, 128, 8, 16), (3000, 64, 6, 32)])
def test_fused_dispatch_writes_every_row(moe, T, E, K, P):
    """moe_dispatch on layers of more than 8 chunks (the cooperative kernel
    that places and copies in one launch), sync-free: poisoned row buffers
    and rows, so every valid, pad and spare row must be written."""
    idx, p = random_routing(T, E, K, seed=T + K, drop=0.1, dup=0.1)
    H = 768
    C = O.worst_case_capacity(T, E, K, P)
    status = torch.zeros(1, dtype=torch.int32, device=DEV)
    rmap, probs, _ = moe.moe_route_to_multihot(idx.to(DEV), p.to(DEV), E, status)
    L = moe.Layout(T, E, K, P, C, device=DEV, status=status)
    L.row_token.fill_(12345)
    L.row_expert.fill_(-7)
    L.row_weight.fill_(float("nan"))
    L.token_row.fill_(999)
    x = torch.randn(T, H, generator=torch.Generator().manual_seed(T)).to(torch.bfloat16)
    x_disp = torch.full((C, H), float("nan"), dtype=torch.bfloat16, device=DEV)
    moe.moe_dispatch(x.to(DEV), rmap, probs, L, host_sync=False, x_disp=x_disp)
    torch.cuda.synchronize()
    g = dict(rmap=rmap, probs=probs, win=moe.moe_route_to_multihot(idx.to(DEV), p.to(DEV), E, status)[2],
             L=L, x=x, x_disp=x_disp, rows=None, status=status)
    _check_layout(g, idx, p, E, P, C)


@pytest.mark.parametrize("T", [40, 600])
def test_dispatch_topk_bad_index(moe, T):
    E, K, P = 16, 2, 4
    idx, p = random_routing(T, E, K, seed=T)
    idx[5, 1] = E + 3
    status = torch.zeros(1, dtype=torch.int32, device=DEV)
    L = moe.Layout(T, E, K, P, O.worst_case_capacity(T, E, K, P), device=DEV, status=status)
    x = torch.zeros(T, 256, dtype=torch.bfloat16, device=DEV)
    with pytest.raises(moe.MoEError) as ei:
        moe.moe_dispatch_topk(x, idx.to(DEV), p.to(DEV), L, host_sync=True)
    assert ei.value.code == moe._native.MOE_ERR_BAD_INDEX
    # sync-free: the status bit, and the bad slot dropped as a -1 slot would be
    status.zero_()
    _, mh, _ = moe.moe_dispatch_topk(x, idx.to(DEV), p.to(DEV), L, host_sync=False)
    torch.cuda.synchronize()
    assert int(status.item()) & moe._native.MOE_DEVERR_BAD_INDEX
    idx2 = idx.clone()
    idx2[5, 1] = -1
    rm, pr, _ = O.route_to_multihot(idx2.numpy(), p.numpy(), E)
    assert np.array_equal(mh[0].cpu().numpy(), rm)
    Lr = O.build_layout(rm, pr, K, P, L.capacity)
    assert np.array_equal(L.row_token.cpu().numpy(), Lr["row_token"])


def test_all_invalid_routing(moe):
    T, E, K, P = 50, 8, 2, 4
    idx = -torch.ones(T, K, dtype=torch.int64)
    p = torch.rand(T, K)
    C = O.worst_case_capacity(T, E, K, P)
    g = _layout_case(moe, idx, p, E, P, C, True)
    assert g["rows"] == (0, 0)
    _check_layout(g, idx, p, E, P, C)


def test_host_synced_exact_capacity(moe):
    """Eager mode: a first call with no rows reports R, a second call with
    exactly R rows fills them."""
    T, E, K, P = 200, 16, 4, 8
    idx, p = random_routing(T, E, K, seed=3, drop=0.1)
    status = torch.zeros(1, dtype=torch.int32, device=DEV)
    rmap, probs, _ = moe.moe_route_to_multihot(idx.to(DEV), p.to(DEV), E, status)
    x = torch.randn(T, 256).to(torch.bfloat16).to(DEV)
    L0 = moe.Layout(T, E, K, P, 0, device=DEV, status=status)
    with pytest.raises(moe.MoEError) as ei:
        moe.moe_dispatch(x, rmap, probs, L0, host_sync=True)
    assert ei.value.code == moe._native.MOE_ERR_CAPACITY
    Lr = O.build_layout(*O.route_to_multihot(idx.numpy(), p.numpy(), E)[:2], K, P)
    R = Lr["rows_used"]
    status.zero_()
    L1 = moe.Layout(T, E, K, P, R, device=DEV, status=status)
    x_disp, rows = moe.moe_dispatch(x, rmap, probs, L1, host_sync=True)
    assert rows == (R, Lr["rows_valid"])
    assert np.array_equal(L1.row_token.cpu().numpy(), Lr["row_token"])
    assert np.array_equal(bits(x_disp), O.dispatch(bits(x), Lr["row_token"]))


@pytest.mark.parametrize("T,E,K,P", [
    (4, 8, 2, 4),        # one CTA lays out and copies
    (40, 8, 2, 4),       # one CTA lays out, the row kernel copies
    (2000, 32, 4, 16),   # the cooperative layout kernel and the row kernel
])
@pytest.mark.parametrize("fp8", [False, True])
def test_host_synced_short_capacity_writes_nothing(moe, T, E, K, P, fp8):
    """Host-synced, capacity one row short of R: MOE_ERR_CAPACITY, R and N
    still reported, and not a single output byte written -- the kernels are
    queued before the host knows R, so they must skip the work themselves."""
    idx, p = random_routing(T, E, K, seed=T + E, drop=0.1)
    Lr = O.build_layout(*O.route_to_multihot(idx.numpy(), p.numpy(), E)[:2], K, P)
    R = Lr["rows_used"]
    status = torch.zeros(1, dtype=torch.int32, device=DEV)
    rmap, probs, _ = moe.moe_route_to_multihot(idx.to(DEV), p.to(DEV), E, status)
    L = moe.Layout(T, E, K, P, R - 1, device=DEV, status=status)
    for f, v in (("row_token", 12345), ("row_expert", -7), ("row_weight", 0.5), ("token_row", 999)):
        getattr(L, f).fill_(v)
    H = 256
    x = torch.randn(T, H, generator=torch.Generator().manual_seed(T)).to(torch.bfloat16).to(DEV)
    rows = (ctypes.c_int64 * 2)()
    if fp8:
        q = torch.full((R - 1, H), 0x5A, dtype=torch.uint8, device=DEV)
        sc = torch.full((R - 1,), 3.0, dtype=torch.float32, device=DEV)
        code = moe._native.lib.moe_dispatch_fp8(moe.moe._ptr(x), moe.moe._ptr(rmap), moe.moe._ptr(probs), H,
                                                L.ref, moe.moe._ptr(q), moe.moe._ptr(sc), rows, None)
    else:
        xd = torch.full((R - 1, H), 7.0, dtype=torch.bfloat16, device=DEV)
        code = moe._native.lib.moe_dispatch(moe.moe._ptr(x), moe.moe._ptr(rmap), moe.moe._ptr(probs), H,
                                            L.ref, moe.moe._ptr(xd), rows, None)
    torch.cuda.synchronize()
    assert code == moe._native.MOE_ERR_CAPACITY
    assert (rows[0], rows[1]) == (R, Lr["rows_valid"])
    assert bool((L.row_token == 12345).all()) and bool((L.row_expert == -7).all())
    assert bool((L.row_weight == 0.5).all()) and bool((L.token_row == 999).all())
    if fp8:
        assert bool((q == 0x5A).all()) and bool((sc == 3.0).all())
    else:
        assert bool((xd == 7.0).all())
    assert int(status.item()) & moe._native.MOE_DEVERR_CAPACITY


def test_sync_free_rejects_small_capacity(moe):
    T, E, K, P = 10, 8, 2, 4
    idx, p = random_routing(T, E, K, seed=1)
    status = torch.zeros(1, dtype=torch.int32, device=DEV)
    rmap, probs, _ = moe.moe_route_to_multihot(idx.to(DEV), p.to(DEV), E, status)
    L = moe.Layout(T, E, K, P, O.worst_case_capacity(T, E, K, P) - 1, device=DEV, status=status)
    with pytest.raises(moe.MoEError) as ei:
        moe.moe_dispatch(torch.zeros(T, 256, dtype=torch.bfloat16, device=DEV), rmap, probs, L,
                         host_sync=False)
    assert ei.value.code == moe._native.MOE_ERR_CAPACITY


@pytest.mark.parametrize("bad", [-2, 8, 1 << 40])
def test_bad_index_is_reported(moe, bad):
    T, E, K, P = 20, 8, 2, 4
    idx, p = random_routing(T, E, K, seed=2)
    idx[5, 1] = bad
    status = torch.zeros(1, dtype=torch.int32, device=DEV)
    rmap, probs, _ = moe.moe_route_to_multihot(idx.to(DEV), p.to(DEV), E, status)
    torch.cuda.synchronize()
    assert int(status.item()) & moe._native.MOE_DEVERR_BAD_INDEX
    # the bad slot is dropped, as a -1 slot would be
    idx2 = idx.clone()
    idx2[5, 1] = -1
    assert np.array_equal(rmap.cpu().numpy(), O.route_to_multihot(idx2.numpy(), p.numpy(), E)[0])
    L = moe.Layout(T, E, K, P, O.worst_case_capacity(T, E, K, P), device=DEV, status=status)
    with pytest.raises(moe.MoEError) as ei:
        moe.moe_dispatch(torch.zeros(T, 256, dtype=torch.bfloat16, device=DEV), rmap, probs, L,
                         host_sync=True)
    assert ei.value.code == moe._native.MOE_ERR_BAD_INDEX


@pytest.mark.parametrize("name", ["qwen3_30b_a3b", "skewed", "decode_1", "decode_256", "decode_1024"])
def test_layout_full_size_configs(moe, name):
    cfg = synthetic.CONFIGS[name]
    idx, p = synthetic.make_routing(cfg.T, cfg.E, cfg.K, cfg.seed, cfg.zipf_s, cfg.drop)
    x = synthetic.make_tokens(cfg.T, cfg.H, cfg.seed)
    C = O.worst_case_capacity(cfg.T, cfg.E, cfg.K, cfg.P)
    g = _layout_case(moe, idx, p, cfg.E, cfg.P, C, host_sync=not cfg.sync_free, H=cfg.H, x=x)
    _check_layout(g, idx, p, cfg.E, cfg.P, C)


# ----------------------------------------------------------------- a5

def _experts_case(moe, T, H, E, K, I, P, seed, drop=0.0, save=True):
    idx, p = random_routing(T, E, K, seed=seed, drop=drop)
    gen = torch.Generator().manual_seed(seed)
    x = torch.randn(T, H, generator=gen).to(torch.bfloat16)
    W1 = (torch.randn(E, 2 * I, H, generator=gen) * 0.02).to(torch.bfloat16)
    W2 = (torch.randn(E, H, I, generator=gen) * 0.02).to(torch.bfloat16)
    C = O.worst_case_capacity(T, E, K, P)
    fwd = moe.moe_layer_forward(x.to(DEV), idx.to(DEV), p.to(DEV), W1.to(DEV), W2.to(DEV), P,
                                capacity=C, save_for_backward=save)
    torch.cuda.synchronize()
    return idx, p, x, W1, W2, C, fwd


@pytest.mark.parametrize("T,H,E,K,I,P", [
    (64, 256, 8, 2, 128, 16),      # the tiny layer
    (300, 512, 8, 2, 256, 16),     # 2 N tiles in each GEMM, ragged groups
    (1000, 256, 4, 2, 128, 1),     # several 128-row tiles per expert, unaligned groups
    (5, 1024, 8, 4, 384, 1),       # decode-like: a few rows, long K
    (260, 768, 12, 3, 128, 128),   # padded groups, 3 N tiles in GEMM2
    # the cases above have few experts with rows, so the GEMMs take 64-column
    # tiles; these have enough for 256-column tiles on every SM
    (64, 256, 64, 4, 384, 16),     # 256-column tiles, a few rows per expert
    (2000, 512, 40, 4, 512, 1),    # CTA pairs, rows on N: ~200 rows per expert, one chunk each
    (2304, 256, 256, 8, 128, 16),  # CTA pairs with two stages (E = 256: the per-expert tables take the third)
    (700, 256, 1024, 4, 128, 1),   # the largest E: per-expert tables take a pipeline stage
])
def test_experts_match_oracle(moe, T, H, E, K, I, P):
    idx, p, x, W1, W2, C, fwd = _experts_case(moe, T, H, E, K, I, P, seed=T + H)
    Lr = O.build_layout(*O.route_to_multihot(idx.numpy(), p.numpy(), E)[:2], K, P, C)
    xd = bits(fwd.x_disp)
    assert np.array_equal(xd, O.dispatch(bits(x), Lr["row_token"]))
    y, h, o = O.grouped_experts(xd, Lr["row_expert"], Lr["row_weight"], bits(W1), bits(W2), I)
    valid = Lr["row_token"] >= 0
    assert_gemm_close(bits(fwd.h)[valid], h[valid], "h", intermediate=True)
    assert_gemm_close(bits(fwd.y)[valid], y[valid], "y")
    assert_gemm_close(bits(fwd.o)[valid], o[valid], "o_save")
    # gate / up pre-activations
    gu = bits(fwd.gu)[valid]
    X = O.bf16_bits_to_f64(xd[valid])
    re = Lr["row_expert"][valid]
    W1f = O.bf16_bits_to_f64(bits(W1))
    gu_ref = np.stack([X[i] @ W1f[re[i]].T for i in range(X.shape[0])]) if X.shape[0] else np.zeros((0, 2 * I))
    assert_gemm_close(gu, O.f64_to_bf16_bits(gu_ref), "gu_save", intermediate=True)
    # the layer output: combine of the GPU's own y is bit-exact ...
    y_gpu = bits(fwd.y).copy()
    y_gpu[~valid] = 0
    assert np.array_equal(bits(fwd.out), O.combine(y_gpu, Lr["token_row"]))
    # ... and close to the oracle's layer output
    assert_gemm_close(bits(fwd.out), O.combine(y, Lr["token_row"]), "out")


@pytest.mark.parametrize("save", [True, False])
def test_experts_skewed_layer_matches_oracle(moe, save):
    """A skewed layer on CTA pairs (log-Zipf router bias, 5 % dropped slots, 40
    experts): the largest expert has over a thousand rows, so its tiles take
    many 256-row chunks and a ragged last one, next to experts with a few
    rows.  The layer averages 300 rows per expert, so with and without saved
    operands it runs the kernel with the expert rows on the MMA's N side;
    with them (training) the pad rows are written as zeros."""
    T, H, E, K, I, P = 3000, 512, 40, 4, 512, 16
    idx, p = synthetic.make_routing(T, E, K, seed=11, zipf_s=1.2, drop=0.05)
    counts = np.bincount(idx[idx >= 0].numpy().ravel(), minlength=E)
    assert counts.max() > 1000 and counts.min() < 64  # the shape the test is about
    gen = torch.Generator().manual_seed(12)
    x = torch.randn(T, H, generator=gen).to(torch.bfloat16)
    W1 = (torch.randn(E, 2 * I, H, generator=gen) * 0.02).to(torch.bfloat16)
    W2 = (torch.randn(E, H, I, generator=gen) * 0.02).to(torch.bfloat16)
    C = O.worst_case_capacity(T, E, K, P)
    fwd = moe.moe_layer_forward(x.to(DEV), idx.to(DEV), p.to(DEV), W1.to(DEV), W2.to(DEV), P,
                                capacity=C, save_for_backward=save)
    torch.cuda.synchronize()
    assert int(fwd.layout.status.item()) == 0
    Lr = O.build_layout(*O.route_to_multihot(idx.numpy(), p.numpy(), E)[:2], K, P, C)
    xd = bits(fwd.x_disp)
    assert np.array_equal(xd, O.dispatch(bits(x), Lr["row_token"]))
    y, h, o = O.grouped_experts(xd, Lr["row_expert"], Lr["row_weight"], bits(W1), bits(W2), I)
    valid = Lr["row_token"] >= 0
    assert_gemm_close(bits(fwd.h)[valid], h[valid], "h", intermediate=True)
    assert_gemm_close(bits(fwd.y)[valid], y[valid], "y")
    if save:
        assert_gemm_close(bits(fwd.o)[valid], o[valid], "o_save")
        # pad rows inside each group come out zero in every saved output
        pad = np.zeros(C, dtype=bool)
        offs, cnt = Lr["offsets"], Lr["tokens_per_expert"]
        for e in range(E):
            pad[offs[e] + cnt[e]:offs[e + 1]] = True
        for name in ("h", "y", "o", "gu"):
            assert not bits(getattr(fwd, name))[pad].any(), name
    assert_gemm_close(bits(fwd.out), O.combine(y, Lr["token_row"]), "out")


@pytest.mark.parametrize("T,H,E,K,I,P", [
    (1, 2048, 128, 8, 768, 1),     # the decode T = 1 layer: CUDA-core path
    (4, 512, 16, 4, 256, 1),       # four tokens: up to four rows per expert
    (3, 256, 8, 2, 128, 16),       # padded groups (pad rows not written)
    (2, 4096, 8, 2, 1536, 1),      # the h4096 expert shape
    (3, 8192, 8, 2, 128, 1),       # wide H: the A rows outgrow the CUDA-core path, tensor cores take it
    (4, 2048, 1024, 8, 768, 1),    # E = 1024: a long expert scan, 32 active experts
    (64, 256, 8, 2, 128, 16),      # tensor-core path without saved operands
    (1500, 512, 40, 8, 512, 1),    # CTA pairs: ~300 rows per expert, ragged last chunks
    (2048, 512, 16, 8, 1536, 128), # CTA pairs: ~1024 rows per expert, four full 256-row chunks each
    (2304, 256, 256, 8, 128, 1),   # CTA pairs with two stages (E = 256), ~72 rows per expert
])
def test_experts_inference_match_oracle(moe, T, H, E, K, I, P):
    """Inference (nothing saved for a backward): layers with at most four rows
    per expert take the CUDA-core path, larger ones the tensor cores; layers
    with rows for every SM and more than 64 rows per expert take CTA pairs
    with the expert rows on the MMA's N side."""
    idx, p, x, W1, W2, C, fwd = _experts_case(moe, T, H, E, K, I, P, seed=3 * T + H, save=False)
    Lr = O.build_layout(*O.route_to_multihot(idx.numpy(), p.numpy(), E)[:2], K, P, C)
    xd = bits(fwd.x_disp)
    y, h, _ = O.grouped_experts(xd, Lr["row_expert"], Lr["row_weight"], bits(W1), bits(W2), I)
    valid = Lr["row_token"] >= 0
    assert_gemm_close(bits(fwd.h)[valid], h[valid], "h", intermediate=True)
    assert_gemm_close(bits(fwd.y)[valid], y[valid], "y")
    assert_gemm_close(bits(fwd.out), O.combine(y, Lr["token_row"]), "out")


@pytest.mark.parametrize("save", [False, True])
def test_pair_gemm_repeated_launches_identical(moe, save):
    """Forty launch pairs of the CTA-pair GEMMs back to back on one stream:
    each pair takes the next of the 16 rotating slots of row-chunk readiness
    counters, which the down launch's last CTA clears for its next use.  A slot
    left dirty would let a down tile read h before it is written; every
    output must equal the first launch's bit for bit, and the first the
    oracle's within the bf16 tolerance."""
    T, H, E, K, I, P = 1500, 512, 40, 8, 512, 16
    idx, p = random_routing(T, E, K, seed=77, drop=0.05)
    gen = torch.Generator().manual_seed(78)
    x = torch.randn(T, H, generator=gen).to(torch.bfloat16)
    W1 = (torch.randn(E, 2 * I, H, generator=gen) * 0.02).to(torch.bfloat16).to(DEV)
    W2 = (torch.randn(E, H, I, generator=gen) * 0.02).to(torch.bfloat16).to(DEV)
    C = O.worst_case_capacity(T, E, K, P)
    L = moe.Layout(T, E, K, P, C, device=DEV)
    xd, _, _ = moe.moe_dispatch_topk(x.to(DEV), idx.to(DEV), p.to(DEV), L, host_sync=False)
    first = moe.moe_grouped_experts(xd, L, W1, W2, save_o=save, save_gu=save)
    ref = {k: v.clone() for k, v in first.items() if v is not None}
    valid_t = L.row_token >= 0  # the rows every launch writes
    outs = [dict(h=torch.empty_like(ref["h"]), y=torch.empty_like(ref["y"])) for _ in range(2)]
    for n in range(40):
        o = outs[n % 2]
        o["h"].fill_(float("nan"))
        o["y"].fill_(float("nan"))
        if save:
            o["o"], o["gu"] = torch.empty_like(ref["o"]), torch.empty_like(ref["gu"])
        moe.moe_grouped_experts(xd, L, W1, W2, save_o=save, save_gu=save, out=o)
        if n % 2:
            torch.cuda.synchronize()
            for k in ("h", "y"):
                for oo in outs:
                    assert torch.equal(oo[k][valid_t].view(torch.int16), ref[k][valid_t].view(torch.int16)), (n, k)
    torch.cuda.synchronize()
    assert int(L.status.item()) == 0
    Lr = O.build_layout(*O.route_to_multihot(idx.numpy(), p.numpy(), E)[:2], K, P, C)
    y, h, _ = O.grouped_experts(bits(xd), Lr["row_expert"], Lr["row_weight"], bits(W1), bits(W2), I)
    valid = Lr["row_token"] >= 0
    assert_gemm_close(bits(ref["h"])[valid], h[valid], "h", intermediate=True)
    assert_gemm_close(bits(ref["y"])[valid], y[valid], "y")


@pytest.mark.parametrize("save", [False, True])
def test_experts_sentinel_rows(moe, save):
    """Spare rows (R..C-1) are never written by the experts.  Pad rows inside
    an expert's group are left untouched in inference and written as zeros
    when the gate/up values are saved for the backward.  The combine reads
    neither: with every sentinel row poisoned with NaN beforehand its output
    is unchanged."""
    T, H, E, K, I, P = 90, 256, 8, 2, 128, 16
    idx, p = random_routing(T, E, K, seed=9, drop=0.3)
    x = torch.randn(T, H).to(torch.bfloat16).to(DEV)
    W1 = (torch.randn(E, 2 * I, H) * 0.02).to(torch.bfloat16).to(DEV)
    W2 = (torch.randn(E, H, I) * 0.02).to(torch.bfloat16).to(DEV)
    C = O.worst_case_capacity(T, E, K, P)
    fwd = moe.moe_layer_forward(x, idx.to(DEV), p.to(DEV), W1, W2, P, capacity=C)
    nan = torch.full((C, H), float("nan"), dtype=torch.bfloat16, device=DEV)
    nan_h = torch.full((C, I), float("nan"), dtype=torch.bfloat16, device=DEV)
    ex = moe.moe_grouped_experts(fwd.x_disp, fwd.layout, W1, W2, out={"y": nan.clone(), "h": nan_h},
                                 save_o=save, save_gu=save)
    R = int(fwd.layout.totals[0].item())
    pad = fwd.layout.row_expert == E
    pad[R:] = False
    assert torch.isnan(ex["y"][R:]).all() and torch.isnan(ex["h"][R:]).all()
    if save:
        assert (ex["y"][pad] == 0).all() and (ex["h"][pad] == 0).all()
        assert (ex["o"][pad] == 0).all() and (ex["gu"][pad] == 0).all()
    else:
        assert torch.isnan(ex["y"][pad]).all() and torch.isnan(ex["h"][pad]).all()
    valid = fwd.layout.row_token >= 0
    assert not torch.isnan(ex["y"][valid]).any()
    out = moe.moe_combine(ex["y"], fwd.layout)
    assert torch.equal(out.view(torch.int16), fwd.out.view(torch.int16))


@pytest.mark.parametrize("name", ["qwen3_30b_a3b"])
def test_experts_full_size_sampled_rows(moe, name):
    """Full-size layer in the benchmark's launch configuration; the oracle
    checks every row of four experts (the largest, the smallest non-empty and
    two others) plus 512 seeded random rows."""
    cfg = synthetic.CONFIGS[name]
    inp = synthetic.make_layer_inputs(cfg, device="cpu")
    d = {k: v.to(DEV) for k, v in inp.items()}
    fwd = moe.moe_layer_forward(d["x"], d["topk_idx"], d["topk_probs"], d["W1"], d["W2"], cfg.P,
                                host_sync=True, save_for_backward=True)
    torch.cuda.synchronize()
    L = fwd.layout
    counts = L.tokens_per_expert.cpu().numpy()
    offs = L.offsets.cpu().numpy()
    rt = L.row_token.cpu().numpy()
    re = L.row_expert.cpu().numpy()
    nz = np.flatnonzero(counts)
    experts = {int(nz[np.argmax(counts[nz])]), int(nz[np.argmin(counts[nz])]), int(nz[0]), int(nz[-1])}
    rows = [r for e in experts for r in range(offs[e], offs[e] + counts[e])]
    rng = np.random.default_rng(0)
    valid_rows = np.flatnonzero(rt >= 0)
    rows = np.unique(np.concatenate([rows, rng.choice(valid_rows, 512, replace=False)]))
    xd = bits(fwd.x_disp)
    assert np.array_equal(xd[rows], bits(inp["x"])[rt[rows]])
    y, h, o = O.grouped_experts(xd, re, L.row_weight.cpu().numpy(), bits(inp["W1"]), bits(inp["W2"]),
                                cfg.I, rows=rows)
    assert_gemm_close(bits(fwd.h)[rows], h[rows], "h", intermediate=True)
    assert_gemm_close(bits(fwd.y)[rows], y[rows], "y")
    # combine at full size: bit-exact against the oracle on the GPU's y
    y_gpu = bits(fwd.y).copy()
    y_gpu[rt < 0] = 0
    tr = L.token_row.cpu().numpy().reshape(cfg.T, cfg.K)
    assert np.array_equal(bits(fwd.out), O.combine(y_gpu, tr))


def test_forward_is_deterministic(moe):
    T, H, E, K, I, P = 700, 512, 16, 4, 256, 8
    a = _experts_case(moe, T, H, E, K, I, P, seed=5)[-1]
    b = _experts_case(moe, T, H, E, K, I, P, seed=5)[-1]
    for name in ("row_token", "row_expert", "row_weight", "token_row", "offsets"):
        assert torch.equal(getattr(a.layout, name), getattr(b.layout, name)), name
    for name in ("x_disp", "out"):
        assert torch.equal(getattr(a, name).view(torch.int16), getattr(b, name).view(torch.int16)), name
    # h and y are written on the valid rows only (pad / spare rows are skipped)
    valid = a.layout.row_token >= 0
    for name in ("h", "y"):
        assert torch.equal(getattr(a, name)[valid].view(torch.int16),
                           getattr(b, name)[valid].view(torch.int16)), name


# ----------------------------------------------------------------- backward a7, a8, a10, multihot

@pytest.mark.parametrize("T,H,E,K,I,P,drop", [(64, 256, 8, 2, 128, 16, 0.0),
                                              (333, 512, 12, 4, 128, 8, 0.15)])
def test_backward_gathers(moe, T, H, E, K, I, P, drop):
    idx, p, x, W1, W2, C, fwd = _experts_case(moe, T, H, E, K, I, P, seed=T, drop=drop)
    L = fwd.layout
    grad_out = torch.randn(T, H, generator=torch.Generator().manual_seed(1)).to(torch.bfloat16)
    grad_y, grad_w = moe.moe_combine_backward(grad_out.to(DEV), L, o_save=fwd.o)
    torch.cuda.synchronize()
    rt = L.row_token.cpu().numpy()
    re = L.row_expert.cpu().numpy()
    # a7 bit-exact
    assert np.array_equal(bits(grad_y), O.combine_backward(bits(grad_out), rt))
    # a8 against the fp64 oracle on the same o_save
    gw_ref = O.routing_weight_grad(bits(grad_y), bits(fwd.o), re, E).astype(np.float64)
    gw = grad_w.cpu().numpy().astype(np.float64)
    # valid rows within the fp32 bound; on pad and spare rows the weight
    # gradient is exactly 0 (the experts never write o there, so o may hold
    # anything and is not read)
    v = rt >= 0
    scale = np.abs(O.bf16_bits_to_f64(bits(grad_y)[v]) * O.bf16_bits_to_f64(bits(fwd.o)[v])).sum(axis=1)
    assert np.all(np.abs(gw[v] - gw_ref[v]) <= 1e-5 * scale + 1e-30)
    assert np.all(gw[~v] == 0)
    # a10 (+scatter) bit-exact given the same grad_x_disp and grad_w
    gxd = torch.randn(C, H, generator=torch.Generator().manual_seed(2)).to(torch.bfloat16)
    gxd_np = bits(gxd)
    grad_x, grad_probs = moe.moe_dispatch_backward(gxd.to(DEV), L, grad_w=grad_w)
    torch.cuda.synchronize()
    tr = L.token_row.cpu().numpy().reshape(T, K)
    gx_ref, gp_ref = O.dispatch_backward(gxd_np, tr, grad_w.cpu().numpy(), rt, re, E)
    assert np.array_equal(bits(grad_x), gx_ref)
    assert np.array_equal(grad_probs.cpu().numpy(), gp_ref)
    # multihot backward bit-exact
    g_topk = moe.moe_route_to_multihot_backward(grad_probs, idx.to(DEV), fwd.winner_slot)
    ref = O.route_to_multihot_backward(gp_ref, idx.numpy(), fwd.winner_slot.cpu().numpy())
    assert np.array_equal(g_topk.cpu().numpy(), ref)


# ----------------------------------------------------------------- sync-free capture

@pytest.mark.parametrize("T", [1, 256, 1024])
def test_sync_free_graph_replay_matches_eager(moe, T):
    """The decode path: worst-case buffers, no host sync, captured once in a
    CUDA graph and replayed on new inputs; replay == eager, bit for bit."""
    cfg = synthetic.CONFIGS[f"decode_{T}"]
    E, K, H, I, P = cfg.E, cfg.K, cfg.H, cfg.I, cfg.P
    W1, W2 = synthetic.make_weights(E, H, I, cfg.seed, device=DEV)
    C = O.worst_case_capacity(T, E, K, P)
    L = moe.Layout(T, E, K, P, C, device=DEV)
    s_x = torch.zeros(T, H, dtype=torch.bfloat16, device=DEV)
    s_idx = torch.zeros(T, K, dtype=torch.int64, device=DEV)
    s_p = torch.zeros(T, K, dtype=torch.float32, device=DEV)
    bufs = {"h": torch.empty(C, I, dtype=torch.bfloat16, device=DEV),
            "y": torch.empty(C, H, dtype=torch.bfloat16, device=DEV)}
    x_disp = torch.empty(C, H, dtype=torch.bfloat16, device=DEV)
    out = torch.empty(T, H, dtype=torch.bfloat16, device=DEV)

    def step():
        rmap, probs, _ = moe.moe_route_to_multihot(s_idx, s_p, E, L.status)
        moe.moe_dispatch(s_x, rmap, probs, L, host_sync=False, x_disp=x_disp)
        moe.moe_grouped_experts(x_disp, L, W1, W2, out=bufs)
        moe.moe_combine(bufs["y"], L, out=out)

    inputs = []
    for k in range(3):
        i = synthetic.make_layer_inputs(cfg, device=DEV, with_weights=False, layer=k)
        inputs.append(i)
    # eager references (also the warm-up before capture)
    eager = []
    side = torch.cuda.Stream()
    side.wait_stream(torch.cuda.current_stream())
    with torch.cuda.stream(side):
        for i in inputs:
            s_x.copy_(i["x"]); s_idx.copy_(i["topk_idx"]); s_p.copy_(i["topk_probs"])
            step()
            eager.append(out.clone())
    torch.cuda.current_stream().wait_stream(side)
    g = torch.cuda.CUDAGraph()
    with torch.cuda.graph(g):
        step()
    for i, ref in zip(reversed(inputs), reversed(eager)):
        s_x.copy_(i["x"]); s_idx.copy_(i["topk_idx"]); s_p.copy_(i["topk_probs"])
        g.replay()
        torch.cuda.synchronize()
        assert torch.equal(out.view(torch.int16), ref.view(torch.int16))
    assert int(L.status.item()) == 0
    # and the replayed output matches the oracle's layer (spot check on the last input)
    i = inputs[0]
    ref = O.layer_forward(bits(i["x"]), i["topk_idx"].cpu().numpy(), i["topk_probs"].cpu().numpy(),
                          bits(W1), bits(W2), I, P, capacity=C)
    assert_gemm_close(bits(out), ref["out"], "decode out")
