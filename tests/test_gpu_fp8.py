"""GPU parity of the FP8 path against the FP8 oracle.

* rowwise e4m3 quantization (moe_quantize_fp8) and the FP8 dispatch
  (moe_dispatch_fp8, host-synced and sync-free): codes and scales bit for bit
  -- the amax and the division are fp32 on both sides and the rounding is
  round-to-nearest-even with saturation, so every code is determined;
* the e4m3 gate/up GEMM (moe_grouped_experts_fp8): h within the
  intermediate tolerance and y within the GEMM tolerance of the fp64 oracle,
  which takes its own layout, FP8 dispatch and W1 quantization from the same
  bf16 inputs, for the three tile shapes (256-column tiles, 64-column tiles,
  64-column tiles with a 32-row A slot) and the full Qwen layer (sampled).
"""
import numpy as np
import pytest
import torch

import oracle as O
import synthetic
from tests._util import assert_gemm_close, bits, random_routing

pytestmark = pytest.mark.gpu
DEV = "cuda"


@pytest.fixture(scope="module")
def moe():
    assert torch.cuda.is_available(), "GPU tests need a GPU"
    import combine_topk_multihot_gb300 as m
    return m


@pytest.mark.parametrize("rows,cols,scale", [(1, 256, 1.0), (333, 512, 1e-3), (64, 4096, 300.0)])
def test_quantize_rows_bit_exact(moe, rows, cols, scale):
    g = torch.Generator().manual_seed(rows + cols)
    src = (torch.randn(rows, cols, generator=g) * scale).to(torch.bfloat16)
    src[0, :7] = 0.0
    if rows > 2:
        src[2] = 0.0                                   # an all-zero row: scale 1
    codes, scales = moe.moe_quantize_fp8(src.to(DEV))
    torch.cuda.synchronize()
    ref_c, ref_s = O.quantize_rows(src.float().numpy())
    assert np.array_equal(codes.cpu().numpy(), ref_c)
    assert np.array_equal(scales.cpu().numpy(), ref_s)


@pytest.mark.parametrize("host_sync", [True, False])
@pytest.mark.parametrize("T,H,E,K,P,drop", [
    (64, 256, 8, 2, 16, 0.0),      # two chunks: the layout kernel, then the FP8 row kernel
    (513, 512, 32, 8, 128, 0.1),   # 17 chunks: the fused cooperative dispatch writes the e4m3 rows
    (600, 4096, 16, 4, 64, 0.05),  # fused, each row in two 2 KiB pieces of codes
    (1, 2048, 128, 8, 1, 0.0),
])
def test_dispatch_fp8_bit_exact(moe, T, H, E, K, P, drop, host_sync):
    idx, p = random_routing(T, E, K, seed=T + H, drop=drop)
    x = torch.randn(T, H, generator=torch.Generator().manual_seed(T)).to(torch.bfloat16)
    C = O.worst_case_capacity(T, E, K, P)
    status = torch.zeros(1, dtype=torch.int32, device=DEV)
    rmap, probs, _ = moe.moe_route_to_multihot(idx.to(DEV), p.to(DEV), E, status)
    L = moe.Layout(T, E, K, P, C, device=DEV, status=status)
    q, sc, rows = moe.moe_dispatch_fp8(x.to(DEV), rmap, probs, L, host_sync=host_sync)
    torch.cuda.synchronize()
    rm, pr, _ = O.route_to_multihot(idx.numpy(), p.numpy(), E)
    Lr = O.build_layout(rm, pr, K, P, C)
    assert np.array_equal(L.row_token.cpu().numpy(), Lr["row_token"])
    assert np.array_equal(L.row_expert.cpu().numpy(), Lr["row_expert"])
    ref_q, ref_s = O.dispatch_fp8(bits(x), Lr["row_token"])
    assert np.array_equal(q.cpu().numpy(), ref_q)
    assert np.array_equal(sc.cpu().numpy(), ref_s)
    assert int(status.item()) == 0


@pytest.mark.parametrize("host_sync", [True, False])
@pytest.mark.parametrize("T,H,E,K,P,drop,dup", [
    (64, 256, 8, 2, 16, 0.0, 0.0),       # two chunks: the multihot kernel, the layout, the FP8 rows
    (256, 512, 128, 8, 1, 0.05, 0.05),   # 8 chunks: the multihot kernel, then the barrier-free layout
    (513, 512, 32, 8, 128, 0.1, 0.05),   # one cooperative kernel from the top-k, drops and duplicates
    (600, 4096, 16, 4, 64, 0.05, 0.0),   # the same, two 2 KiB pieces of codes per row
    (333, 512, 64, 40, 2, 0.2, 0.2),     # K > 32: slots in two registers per lane
    (700, 256, 1024, 4, 1, 0.0, 0.0),    # the largest E
    (40000, 256, 128, 8, 4, 0.05, 0.0),  # more chunks than resident CTAs
    (0, 256, 8, 2, 16, 0.0, 0.0),        # no tokens: spare rows only
])
def test_dispatch_topk_fp8_bit_exact(moe, T, H, E, K, P, drop, dup, host_sync):
    """moe_dispatch_topk_fp8 = moe_route_to_multihot + moe_dispatch_fp8: the
    multihot outputs, the layout, the codes and the scales all equal the
    oracle's, with every output buffer poisoned first so that each entry must
    be written."""
    idx, p = random_routing(T, E, K, seed=T + H + 1, drop=drop, dup=dup)
    x = torch.randn(T, H, generator=torch.Generator().manual_seed(T + 1)).to(torch.bfloat16)
    C = O.worst_case_capacity(T, E, K, P)
    status = torch.zeros(1, dtype=torch.int32, device=DEV)
    L = moe.Layout(T, E, K, P, C, device=DEV, status=status)
    L.row_token.fill_(12345)
    L.row_expert.fill_(-7)
    L.row_weight.fill_(float("nan"))
    L.token_row.fill_(999)
    q = torch.full((C, H), 0x7F, dtype=torch.uint8, device=DEV)
    sc = torch.full((C,), float("nan"), dtype=torch.float32, device=DEV)
    mh = (torch.full((T, E), 7, dtype=torch.uint8, device=DEV),
          torch.full((T, E), float("nan"), dtype=torch.float32, device=DEV),
          torch.full((T, E), 5, dtype=torch.int8, device=DEV))
    q, sc, (rmap, probs, win), rows = moe.moe_dispatch_topk_fp8(x.to(DEV), idx.to(DEV), p.to(DEV), L,
                                                                host_sync=host_sync, out=(q, sc), multihot=mh)
    torch.cuda.synchronize()
    assert int(status.item()) == 0
    rm, pr, wn = O.route_to_multihot(idx.numpy(), p.numpy(), E)
    assert np.array_equal(rmap.cpu().numpy(), rm)
    assert np.array_equal(probs.cpu().numpy(), pr)
    assert np.array_equal(win.cpu().numpy(), wn)
    Lr = O.build_layout(rm, pr, K, P, C)
    for k in ("row_token", "row_expert", "token_row"):
        assert np.array_equal(getattr(L, k).cpu().numpy().reshape(np.shape(Lr[k])), Lr[k]), k
    assert np.array_equal(L.row_weight.cpu().numpy(), Lr["row_weight"])
    if host_sync:
        assert rows == (Lr["rows_used"], Lr["rows_valid"])
    ref_q, ref_s = O.dispatch_fp8(bits(x), Lr["row_token"])
    assert np.array_equal(q.cpu().numpy(), ref_q)
    assert np.array_equal(sc.cpu().numpy(), ref_s)


def _run_fp8_experts(moe, x, idx, p, W1, W2, E, K, P, host_sync=True):
    """The FP8 path on the GPU: multihot, FP8 dispatch, W1 quantization, experts."""
    T, H = x.shape
    C = O.worst_case_capacity(T, E, K, P)
    status = torch.zeros(1, dtype=torch.int32, device=DEV)
    rmap, probs, _ = moe.moe_route_to_multihot(idx.to(DEV), p.to(DEV), E, status)
    L = moe.Layout(T, E, K, P, C, device=DEV, status=status)
    q, sc, _ = moe.moe_dispatch_fp8(x.to(DEV), rmap, probs, L, host_sync=host_sync)
    W1q, W1s = moe.moe_quantize_fp8(W1.to(DEV))
    out = moe.moe_grouped_experts_fp8(q, sc, L, W1q, W1s, W2.to(DEV))
    torch.cuda.synchronize()
    assert int(status.item()) == 0
    return L, out


def _check_fp8_experts(L, out, x, idx, p, W1, W2, E, K, P, I, experts=None, rows=None):
    """Against the oracle on the oracle's own inputs: its layout (which must
    equal the GPU's), its FP8 dispatch of x and its quantization of W1."""
    T = x.shape[0]
    C = O.worst_case_capacity(T, E, K, P)
    rm, pr, _ = O.route_to_multihot(idx.numpy(), p.numpy(), E)
    Lr = O.build_layout(rm, pr, K, P, C)
    assert np.array_equal(L.row_token.cpu().numpy(), Lr["row_token"])
    q, sc = O.dispatch_fp8(bits(x), Lr["row_token"])
    todo = range(E) if experts is None else experts
    W1f = W1.float().numpy()
    quant = {e: O.quantize_rows(W1f[e]) for e in todo}
    qW1 = {e: c for e, (c, _) in quant.items()}
    sW1 = {e: s for e, (_, s) in quant.items()}
    y_ref, h_ref = O.grouped_experts_fp8(q, sc, Lr["row_expert"], Lr["row_weight"], qW1, sW1,
                                         bits(W2), I, experts=todo)
    if rows is None:
        rows = np.flatnonzero(Lr["row_token"] >= 0)
    assert_gemm_close(bits(out["h"])[rows], h_ref[rows], "fp8 h", intermediate=True)
    assert_gemm_close(bits(out["y"])[rows], y_ref[rows], "fp8 y")


@pytest.mark.parametrize("T,H,E,K,I,P", [
    (64, 256, 64, 4, 384, 16),      # 256-column tiles
    (300, 512, 8, 2, 256, 16),      # 64-column tiles, several 128-row tiles
    (5, 1024, 8, 4, 384, 1),        # 64-column tiles with a 32-row A slot
    (2000, 512, 40, 4, 512, 1),     # 256-column tiles, two 128-row tiles per expert
    (2304, 256, 256, 8, 128, 1),    # 256 experts: the per-expert tables take a pipeline stage
])
def test_experts_fp8_match_oracle(moe, T, H, E, K, I, P):
    seed = T + 7 * I
    idx, p = random_routing(T, E, K, seed=seed)
    g = torch.Generator().manual_seed(seed)
    x = torch.randn(T, H, generator=g).to(torch.bfloat16)
    W1 = (torch.randn(E, 2 * I, H, generator=g) * 0.02).to(torch.bfloat16)
    W2 = (torch.randn(E, H, I, generator=g) * 0.02).to(torch.bfloat16)
    L, out = _run_fp8_experts(moe, x, idx, p, W1, W2, E, K, P)
    _check_fp8_experts(L, out, x, idx, p, W1, W2, E, K, P, I)


def test_experts_fp8_full_size_qwen_sampled(moe):
    """The Qwen3-30B-A3B layer (T 4096, H 2048, E 128, top-8, I 768, P 128),
    host-synced: every row of four experts (the largest, the smallest and two
    others)."""
    cfg = synthetic.CONFIGS["qwen3_30b_a3b"]
    T, H, E, K, I, P = cfg.T, cfg.H, cfg.E, cfg.K, cfg.I, cfg.P
    d = synthetic.make_layer_inputs(cfg)
    L, out = _run_fp8_experts(moe, d["x"], d["topk_idx"], d["topk_probs"], d["W1"], d["W2"], E, K, P)
    counts = L.tokens_per_expert.cpu().numpy()
    offs = L.offsets.cpu().numpy()
    nz = np.flatnonzero(counts)
    experts = sorted({int(nz[np.argmax(counts[nz])]), int(nz[np.argmin(counts[nz])]), 5, 77})
    rows = np.concatenate([np.arange(offs[e], offs[e] + counts[e]) for e in experts])
    _check_fp8_experts(L, out, d["x"], d["topk_idx"], d["topk_probs"], d["W1"], d["W2"], E, K, P, I,
                       experts=experts, rows=rows)
