"""The dispatch fused into the gate/up GEMM (moe_dispatch_layout +
moe_grouped_experts_gather): the GEMM's producer gathers A rows from the tokens
by row_token instead of reading x_disp.

The A tile it builds in shared memory is the one the TMA load of x_disp builds,
so every output must equal the materialised path's bit for bit -- for the
256- and 64-column tiles, the CUDA-core path (T <= 4), padded groups, drops,
both modes, and with the operands saved for a backward.  The layout alone must
equal moe_dispatch's.  One case also goes to the oracle end to end.
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


def _both(moe, x, idx, p, W1, W2, E, K, P, host_sync, save):
    T = x.shape[0]
    C = O.worst_case_capacity(T, E, K, P)
    st1 = torch.zeros(1, dtype=torch.int32, device=DEV)
    st2 = torch.zeros(1, dtype=torch.int32, device=DEV)
    rmap, probs, _ = moe.moe_route_to_multihot(idx.to(DEV), p.to(DEV), E, st1)
    L1 = moe.Layout(T, E, K, P, C, device=DEV, status=st1)
    L2 = moe.Layout(T, E, K, P, C, device=DEV, status=st2)
    x_disp, rows1 = moe.moe_dispatch(x.to(DEV), rmap, probs, L1, host_sync=host_sync)
    rows2 = moe.moe_dispatch_layout(rmap, probs, L2, host_sync=host_sync)
    ref = moe.moe_grouped_experts(x_disp, L1, W1.to(DEV), W2.to(DEV), save_o=save, save_gu=save)
    got = moe.moe_grouped_experts_gather(x.to(DEV), L2, W1.to(DEV), W2.to(DEV), save_o=save, save_gu=save)
    torch.cuda.synchronize()
    assert rows1 == rows2
    for f in ("tokens_per_expert", "offsets", "totals", "row_token", "row_expert", "row_weight", "token_row"):
        assert torch.equal(getattr(L1, f), getattr(L2, f)), f
    assert int(st1.item()) == 0 and int(st2.item()) == 0
    return L1, ref, got


CASES = [  # T, H, E, K, I, P, drop
    (64, 256, 64, 4, 384, 16, 0.0),     # 256-column tiles
    (300, 512, 8, 2, 256, 16, 0.1),     # 64-column tiles, drops
    (2000, 512, 40, 4, 512, 1, 0.0),    # 256-column tiles, two 128-row tiles per expert
    (260, 768, 12, 3, 128, 128, 0.2),   # groups padded to 128
    (3, 256, 8, 2, 128, 16, 0.0),       # CUDA-core path
    (1, 2048, 128, 8, 768, 1, 0.0),     # decode T = 1
]


@pytest.mark.parametrize("host_sync", [True, False])
@pytest.mark.parametrize("T,H,E,K,I,P,drop", CASES)
def test_gather_equals_materialised(moe, T, H, E, K, I, P, drop, host_sync):
    idx, p = random_routing(T, E, K, seed=T + 5 * H, drop=drop)
    g = torch.Generator().manual_seed(T + H)
    x = torch.randn(T, H, generator=g).to(torch.bfloat16)
    W1 = (torch.randn(E, 2 * I, H, generator=g) * 0.02).to(torch.bfloat16)
    W2 = (torch.randn(E, H, I, generator=g) * 0.02).to(torch.bfloat16)
    L, ref, got = _both(moe, x, idx, p, W1, W2, E, K, P, host_sync, save=False)
    valid = L.row_token >= 0
    for k in ("h", "y"):
        assert torch.equal(ref[k][valid].view(torch.int16), got[k][valid].view(torch.int16)), k


@pytest.mark.parametrize("T,H,E,K,I,P,drop", [CASES[1], CASES[3]])
def test_gather_with_saved_operands(moe, T, H, E, K, I, P, drop):
    """Training outputs (o, gu, pad rows written) are the same too."""
    idx, p = random_routing(T, E, K, seed=2 * T + H, drop=drop)
    g = torch.Generator().manual_seed(T)
    x = torch.randn(T, H, generator=g).to(torch.bfloat16)
    W1 = (torch.randn(E, 2 * I, H, generator=g) * 0.02).to(torch.bfloat16)
    W2 = (torch.randn(E, H, I, generator=g) * 0.02).to(torch.bfloat16)
    L, ref, got = _both(moe, x, idx, p, W1, W2, E, K, P, True, save=True)
    R = int(L.totals[0].item())   # valid and pad rows (spare rows are never written)
    for k in ("h", "y", "o", "gu"):
        assert torch.equal(ref[k][:R].view(torch.int16), got[k][:R].view(torch.int16)), k


def test_gather_matches_oracle(moe):
    T, H, E, K, I, P = 300, 512, 8, 2, 256, 16
    idx, p = random_routing(T, E, K, seed=77, drop=0.1)
    g = torch.Generator().manual_seed(77)
    x = torch.randn(T, H, generator=g).to(torch.bfloat16)
    W1 = (torch.randn(E, 2 * I, H, generator=g) * 0.02).to(torch.bfloat16)
    W2 = (torch.randn(E, H, I, generator=g) * 0.02).to(torch.bfloat16)
    C = O.worst_case_capacity(T, E, K, P)
    st = torch.zeros(1, dtype=torch.int32, device=DEV)
    rmap, probs, _ = moe.moe_route_to_multihot(idx.to(DEV), p.to(DEV), E, st)
    L = moe.Layout(T, E, K, P, C, device=DEV, status=st)
    moe.moe_dispatch_layout(rmap, probs, L)
    r = moe.moe_grouped_experts_gather(x.to(DEV), L, W1.to(DEV), W2.to(DEV))
    out = moe.moe_combine(r["y"], L)
    torch.cuda.synchronize()
    ref = O.layer_forward(bits(x), idx.numpy(), p.numpy(), bits(W1), bits(W2), I, P, capacity=C)
    valid = ref["layout"]["row_token"] >= 0
    assert_gemm_close(bits(r["h"])[valid], ref["h"][valid], "h", intermediate=True)
    assert_gemm_close(bits(r["y"])[valid], ref["y"][valid], "y")
    assert_gemm_close(bits(out), ref["out"], "out")


def test_gather_full_size_qwen(moe):
    """The Qwen3-30B-A3B layer (T 4096): every valid row equals the materialised path."""
    cfg = synthetic.CONFIGS["qwen3_30b_a3b"]
    d = synthetic.make_layer_inputs(cfg)
    L, ref, got = _both(moe, d["x"], d["topk_idx"], d["topk_probs"], d["W1"], d["W2"], cfg.E, cfg.K,
                        cfg.P, True, save=False)
    valid = L.row_token >= 0
    for k in ("h", "y"):
        assert torch.equal(ref[k][valid].view(torch.int16), got[k][valid].view(torch.int16)), k
