"""The bounds-checked build (libmoe_bounds.so, MOE_DEBUG_BOUNDS) on the GPU.

Its kernels check every index they derive from the layout (placed rows, rows
read back from token_row, epilogue rows, experts) against the buffer before
the access.  The whole layer -- forward and backward, host-synced and
sync-free, the fused and the one-CTA dispatch, single-CTA and CTA-pair
GEMM tiles, the CUDA-core decode experts -- runs through the binding switched
onto that build: no check may fail (no MOE_DEVERR_BOUNDS, nor any other
status bit), and every result must equal the normal build's bit for bit.
"""
import pytest
import torch

from tests._util import random_routing

pytestmark = pytest.mark.gpu
DEV = "cuda"


@pytest.fixture(scope="module")
def libs():
    assert torch.cuda.is_available(), "GPU tests need a GPU"
    import combine_topk_multihot_gb300 as m
    from combine_topk_multihot_gb300 import build
    checked = m._native.load(build.build(variant="bounds"))
    assert checked.moe_build_flags() == m._native.MOE_BUILD_BOUNDS_CHECKS
    return m, m._native.lib, checked


def _layer(m, x, idx, p, W1, W2, g, P, host_sync):
    fwd = m.moe_layer_forward(x, idx, p, W1, W2, P, host_sync=host_sync, save_for_backward=True)
    go, gw = m.moe_combine_backward(g, fwd.layout, o_save=fwd.o, scaled=True)
    gxd, dW1, dW2 = m.moe_grouped_experts_backward(go, fwd.x_disp, fwd.h, fwd.gu, fwd.layout, W1, W2,
                                                   scaled=True)
    gx, gp = m.moe_dispatch_backward(gxd, fwd.layout, gw)
    gt = m.moe_route_to_multihot_backward(gp, idx, fwd.winner_slot)
    inf = m.moe_grouped_experts(fwd.x_disp, fwd.layout, W1, W2)        # inference: no saves
    torch.cuda.synchronize()
    valid = fwd.layout.row_token >= 0
    return {"status": int(fwd.layout.status.item()), "out": fwd.out, "x_disp": fwd.x_disp,
            "row_token": fwd.layout.row_token, "y": fwd.y[valid], "y_inf": inf["y"][valid],
            "grad_x": gx, "grad_topk": gt, "dW1": dW1, "dW2": dW2}


@pytest.mark.parametrize("T,H,E,K,I,P,host_sync", [
    (64, 256, 8, 2, 128, 16, True),      # one-CTA layout
    (300, 512, 8, 2, 256, 16, False),    # cooperative dispatch kernel, ragged groups
    (2000, 512, 40, 4, 512, 128, True),  # CTA-pair GEMM tiles, forward and backward
    (1, 2048, 128, 8, 768, 1, False),    # decode: the layout kernel copies the rows, CUDA-core experts
])
def test_checked_build_reports_nothing_and_matches(libs, monkeypatch, T, H, E, K, I, P, host_sync):
    m, normal, checked = libs
    idx, p = random_routing(T, E, K, seed=3 * T + E, drop=0.1, dup=0.1)
    gen = torch.Generator().manual_seed(T + 1)
    bf = torch.bfloat16
    x = torch.randn(T, H, generator=gen).to(bf).to(DEV)
    W1 = (torch.randn(E, 2 * I, H, generator=gen) * 0.02).to(bf).to(DEV)
    W2 = (torch.randn(E, H, I, generator=gen) * 0.02).to(bf).to(DEV)
    g = torch.randn(T, H, generator=gen).to(bf).to(DEV)
    idx, p = idx.to(DEV), p.to(DEV)
    with monkeypatch.context() as mp:
        mp.setattr(m._native, "lib", checked)
        a = _layer(m, x, idx, p, W1, W2, g, P, host_sync)
    b = _layer(m, x, idx, p, W1, W2, g, P, host_sync)
    assert a["status"] == 0, f"device status {a['status']} (MOE_DEVERR_BOUNDS = {m._native.MOE_DEVERR_BOUNDS})"
    assert b["status"] == 0
    for k in ("out", "x_disp", "row_token", "y", "y_inf", "grad_x", "grad_topk", "dW1", "dW2"):
        u, v = a[k], b[k]
        if u.dtype == torch.bfloat16:
            u, v = u.view(torch.int16), v.view(torch.int16)
        assert torch.equal(u, v), k
