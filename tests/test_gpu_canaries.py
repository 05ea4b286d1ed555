"""Out-of-bounds writes, caught with guard regions (the race and bounds checks
that stand in for a memory sanitizer on the GPU).

Every buffer a call writes -- layout arrays, rows, expert outputs, gradients,
workspaces -- is the middle of a larger allocation whose 4 KiB on either side
hold a canary byte.  One whole layer runs through the C ABI (multihot,
dispatch in both modes and from the top-k, both expert forwards, combine,
both combine backwards, both expert backwards, dispatch and multihot
backward, the FP8 dispatch (from the multihot map and from the top-k) and
gate/up GEMM, the gathered gate/up GEMM, the router), then every canary must be intact and the status word clear.  The
shapes cover the one-CTA and cooperative layouts, one-CTA and CTA-pair GEMM
tiles, 128-row tiles with ragged groups, and the CUDA-core decode experts.
"""
import ctypes

import pytest
import torch

from tests._util import random_routing

pytestmark = pytest.mark.gpu
DEV = "cuda"
GUARD = 4096
CANARY = 0xA5


@pytest.fixture(scope="module")
def moe():
    assert torch.cuda.is_available(), "GPU tests need a GPU"
    import combine_topk_multihot_gb300 as m
    return m


class Guarded:
    """Allocations with canary-filled guard regions on both sides."""

    def __init__(self):
        self.bufs = []

    def __call__(self, shape, dtype, fill=None):
        shape = tuple(shape) if isinstance(shape, (tuple, list)) else (shape,)
        n = int(torch.Size(shape).numel()) * torch.empty((), dtype=dtype).element_size()
        buf = torch.full((GUARD + max(n, 0) + GUARD,), CANARY, dtype=torch.uint8, device=DEV)
        view = buf[GUARD:GUARD + n].view(dtype).view(shape)
        if fill is not None:
            view.fill_(fill)
        self.bufs.append((buf, n))
        return view

    def check(self):
        for i, (buf, n) in enumerate(self.bufs):
            assert bool((buf[:GUARD] == CANARY).all()), f"buffer {i}: write before its start"
            assert bool((buf[GUARD + n:] == CANARY).all()), f"buffer {i}: write past its end"


def _p(t):
    return ctypes.c_void_p(t.data_ptr()) if t is not None and t.numel() else None


def _layout(moe, g, T, E, K, P, C):
    N = moe._native
    i32 = torch.int32
    tensors = (g(E, i32), g(E + 1, i32), g(2, i32), g(C, i32), g(C, i32), g(C, torch.float32),
               g(T * K, i32), g(1, i32, fill=0))
    nbytes = ctypes.c_size_t(0)
    assert N.lib.moe_layout_workspace_bytes(T, E, ctypes.byref(nbytes)) == 0
    ws = g(nbytes.value, torch.uint8)
    return moe.Layout.from_tensors(T, E, K, P, tensors, workspace=ws)


@pytest.mark.parametrize("T,H,E,K,I,P", [
    (64, 256, 8, 2, 128, 16),       # one-CTA layout, 128-column tiles
    (300, 512, 8, 2, 256, 16),      # cooperative layout, ragged groups
    (2000, 512, 40, 4, 512, 128),   # CTA-pair GEMM tiles forward and backward
    (1, 2048, 128, 8, 768, 1),      # decode: one-kernel dispatch, CUDA-core experts
])
def test_no_write_outside_any_output(moe, T, H, E, K, I, P):
    N = moe._native
    st = lambda: ctypes.c_void_p(torch.cuda.current_stream().cuda_stream)
    bf = torch.bfloat16
    g = Guarded()
    idx, p = random_routing(T, E, K, seed=T + E, drop=0.1, dup=0.1)
    gen = torch.Generator().manual_seed(T)
    x = torch.randn(T, H, generator=gen).to(bf).to(DEV)
    W1 = (torch.randn(E, 2 * I, H, generator=gen) * 0.02).to(bf).to(DEV)
    W2 = (torch.randn(E, H, I, generator=gen) * 0.02).to(bf).to(DEV)
    gout = torch.randn(T, H, generator=gen).to(bf).to(DEV)
    idx, p = idx.to(DEV), p.to(DEV)
    C = moe.worst_case_rows(T, E, K, P)

    # a1: multihot; a2-a4 host-synced and sync-free; a1-a4 from the top-k
    rmap, probs, win = g((T, E), torch.uint8), g((T, E), torch.float32), g((T, E), torch.int8)
    L0 = _layout(moe, g, T, E, K, P, C)
    assert N.lib.moe_route_to_multihot(_p(idx), _p(p), T, K, E, _p(rmap), _p(probs), _p(win),
                                       _p(L0.status), st()) == 0
    rows = (ctypes.c_int64 * 2)()
    xd0 = g((C, H), bf)
    assert N.lib.moe_dispatch(_p(x), _p(rmap), _p(probs), H, L0.ref, _p(xd0), rows, st()) == 0
    R = rows[0]
    Lh = _layout(moe, g, T, E, K, P, R)   # exactly R rows, host-synced
    xdh = g((R, H), bf)
    assert N.lib.moe_dispatch(_p(x), _p(rmap), _p(probs), H, Lh.ref, _p(xdh), rows, st()) == 0
    L = _layout(moe, g, T, E, K, P, C)
    xd = g((C, H), bf)
    m2 = g((T, E), torch.uint8), g((T, E), torch.float32), g((T, E), torch.int8)
    assert N.lib.moe_dispatch_topk(_p(x), _p(idx), _p(p), H, L.ref, _p(m2[0]), _p(m2[1]), _p(m2[2]),
                                   _p(xd), None, st()) == 0
    Ll = _layout(moe, g, T, E, K, P, C)
    assert N.lib.moe_dispatch_layout(_p(rmap), _p(probs), Ll.ref, None, st()) == 0

    # a5 training (saves) and inference; the gathered gate/up GEMM; FP8
    h, y, o, gu = g((C, I), bf), g((C, H), bf), g((C, H), bf), g((C, 2 * I), bf)
    assert N.lib.moe_grouped_experts(_p(xd), L.ref, H, I, _p(W1), _p(W2), _p(h), _p(y), _p(o), _p(gu),
                                     st()) == 0
    h2, y2 = g((C, I), bf), g((C, H), bf)
    assert N.lib.moe_grouped_experts(_p(xd), L.ref, H, I, _p(W1), _p(W2), _p(h2), _p(y2), None, None,
                                     st()) == 0
    h3, y3 = g((C, I), bf), g((C, H), bf)
    assert N.lib.moe_grouped_experts_gather(_p(x), Ll.ref, H, I, _p(W1), _p(W2), _p(h3), _p(y3), None, None,
                                            st()) == 0
    w1q, w1s = g((E, 2 * I, H), torch.uint8), g((E * 2 * I,), torch.float32)
    assert N.lib.moe_quantize_fp8(_p(W1), E * 2 * I, H, _p(w1q), _p(w1s), st()) == 0
    Lq = _layout(moe, g, T, E, K, P, C)
    xq, xs = g((C, H), torch.uint8), g((C,), torch.float32)
    assert N.lib.moe_dispatch_fp8(_p(x), _p(rmap), _p(probs), H, Lq.ref, _p(xq), _p(xs), None, st()) == 0
    Lq2 = _layout(moe, g, T, E, K, P, C)
    xq2, xs2 = g((C, H), torch.uint8), g((C,), torch.float32)
    m3 = g((T, E), torch.uint8), g((T, E), torch.float32), g((T, E), torch.int8)
    assert N.lib.moe_dispatch_topk_fp8(_p(x), _p(idx), _p(p), H, Lq2.ref, _p(m3[0]), _p(m3[1]), _p(m3[2]),
                                       _p(xq2), _p(xs2), rows, st()) == 0
    h4, y4 = g((C, I), bf), g((C, H), bf)
    assert N.lib.moe_grouped_experts_fp8(_p(xq), _p(xs), Lq.ref, H, I, _p(w1q), _p(w1s), _p(W2), _p(h4),
                                         _p(y4), st()) == 0

    # a6; a7 + a8 both ways; a9 both ways; a10; multihot backward
    out = g((T, H), bf)
    assert N.lib.moe_combine(_p(y), L.ref, H, _p(out), st()) == 0
    gy, gw = g((C, H), bf), g((C,), torch.float32)
    assert N.lib.moe_combine_backward(_p(gout), _p(o), L.ref, H, _p(gy), _p(gw), st()) == 0
    go, gw2 = g((C, H), bf), g((C,), torch.float32)
    assert N.lib.moe_combine_backward_scaled(_p(gout), _p(o), L.ref, H, _p(go), _p(gw2), st()) == 0
    nb = ctypes.c_size_t(0)
    assert N.lib.moe_experts_backward_workspace_bytes(C, H, I, ctypes.byref(nb)) == 0
    for grad, fn in ((gy, N.lib.moe_grouped_experts_backward), (go, N.lib.moe_grouped_experts_backward_scaled)):
        gxd, dW1, dW2 = g((C, H), bf), g((E, 2 * I, H), torch.float32), g((E, H, I), torch.float32)
        ws = g(nb.value, torch.uint8)
        assert fn(_p(grad), _p(xd), _p(h), _p(gu), L.ref, H, I, _p(W1), _p(W2), _p(gxd), _p(dW1), _p(dW2),
                  _p(ws), st()) == 0
    gx, gp = g((T, H), bf), g((T, E), torch.float32)
    assert N.lib.moe_dispatch_backward(_p(gxd), _p(gw), L.ref, H, _p(gx), _p(gp), st()) == 0
    gt = g((T, K), torch.float32)
    assert N.lib.moe_route_to_multihot_backward(_p(gp), _p(idx), _p(m2[2]), T, K, E, _p(gt), st()) == 0

    # r0: the router with its multihot outputs, and its backward
    logits = torch.randn(T, E, generator=gen).to(DEV)
    ri, rp = g((T, K), torch.int64), g((T, K), torch.float32)
    rm = g((T, E), torch.uint8), g((T, E), torch.float32), g((T, E), torch.int8)
    assert N.lib.moe_router_topk(_p(logits), T, E, K, _p(ri), _p(rp), _p(rm[0]), _p(rm[1]), _p(rm[2]),
                                 st()) == 0
    gl = g((T, E), torch.float32)
    assert N.lib.moe_router_topk_backward(_p(gt), _p(rp), _p(ri), T, E, K, _p(gl), st()) == 0

    torch.cuda.synchronize()
    for lay in (L0, Lh, L, Ll, Lq):
        assert int(lay.status.item()) == 0
    g.check()
    assert torch.equal(L.row_token, L0.row_token) and torch.equal(xd.view(torch.int16), xd0.view(torch.int16))
