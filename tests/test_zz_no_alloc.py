"""moe_dispatch_static_scratch: the dispatch for callers that cannot allocate.

Callers such as an engine plugin that is handed only its inputs and outputs,
or a serving loop that may not call cudaMalloc, cannot provide the layout's
scratch buffer.  This entry point keeps that scratch in a static device array
inside the library.  The test calls it through the C ABI and checks that two
calls in a row (different routings, so the second call sees the first call's
leftover counters) give exactly what moe_dispatch gives with its own
caller-provided workspace: the layout and the dispatched rows are integer /
bit-copy results, so the tolerance is bit-exactness.

The sizes cover both kinds of layout launch: the cooperative one with grid
barriers (T = 1000, 333) and the barrier-free one of decode-sized layers,
with the row pass in the same kernel (T = 1) and without it (T = 200).  The
first call on a device, which looks up the array's address, is refused while
its stream is being captured; that is checked in a fresh process, where the
lookup has not happened yet.

This file is collected last on purpose and must also pass on its own.
"""
import ctypes
import os
import subprocess
import sys
import textwrap

import numpy as np
import pytest
import torch

pytestmark = pytest.mark.gpu

DEV = "cuda"


@pytest.fixture(scope="module")
def moe():
    assert torch.cuda.is_available(), "GPU tests need a GPU"
    import combine_topk_multihot_gb300 as m
    assert m._native.lib.moe_device_check() == 0, m._native.last_error()
    return m


def _routing(T, E, K, seed):
    g = torch.Generator().manual_seed(seed)
    logits = torch.randn(T, E, generator=g)
    p, idx = torch.topk(torch.softmax(logits, -1), K, dim=-1)
    idx[torch.rand(T, K, generator=g) < 0.05] = -1
    return idx.to(torch.int64), (p / p.sum(-1, keepdim=True)).to(torch.float32)


def _layout_tensors(L):
    return {k: getattr(L, k).clone() for k in ("tokens_per_expert", "offsets", "totals", "row_token",
                                               "row_expert", "row_weight", "token_row")}


@pytest.mark.parametrize("cases,P", [
    ([(1000, 11), (333, 12)], 16),     # cooperative layout, grid barriers
    ([(1, 13), (200, 14)], 1),         # barrier-free layout: with its row pass, then without
])
@pytest.mark.parametrize("host_sync", [True, False])
def test_static_scratch_dispatch_matches_dispatch_twice(moe, host_sync, cases, P):
    N = moe._native
    E, K, H = 64, 4, 256
    for T, seed in cases:                # two calls in a row, different sizes and routings
        idx, p = _routing(T, E, K, seed)
        x = torch.randn(T, H, generator=torch.Generator().manual_seed(seed)).to(torch.bfloat16).to(DEV)
        C = moe.worst_case_rows(T, E, K, P)
        status = torch.zeros(1, dtype=torch.int32, device=DEV)
        rmap, probs, _ = moe.moe_route_to_multihot(idx.to(DEV), p.to(DEV), E, status)

        # the existing entry point, with a caller-provided workspace
        ref_layout = moe.Layout(T, E, K, P, C, device=DEV, status=status)
        ref_x, ref_rows = moe.moe_dispatch(x, rmap, probs, ref_layout, host_sync=host_sync)

        # the static-scratch entry point, called through the C ABI with no workspace
        lay = moe.Layout(T, E, K, P, C, device=DEV, status=status)
        lay.c.workspace = None
        x_disp = torch.full((C, H), float("nan"), dtype=torch.bfloat16, device=DEV)
        rows = (ctypes.c_int64 * 2)(-1, -1) if host_sync else None
        st = N.lib.moe_dispatch_static_scratch(
            ctypes.c_void_p(x.data_ptr()), ctypes.c_void_p(rmap.data_ptr()),
            ctypes.c_void_p(probs.data_ptr()), H, ctypes.byref(lay.c),
            ctypes.c_void_p(x_disp.data_ptr()), rows,
            ctypes.c_void_p(torch.cuda.current_stream().cuda_stream))
        assert st == N.MOE_OK, N.last_error()
        torch.cuda.synchronize()

        assert int(status.item()) == 0
        if host_sync:
            assert (rows[0], rows[1]) == ref_rows
        got, ref = _layout_tensors(lay), _layout_tensors(ref_layout)
        for k in ref:
            assert torch.equal(got[k], ref[k]), k
        assert torch.equal(x_disp.view(torch.int16), ref_x.view(torch.int16))


def test_static_scratch_rejects_sizes_beyond_its_limit(moe):
    N = moe._native
    E = 128
    T = 32 * (N.MOE_STATIC_SCRATCH_INTS // E) + 1      # one chunk too many
    L = N.MoeLayout(T, E, 8, 1, T * 8)
    st = N.lib.moe_dispatch_static_scratch(None, None, None, 2048, ctypes.byref(L), None, None, None)
    assert st == N.MOE_ERR_UNSUPPORTED_SHAPE
    assert b"static scratch" in N.lib.moe_last_error()
    # the largest size that fits is accepted by the size check (it then fails
    # on the NULL buffers of this bare layout, not on the size)
    L = N.MoeLayout(32 * (N.MOE_STATIC_SCRATCH_INTS // E), E, 8, 1, 8)
    st = N.lib.moe_dispatch_static_scratch(None, None, None, 2048, ctypes.byref(L), None, None, None)
    assert st == N.MOE_ERR_INVALID_ARG


_CAPTURE_CHILD = textwrap.dedent("""
    import ctypes, sys
    import torch
    sys.path.insert(0, sys.argv[1])
    import combine_topk_multihot_gb300 as m
    N = m._native
    assert N.lib.moe_device_check() == 0
    T, E, K, P, H = 64, 8, 2, 1, 256
    g = torch.Generator().manual_seed(3)
    idx = torch.stack([torch.randperm(E, generator=g)[:K] for _ in range(T)]).cuda()
    p = torch.rand(T, K, generator=g).cuda()
    x = torch.randn(T, H, generator=g).to(torch.bfloat16).cuda()
    status = torch.zeros(1, dtype=torch.int32, device="cuda")
    rmap, probs, _ = m.moe_route_to_multihot(idx, p, E, status)
    C = m.worst_case_rows(T, E, K, P)
    lay = m.Layout(T, E, K, P, C, device="cuda", status=status)
    lay.c.workspace = None
    x_disp = torch.zeros(C, H, dtype=torch.bfloat16, device="cuda")
    args = lambda s: (ctypes.c_void_p(x.data_ptr()), ctypes.c_void_p(rmap.data_ptr()),
                      ctypes.c_void_p(probs.data_ptr()), H, ctypes.byref(lay.c),
                      ctypes.c_void_p(x_disp.data_ptr()), None, ctypes.c_void_p(s.cuda_stream))
    torch.cuda.synchronize()
    s = torch.cuda.Stream()
    graph = torch.cuda.CUDAGraph()
    with torch.cuda.graph(graph, stream=s):
        st = N.lib.moe_dispatch_static_scratch(*args(s))
    assert st == N.MOE_ERR_INVALID_ARG, st
    assert b"captured" in N.lib.moe_last_error()
    # outside the capture the first call goes through and equals moe_dispatch
    st = N.lib.moe_dispatch_static_scratch(*args(torch.cuda.current_stream()))
    assert st == N.MOE_OK, N.last_error()
    ref_layout = m.Layout(T, E, K, P, C, device="cuda", status=status)
    ref_x, _ = m.moe_dispatch(x, rmap, probs, ref_layout, host_sync=False)
    torch.cuda.synchronize()
    assert torch.equal(x_disp.view(torch.int16), ref_x.view(torch.int16))
    assert torch.equal(lay.row_token, ref_layout.row_token)
    print("ok")
""")


def test_first_call_under_capture_is_refused(moe):
    """In a fresh process, the first call on the device made inside a stream
    capture returns MOE_ERR_INVALID_ARG and queues nothing; the next call,
    outside the capture, looks the address up and matches moe_dispatch."""
    root = os.path.dirname(os.path.dirname(os.path.abspath(__file__)))
    r = subprocess.run([sys.executable, "-c", _CAPTURE_CHILD, root], capture_output=True, text=True,
                       timeout=300)
    assert r.returncode == 0 and r.stdout.strip().endswith("ok"), r.stdout + r.stderr
