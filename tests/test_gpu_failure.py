"""Failure detection without a GPU fault: a bounded device wait that runs
out reports MOE_DEVERR_TIMEOUT and the context stays usable."""
import ctypes

import numpy as np
import pytest
import torch

import oracle as O
from tests._util import random_routing

pytestmark = pytest.mark.gpu


def test_bounded_wait_times_out_and_context_survives():
    import combine_topk_multihot_gb300 as moe
    N = moe._native
    status = torch.zeros(1, dtype=torch.int32, device="cuda")
    waited = torch.zeros(1, dtype=torch.int64, device="cuda")
    limit = 50_000_000  # 50 ms
    st = N.lib.moe_selftest_wait_timeout(ctypes.c_void_p(status.data_ptr()), limit,
                                         ctypes.c_void_p(waited.data_ptr()),
                                         ctypes.c_void_p(torch.cuda.current_stream().cuda_stream))
    assert st == N.MOE_OK, N.last_error()
    torch.cuda.synchronize()
    assert int(status.item()) == N.MOE_DEVERR_TIMEOUT
    w = int(waited.item())
    assert limit <= w < 20 * limit, w
    # the GPU still works: a dispatch right after is still exact
    T, E, K, P = 40, 8, 2, 4
    idx, p = random_routing(T, E, K, seed=7)
    st2 = torch.zeros(1, dtype=torch.int32, device="cuda")
    rmap, probs, _ = moe.moe_route_to_multihot(idx.cuda(), p.cuda(), E, st2)
    torch.cuda.synchronize()
    assert np.array_equal(rmap.cpu().numpy(), O.route_to_multihot(idx.numpy(), p.numpy(), E)[0])
    assert int(st2.item()) == 0


def test_selftest_rejects_bad_limits():
    import combine_topk_multihot_gb300 as moe
    N = moe._native
    status = torch.zeros(1, dtype=torch.int32, device="cuda")
    for bad in (0, -1, 2_000_000_000):
        assert N.lib.moe_selftest_wait_timeout(ctypes.c_void_p(status.data_ptr()), bad, None, None) \
            == N.MOE_ERR_INVALID_ARG
