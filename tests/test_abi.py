"""The C-ABI library loads and exports every symbol include/moe.h declares.
CPU only: no compute call is made."""
import ctypes
import os
import re

import pytest

ROOT = os.path.dirname(os.path.dirname(os.path.abspath(__file__)))


def _declared_symbols():
    with open(os.path.join(ROOT, "include", "moe.h")) as f:
        src = f.read()
    return sorted(set(re.findall(r"^MOE_API\s+[\w\s\*]+?\b(moe_\w+)\s*\(", src, flags=re.M)))


@pytest.fixture(scope="module")
def lib():
    import __graft_entry__
    path = __graft_entry__._build_module().build()
    return ctypes.CDLL(path)


def test_header_declares_the_path():
    syms = _declared_symbols()
    for name in ("moe_route_to_multihot", "moe_dispatch", "moe_grouped_experts", "moe_combine",
                 "moe_combine_backward", "moe_dispatch_backward", "moe_route_to_multihot_backward"):
        assert name in syms


def test_every_declared_symbol_is_exported(lib):
    for name in _declared_symbols():
        assert hasattr(lib, name), name


def test_binding_covers_every_declared_symbol(lib):
    from combine_topk_multihot_gb300 import _native
    assert set(_native.SIGNATURES) == set(_declared_symbols())


def test_host_only_helpers(lib):
    lib.moe_worst_case_rows.restype = ctypes.c_int64
    lib.moe_worst_case_rows.argtypes = [ctypes.c_int32] * 4
    assert lib.moe_worst_case_rows(4096, 128, 8, 128) == 4096 * 8 + 128 * 127
    assert lib.moe_worst_case_rows(1, 128, 8, 1) == 8
    lib.moe_status_string.restype = ctypes.c_char_p
    assert lib.moe_status_string(4) == b"MOE_ERR_BAD_INDEX"
    n = ctypes.c_size_t(0)
    assert lib.moe_layout_workspace_bytes(100, 8, ctypes.byref(n)) == 0
    assert n.value >= 4 * 8 * 4 and n.value % 256 == 0


def test_validation_rejects_bad_shapes_without_a_gpu(lib):
    """Shape checks run on the host before any CUDA call."""
    from combine_topk_multihot_gb300 import _native as N
    st = N.lib.moe_route_to_multihot(None, None, 4, 0, 8, None, None, None, None, None)
    assert st == N.MOE_ERR_UNSUPPORTED_SHAPE
    st = N.lib.moe_route_to_multihot(None, None, 4, 2, 6, None, None, None, None, None)  # E % 4
    assert st == N.MOE_ERR_UNSUPPORTED_SHAPE
    L = N.MoeLayout(4, 8, 2, 1, 8)
    st = N.lib.moe_combine(None, ctypes.byref(L), 100, None, None)  # layout pointers NULL
    assert st == N.MOE_ERR_INVALID_ARG
    assert b"NULL" in N.lib.moe_last_error()


def test_router_validation_without_a_gpu(lib):
    """The router entry points check shapes, NULLs and the all-or-none rule
    for the fused multihot outputs on the host."""
    from combine_topk_multihot_gb300 import _native as N
    fake = ctypes.c_void_p(16)        # never dereferenced: validation fails first
    odd = ctypes.c_void_p(16 + 4)     # not 16-byte aligned
    # K > E
    assert N.lib.moe_router_topk(fake, 4, 8, 9, fake, fake, None, None, None, None) == N.MOE_ERR_UNSUPPORTED_SHAPE
    # E not a multiple of 4, E above 1024
    assert N.lib.moe_router_topk(fake, 4, 6, 2, fake, fake, None, None, None, None) == N.MOE_ERR_UNSUPPORTED_SHAPE
    assert N.lib.moe_router_topk(fake, 4, 1028, 2, fake, fake, None, None, None, None) == N.MOE_ERR_UNSUPPORTED_SHAPE
    # NULL logits with tokens
    assert N.lib.moe_router_topk(None, 4, 8, 2, fake, fake, None, None, None, None) == N.MOE_ERR_INVALID_ARG
    # only some of the multihot outputs
    assert N.lib.moe_router_topk(fake, 4, 8, 2, fake, fake, fake, None, fake, None) == N.MOE_ERR_INVALID_ARG
    assert b"all three" in N.lib.moe_last_error()
    # misaligned multihot output
    assert N.lib.moe_router_topk(fake, 4, 8, 2, fake, fake, odd, fake, fake, None) == N.MOE_ERR_INVALID_ARG
    # backward: misaligned grad_logits, bad K
    assert N.lib.moe_router_topk_backward(fake, fake, fake, 4, 8, 2, odd, None) == N.MOE_ERR_INVALID_ARG
    assert N.lib.moe_router_topk_backward(fake, fake, fake, 4, 8, 0, fake, None) == N.MOE_ERR_UNSUPPORTED_SHAPE
