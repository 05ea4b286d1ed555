"""ctypes view of the C ABI in include/moe.h.

Loads the in-tree ``_lib/libmoe.so``.  There is no fallback: if the library
has not been built, importing this module raises ImportError.
"""
from __future__ import annotations

import ctypes
import os

_LIB_PATH = os.path.join(os.path.dirname(os.path.abspath(__file__)), "_lib", "libmoe.so")

if not os.path.exists(_LIB_PATH):
    raise ImportError(
        f"the CUDA library {_LIB_PATH} is not built; run "
        "`python -c 'import __graft_entry__ as g; g.build()'` (needs nvcc)")


c_int32 = ctypes.c_int32
c_int64 = ctypes.c_int64
c_void_p = ctypes.c_void_p
c_size_t = ctypes.c_size_t

# Status codes and device status bits (include/moe.h).
MOE_OK = 0
MOE_ERR_INVALID_ARG = 1
MOE_ERR_UNSUPPORTED_SHAPE = 2
MOE_ERR_CAPACITY = 3
MOE_ERR_BAD_INDEX = 4
MOE_ERR_TIMEOUT = 5
MOE_ERR_DEVICE = 6
MOE_ERR_CUDA = 7
MOE_DEVERR_BAD_INDEX = 1
MOE_DEVERR_CAPACITY = 2
MOE_DEVERR_TIMEOUT = 4
MOE_DEVERR_BOUNDS = 8
MOE_BUILD_BOUNDS_CHECKS = 1
MOE_STATIC_SCRATCH_INTS = 262144


class MoeLayout(ctypes.Structure):
    """struct moe_layout."""
    _fields_ = [
        ("T", c_int32), ("E", c_int32), ("K", c_int32), ("pad_multiple", c_int32),
        ("capacity", c_int64),
        ("tokens_per_expert", c_void_p), ("offsets", c_void_p), ("totals", c_void_p),
        ("row_token", c_void_p), ("row_expert", c_void_p), ("row_weight", c_void_p),
        ("token_row", c_void_p), ("status", c_void_p), ("workspace", c_void_p),
    ]


_P = c_void_p
_LP = ctypes.POINTER(MoeLayout)

# name -> (restype, argtypes); every entry point of include/moe.h
SIGNATURES = {
    "moe_status_string": (ctypes.c_char_p, [c_int32]),
    "moe_last_error": (ctypes.c_char_p, []),
    "moe_device_check": (c_int32, []),
    "moe_build_flags": (ctypes.c_uint32, []),
    "moe_worst_case_rows": (c_int64, [c_int32, c_int32, c_int32, c_int32]),
    "moe_layout_workspace_bytes": (c_int32, [c_int32, c_int32, ctypes.POINTER(c_size_t)]),
    "moe_router_topk": (c_int32, [_P, c_int32, c_int32, c_int32, _P, _P, _P, _P, _P, _P]),
    "moe_router_topk_backward": (c_int32, [_P, _P, _P, c_int32, c_int32, c_int32, _P, _P]),
    "moe_route_to_multihot": (c_int32, [_P, _P, c_int32, c_int32, c_int32, _P, _P, _P, _P, _P]),
    "moe_dispatch_layout": (c_int32, [_P, _P, _LP, ctypes.POINTER(c_int64), _P]),
    "moe_grouped_experts_gather": (c_int32, [_P, _LP, c_int32, c_int32, _P, _P, _P, _P, _P, _P, _P]),
    "moe_dispatch_fp8": (c_int32, [_P, _P, _P, c_int32, _LP, _P, _P, ctypes.POINTER(c_int64), _P]),
    "moe_quantize_fp8": (c_int32, [_P, c_int64, c_int32, _P, _P, _P]),
    "moe_grouped_experts_fp8": (c_int32, [_P, _P, _LP, c_int32, c_int32, _P, _P, _P, _P, _P, _P]),
    "moe_dispatch": (c_int32, [_P, _P, _P, c_int32, _LP, _P, ctypes.POINTER(c_int64), _P]),
    "moe_dispatch_topk": (c_int32, [_P, _P, _P, c_int32, _LP, _P, _P, _P, _P, ctypes.POINTER(c_int64), _P]),
    "moe_dispatch_topk_fp8": (c_int32, [_P, _P, _P, c_int32, _LP, _P, _P, _P, _P, _P, ctypes.POINTER(c_int64), _P]),
    "moe_dispatch_static_scratch": (c_int32, [_P, _P, _P, c_int32, _LP, _P, ctypes.POINTER(c_int64), _P]),
    "moe_grouped_experts": (c_int32, [_P, _LP, c_int32, c_int32, _P, _P, _P, _P, _P, _P, _P]),
    "moe_combine": (c_int32, [_P, _LP, c_int32, _P, _P]),
    "moe_combine_backward": (c_int32, [_P, _P, _LP, c_int32, _P, _P, _P]),
    "moe_combine_backward_scaled": (c_int32, [_P, _P, _LP, c_int32, _P, _P, _P]),
    "moe_dispatch_backward": (c_int32, [_P, _P, _LP, c_int32, _P, _P, _P]),
    "moe_experts_backward_workspace_bytes": (c_int32, [c_int64, c_int32, c_int32, ctypes.POINTER(c_size_t)]),
    "moe_grouped_experts_backward": (c_int32, [_P, _P, _P, _P, _LP, c_int32, c_int32, _P, _P, _P, _P, _P, _P, _P]),
    "moe_grouped_experts_backward_scaled": (c_int32, [_P, _P, _P, _P, _LP, c_int32, c_int32, _P, _P, _P, _P, _P,
                                                      _P, _P]),
    "moe_selftest_wait_timeout": (c_int32, [_P, c_int64, _P, _P]),
    "moe_route_to_multihot_backward": (c_int32, [_P, _P, _P, c_int32, c_int32, c_int32, _P, _P]),
}

def load(path: str) -> ctypes.CDLL:
    """Opens a copy of the library (the normal build, or the bounds-checked
    libmoe_bounds.so) with the ABI's signatures attached."""
    handle = ctypes.CDLL(path)
    for name, (res, args) in SIGNATURES.items():
        fn = getattr(handle, name)
        fn.restype = res
        fn.argtypes = args
    return handle


lib = load(_LIB_PATH)


def status_string(code: int) -> str:
    return lib.moe_status_string(code).decode()


def last_error() -> str:
    return lib.moe_last_error().decode()
