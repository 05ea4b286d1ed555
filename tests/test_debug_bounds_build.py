"""The bounds-checked build of the library, on the CPU: it builds as a variant
of its own (libmoe_bounds.so, compiled with MOE_DEBUG_BOUNDS), says so through
moe_build_flags(), exports the same ABI, and the normal build says it has no
checks.  No compute call is made; the GPU side is tests/test_gpu_debug_bounds.py.
"""
import ctypes
import os

import pytest

from tests.test_abi import _declared_symbols


@pytest.fixture(scope="module")
def libs():
    import __graft_entry__
    build = __graft_entry__._build_module()
    normal = ctypes.CDLL(build.build())
    checked = ctypes.CDLL(build.build(variant="bounds"))
    for l in (normal, checked):
        l.moe_build_flags.restype = ctypes.c_uint32
    return build, normal, checked


def test_variant_is_a_separate_library(libs):
    build, _, _ = libs
    assert build.library_path("bounds") != build.library_path()
    assert os.path.basename(build.library_path("bounds")) == "libmoe_bounds.so"
    assert os.path.exists(build.library_path("bounds"))


def test_build_flags_report_the_checks(libs):
    from combine_topk_multihot_gb300 import _native as N
    _, normal, checked = libs
    assert normal.moe_build_flags() == 0
    assert checked.moe_build_flags() == N.MOE_BUILD_BOUNDS_CHECKS


def test_checked_build_exports_the_same_abi(libs):
    _, _, checked = libs
    for name in _declared_symbols():
        assert hasattr(checked, name), name


def test_binding_loads_either_build(libs):
    from combine_topk_multihot_gb300 import _native as N
    build, _, _ = libs
    h = N.load(build.library_path("bounds"))
    assert h.moe_build_flags() == N.MOE_BUILD_BOUNDS_CHECKS
    assert h.moe_worst_case_rows(4096, 128, 8, 128) == 4096 * 8 + 128 * 127
