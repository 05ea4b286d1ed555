"""Host logic of bench.py that the JSON line's claims rest on, checked without a GPU:
the number of our kernel launches per step (the `gpu_launches` claim) for each
workload shape the bench runs, and both sides of the one-kernel dispatch limit."""
import os
import sys

import pytest

ROOT = os.path.dirname(os.path.dirname(os.path.abspath(__file__)))
sys.path.insert(0, ROOT)

import bench  # noqa: E402
import synthetic  # noqa: E402
from oracle import worst_case_capacity  # noqa: E402


def _launches(name, fp8=False, gather=False):
    c = synthetic.CONFIGS[name]
    C = worst_case_capacity(c.T, c.E, c.K, c.P)
    return bench.step_launches(c.T, c.H, c.E, C, fp8, gather, c.backward)


@pytest.mark.parametrize("name,expected", [
    ("decode_1", 5),             # multihot, one-CTA layout with the rows, 2 expert kernels, combine
    ("decode_256", 6),           # 8 chunks: multihot, layout and row copy separate
    ("decode_1024", 4),          # 32 chunks: one dispatch kernel (multihot to rows), experts, combine
    ("qwen3_30b_a3b", 4),
    ("qwen3_30b_a3b_16k", 4),
    ("skewed", 4),
    ("tiny", 6),                 # 64 tokens and 248 rows: more than 64 items
    ("h4096", 11),               # + combine backward, 4 expert-backward GEMMs, dispatch and multihot backward
])
def test_launches_per_step(name, expected):
    assert _launches(name) == expected


def test_fp8_dispatch_is_fused_above_eight_chunks():
    assert _launches("decode_1", fp8=True) == 6           # multihot, layout, FP8 rows
    assert _launches("qwen3_30b_a3b", fp8=True) == 4      # the fused dispatch (multihot included) with e4m3 rows


def test_gather_step_runs_the_multihot_kernel_and_the_layout():
    assert _launches("qwen3_30b_a3b", gather=True) == 5


@pytest.mark.parametrize("T,K,E,H,expected", [
    (8, 7, 8, 512, 5),     # T + C = 8 + 56 = 64 items: one kernel
    (9, 7, 8, 512, 6),     # 72 items
    (1, 8, 128, 65536, 6), # 9 items, but 9 * 128 KiB of rows
])
def test_one_kernel_dispatch_limit(T, K, E, H, expected):
    C = worst_case_capacity(T, E, K, 1)
    assert bench.step_launches(T, H, E, C, False, False, False) == expected


def test_experts_bytes_agree_with_profiled_traffic():
    """The roofline's algorithmic byte count for the Qwen3-30B-A3B experts
    (first layer of the bench, its layout from the oracle) is within 3 % of the
    DRAM traffic ncu measured for the same two launches."""
    import oracle as O
    cfg = synthetic.CONFIGS["qwen3_30b_a3b"]
    d = synthetic.make_layer_inputs(cfg, with_weights=False)
    rm, pr, _ = O.route_to_multihot(d["topk_idx"].numpy(), d["topk_probs"].numpy(), cfg.E)
    lay = O.build_layout(rm, pr, cfg.K, cfg.P)
    R, N = lay["rows_used"], lay["rows_valid"]
    a = bench.algorithmic(cfg, lay["tokens_per_expert"], R, N, R, backward=False)
    measured = bench.PROFILED_TRAFFIC["qwen3_30b_a3b"]["bytes"]
    assert abs(a["experts_bytes"] - measured) / measured < 0.03
    assert a["experts_flops"] == 6.0 * N * cfg.H * cfg.I


@pytest.mark.parametrize("n", [1, 3, 5, 7, 20, 41])
def test_timing_windows_cover_every_step_once(n):
    b = bench.window_bounds(n)
    assert b[0][0] == 0 and b[-1][1] == n
    assert all(x[1] == y[0] for x, y in zip(b, b[1:]))
    assert len(b) == min(5, n) and all(e > s for s, e in b)
    sizes = [e - s for s, e in b]
    assert max(sizes) - min(sizes) <= 1


def test_window_summary_takes_the_median_window():
    w = bench.window_summary([4.0, 4.4, 8.0, 4.2, 4.0], [4, 4, 4, 4, 4])
    assert w["median_ms_per_step"] == 1.05
    assert abs(w["spread"] - (2.0 - 1.0) / 1.05) < 1e-12


def test_clock_summary_of_the_timed_samples_and_of_all():
    """The timed region's clock record uses only the samples taken up to its
    end; the extended record (the same steps repeated after it) all of them,
    with every throttle reason seen."""
    c = bench.ClockSampler(0)
    row = "0, {sm}, 2070, 900, 0x0, Not Active, Not Active, Not Active, {cap}\n"
    c.lines = [row.format(sm=2070, cap="Not Active"), row.format(sm=2070, cap="Not Active"),
               row.format(sm=1800, cap="Active"), "garbled\n"]
    timed = c.summary(2)
    assert timed == {"sm_mhz": 2070.0, "sm_max_mhz": 2070.0, "reasons": [], "samples": 2}
    every = c.summary()
    assert every["samples"] == 3 and every["reasons"] == ["sw_power_cap"] and every["sm_mhz"] == 2070.0
