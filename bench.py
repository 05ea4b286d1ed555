"""Benchmark of the MoE dispatch -> experts -> combine layer on GB300.

One step = one forward pass of the whole layer (multihot, counts/offsets,
layout + dispatch gather, grouped SwiGLU experts, combine) over one batch of
the configured layer; with a backward config (h4096) the step also runs the
backward entry points.  Four distinct layers (weights, tokens, routing) are
cycled so the working set does not sit in L2 (each layer's weights alone are
larger than the 126 MB L2).

The timed steps run in five consecutive windows, each timed with its own
pair of CUDA events on the launching stream, and the step time is the median
window's (the pages time four distinct layers back to back and take medians
of windows).  The default run (the Qwen3-30B-A3B layer at T = 4096) also
times the same shape at T = 16384 and reports it under
``kernels.target_layer_T16384``.

Prints one JSON line (rank 0).  ``--impl reference`` times the CPU oracle
instead, on a bounded sample of the same workload.
"""
from __future__ import annotations

import argparse
import json
import os
import statistics
import subprocess
import sys
import time

ROOT = os.path.dirname(os.path.abspath(__file__))
sys.path.insert(0, ROOT)

import numpy as np  # noqa: E402
import torch  # noqa: E402

import synthetic  # noqa: E402

MEASURED_PEAKS = os.path.join(ROOT, "MEASURED_PEAKS.json")

# DRAM traffic (dram__bytes_read.sum + dram__bytes_write.sum) of the experts'
# two GEMM launches on one layer, from an ncu capture of the kernels whose
# sources hash to `src` (profiles/experts_gemm_qwen3_30b_a3b_T4096.md); the
# figure is reported only while the sources still match.
PROFILED_TRAFFIC = {
    "qwen3_30b_a3b": {"src": "91925a54da15a583", "bytes": (951.97 + 44.78 + 457.13 + 108.96) * 1e6,
                      "profile": "profiles/experts_gemm_qwen3_30b_a3b_T4096.md"},
}
GEMM_SOURCES = ("combine_topk_multihot_gb300/csrc/gemm.cu", "combine_topk_multihot_gb300/csrc/gemm_pair.cu",
                "combine_topk_multihot_gb300/csrc/common.cuh", "combine_topk_multihot_gb300/csrc/tma.cu")


def profiled_traffic(workload: str):
    import hashlib
    rec = PROFILED_TRAFFIC.get(workload)
    if rec is None:
        return None
    h = hashlib.sha256()
    for f in GEMM_SOURCES:
        with open(os.path.join(ROOT, f), "rb") as fh:
            h.update(fh.read())
    return rec["bytes"] if h.hexdigest()[:16] == rec["src"] else None
CLOCK_EXTRA_S = 0.6
FALLBACK_HBM_GBS = 6800.0
FALLBACK_BF16_TFLOPS = 1900.0


def peaks():
    try:
        with open(MEASURED_PEAKS) as f:
            p = json.load(f)
        return float(p["hbm_gbs"]), float(p["bf16_tflops"]), float(p.get("bf16_tflops_sustained", p["bf16_tflops"])), "measured"
    except Exception:
        return FALLBACK_HBM_GBS, FALLBACK_BF16_TFLOPS, 1700.0, "fallback"


# ----------------------------------------------------------------------------- distributed

def dist_setup(n_gpus: int):
    world = int(os.environ.get("WORLD_SIZE", "1"))
    rank = int(os.environ.get("RANK", "0"))
    local = int(os.environ.get("LOCAL_RANK", "0"))
    if world > 1:
        import torch.distributed as dist
        backend = "nccl" if torch.cuda.is_available() else "gloo"
        if torch.cuda.is_available():
            torch.cuda.set_device(local)
        dist.init_process_group(backend)
    return world, rank, local


def barrier(world):
    if world > 1:
        import torch.distributed as dist
        dist.barrier()


def max_over_ranks(value: float, world: int) -> float:
    """The slowest rank's time: an all-reduce MAX over ranks."""
    if world == 1:
        return value
    import torch.distributed as dist
    dev = torch.device("cuda", torch.cuda.current_device()) if dist.get_backend() == "nccl" else torch.device("cpu")
    t = torch.tensor([value], dtype=torch.float64, device=dev)
    dist.all_reduce(t, op=dist.ReduceOp.MAX)
    return float(t.item())


# ----------------------------------------------------------------------------- clocks

class ClockSampler:
    """nvidia-smi clocks and throttle reasons, sampled during the timed region."""

    FIELDS = ("index,clocks.sm,clocks.max.sm,power.draw,clocks_event_reasons.active,"
              "clocks_event_reasons.hw_slowdown,clocks_event_reasons.hw_thermal_slowdown,"
              "clocks_event_reasons.sw_thermal_slowdown,clocks_event_reasons.sw_power_cap")

    def __init__(self, device_index: int):
        self.dev = device_index
        self.proc = None
        self.lines = []

    def __enter__(self):
        import threading
        self._first = threading.Event()
        try:
            self.proc = subprocess.Popen(
                ["nvidia-smi", "-i", str(self.dev), f"--query-gpu={self.FIELDS}",
                 "--format=csv,noheader,nounits", "-lms", "100"],
                stdout=subprocess.PIPE, stderr=subprocess.DEVNULL, text=True)
        except Exception:
            self.proc = None
            return self

        def read():
            for line in self.proc.stdout:
                if line.strip():
                    self.lines.append(line)
                    self._first.set()

        self._reader = threading.Thread(target=read, daemon=True)
        self._reader.start()
        # nvidia-smi's start-up (NVML initialisation) can hold driver locks
        # that stall the host's CUDA calls for tens of milliseconds: let it
        # finish before the timed region starts.
        self._first.wait(timeout=5.0)
        return self

    def __exit__(self, *a):
        if self.proc is not None:
            time.sleep(0.15)
            self.proc.terminate()
            try:
                self.proc.wait(timeout=5)
            except Exception:
                self.proc.kill()
            self._reader.join(timeout=5)

    def summary(self, upto=None):
        """Median SM clock, the maximum and the throttle reasons seen, over the
        first ``upto`` samples (all when None)."""
        sm, mx, reasons = [], None, set()
        names = ["hw_slowdown", "hw_thermal_slowdown", "sw_thermal_slowdown", "sw_power_cap"]
        for l in (self.lines if upto is None else self.lines[:upto]):
            f = [x.strip() for x in l.split(",")]
            if len(f) < 9:
                continue
            try:
                sm.append(float(f[1]))
                mx = float(f[2])
            except ValueError:
                continue
            for n, v in zip(names, f[5:9]):
                if v.lower() == "active":
                    reasons.add(n)
        return {"sm_mhz": statistics.median(sm) if sm else None, "sm_max_mhz": mx,
                "reasons": sorted(reasons), "samples": len(sm)}


# ----------------------------------------------------------------------------- algorithmic work

def experts_kernel_label(cfg, fp8: bool, gather: bool, backward: bool) -> str:
    """Which expert GEMM kernels a bench step runs, as the library picks them:
    bf16 layers with rows for every SM take pair_gemm_kernel (CTA pairs,
    expert rows on the MMA's N side) above 64 rows per expert on average and
    grouped_gemm_kernel (one CTA per tile) up to that; e4m3 operands, the
    gathered A and small layers grouped_gemm_kernel; T <= 4 in inference the
    CUDA-core gemv_experts_kernel."""
    wide = min(cfg.T * cfg.K, cfg.E) * (cfg.I // 128) >= 152
    if cfg.T <= 4 and not backward and not fp8:
        fwd = "experts: gemv_experts_kernel<1> (gate/up + SwiGLU) + gemv_experts_kernel<2> (down x weight), CUDA cores"
    elif fp8 or gather or not wide:
        fwd = ("experts: grouped_gemm_kernel<0> (gate/up + SwiGLU" + (", e4m3 operands" if fp8 else "")
               + (", A gathered" if gather else "") + ("" if wide else ", 64-column tiles")
               + ") + grouped_gemm_kernel<1> (down x weight)")
    elif cfg.T * cfg.K <= 64 * cfg.E:
        fwd = "experts: grouped_gemm_kernel<0> (gate/up + SwiGLU, one CTA per tile) + grouped_gemm_kernel<1> (down x weight)"
    else:
        fwd = "experts: pair_gemm_kernel<0> (gate/up + SwiGLU) + pair_gemm_kernel<1> (down x weight)"
    return fwd + (" + the backward's 4 bwd_gemm_kernel launches" if backward else "")


def step_launches(T: int, H: int, E: int, C: int, fp8: bool, gather: bool, backward: bool) -> int:
    """Our kernel launches in one step (the dispatch's barrier-counter memset is
    a driver memset, not one of ours), then the two expert kernels and the
    combine, and with the backward the combine backward (which also applies the
    routing weight), the four expert-backward GEMMs, the dispatch backward and
    the multihot backward.
    The dispatch of a layer of more than 8 chunks of 32 tokens is one
    cooperative kernel, which in the bf16 step also does the multihot step; the
    --gather step runs the multihot kernel and that kernel without rows, the
    FP8 step that kernel with e4m3 rows (the multihot step included).  Smaller layers run the
    multihot kernel, the barrier-free layout kernel and the row copy, except
    that a layer of at most two chunks, whose one-CTA layout fits 48 KiB of
    shared memory and whose row pass has at most 64 items (tokens + rows) and
    256 KiB, lays out and copies in one kernel (bf16 only)."""
    chunks = -(-T // 32)
    fused_smem = (4 * E + 2) * 4 + 8 * 128 * 4
    if chunks > 8 and fused_smem <= 48 * 1024:
        n = 2 if gather else 1
    elif chunks > 8:
        n = 3
    else:
        single_smem = 32 * E + 32 * (-(-E // 32)) * 4 + (2 * E + 1) * 4 + chunks * E * 4
        single_rows = (not fp8 and chunks <= 2 and single_smem <= 48 * 1024 and T + C <= 64
                       and (0 if gather else (T + C) * H * 2) <= 256 * 1024)
        n = 1 + (1 if single_rows else 2)
    n += 2 + 1
    if backward:
        n += 1 + 4 + 1 + 1
    return n


N_WINDOWS = 5


def window_bounds(n_units: int, n_windows: int = N_WINDOWS):
    """Splits n_units consecutive timed units into up to n_windows contiguous
    windows of nearly equal size: [(start, end), ...] covering every unit."""
    n = max(1, min(n_windows, n_units))
    cuts = [round(i * n_units / n) for i in range(n + 1)]
    return [(cuts[i], cuts[i + 1]) for i in range(n) if cuts[i + 1] > cuts[i]]


def window_summary(win_ms, win_steps):
    """Per-step time of each window, their median and relative spread."""
    per = [t / s for t, s in zip(win_ms, win_steps)]
    med = statistics.median(per)
    return {"n": len(per), "steps": list(win_steps), "ms_per_step": per, "median_ms_per_step": med,
            "spread": (max(per) - min(per)) / med if med > 0 else 0.0}


def algorithmic(cfg, counts: np.ndarray, R: int, N: int, C: int, backward: bool, fp8: bool = False,
                gather: bool = False, fused_multihot: bool = False):
    """Bytes / flops the layer's steps must move, per call: what each step has to
    read and write at the least, and the experts' 2 flops per multiply-add.
    With fp8 the dispatched rows and W1 are e4m3 (1 byte) with fp32 per-row scales.
    With gather no rows are dispatched: the gate/up GEMM reads the tokens x once.
    With fused_multihot the dispatch call also does the multihot step (reads
    the top-k choices, writes the multihot rows) and its bytes count there."""
    T, H, E, K, I = cfg.T, cfg.H, cfg.E, cfg.K, cfg.I
    active = int((counts > 0).sum())
    meta_disp = T * E * 1 + 4 * N + 12 * C + 4 * T * K + 8 * (E + 1)
    row_b = 1 if fp8 else 2
    disp = (meta_disp if gather else
            T * H * 2 + C * H * row_b + meta_disp + (4 * C if fp8 else 0))
    if fused_multihot:
        disp += T * K * 12 + T * E * 6
    comb = N * H * 2 + T * H * 2 + 4 * T * K
    w_bytes = active * (2 * I * H * row_b + H * I * 2) + (active * 2 * I * 4 if fp8 else 0)
    ex_bytes = w_bytes + (T * H * 2 if gather else N * H * row_b) + 2 * N * I * 2 + N * H * 2
    ex_flops = 6.0 * N * H * I
    out = {"dispatch_bytes": disp, "combine_bytes": comb, "experts_bytes": ex_bytes,
           "experts_flops": ex_flops, "multihot_bytes": T * K * 12 + T * E * 6}
    if backward:
        out["combine_bwd_bytes"] = T * H * 2 + C * H * 2 + N * H * 2 + 4 * C
        out["dispatch_bwd_bytes"] = N * H * 2 + T * H * 2 + T * E * 4
        # dgrad1 (W2, gu), dgrad2 (W1), wgrad2, wgrad1 (fp32 dW written); G_o
        # comes from the combine backward's scatter
        out["experts_bwd_bytes"] = (w_bytes + 2 * w_bytes  # weights read, fp32 dW written
                                    + N * H * 2 * 3        # G_o (2 reads), x_disp
                                    + N * 2 * I * 2 * 4    # gu read, G_gu (w + 2 r)
                                    + N * I * 2 + N * H * 2)  # h read, grad_x_disp written
        out["experts_bwd_flops"] = 12.0 * N * H * I
    return out


# ----------------------------------------------------------------------------- our arm

def run_ours(args, world, rank, local, leg: bool = False):
    """Times the configured layer.  With ``leg`` only the device-timed steps
    and their per-stage split are measured (no sync-free dispatch timing and no
    end-to-end copies): the extra workload line inside the default run."""
    import combine_topk_multihot_gb300 as moe

    dev = torch.device("cuda", local)
    torch.cuda.set_device(dev)
    cfg = synthetic.CONFIGS[args.config]
    T, H, E, K, I, P = cfg.T, cfg.H, cfg.E, cfg.K, cfg.I, cfg.P
    host_sync = not cfg.sync_free
    n_layers = args.layers
    fp8 = args.fp8
    gather = args.gather
    if (fp8 or gather) and cfg.backward:
        raise SystemExit("--fp8 and --gather are inference paths (the backward reads x_disp)")
    if fp8 and gather:
        raise SystemExit("--fp8 and --gather are separate paths")

    layers = []
    for l in range(n_layers):
        s = cfg.seed + 7919 * l + 104729 * rank
        x = synthetic.make_tokens(T, H, s, device=dev)
        idx, p = synthetic.make_routing(T, E, K, s, cfg.zipf_s, cfg.drop)
        W1, W2 = synthetic.make_weights(E, H, I, s, device=dev)
        layers.append({"x": x, "topk_idx": idx.to(dev), "topk_probs": p.to(dev), "W1": W1, "W2": W2})
        if fp8:  # weights are quantized once, like a checkpoint converted at load time
            layers[-1]["W1q"], layers[-1]["W1s"] = moe.moe_quantize_fp8(W1)
    worst = moe.worst_case_rows(T, E, K, P)
    # host-synced mode: buffers sized once to the largest R over the layers, as
    # a caching allocator would hold them; sync-free: the worst case
    C = worst
    lay = moe.Layout(T, E, K, P, C, device=dev)
    x_disp = torch.empty(C, H, dtype=torch.bfloat16, device=dev)
    bufs = {"h": torch.empty(C, I, dtype=torch.bfloat16, device=dev),
            "y": torch.empty(C, H, dtype=torch.bfloat16, device=dev)}
    out = torch.empty(T, H, dtype=torch.bfloat16, device=dev)
    # find the exact rows of each layer, then size the buffers to the largest
    rows = []
    for L in layers:
        rmap, probs, _ = moe.moe_route_to_multihot(L["topk_idx"], L["topk_probs"], E, lay.status)
        _, rc = moe.moe_dispatch(L["x"], rmap, probs, lay, host_sync=True, x_disp=x_disp)
        rows.append(rc)
        L["counts"] = lay.tokens_per_expert.cpu().numpy()
    if host_sync:
        C = max(r[0] for r in rows)
        lay = moe.Layout(T, E, K, P, C, device=dev)
        x_disp = torch.empty(C, H, dtype=torch.bfloat16, device=dev)
        bufs = {"h": torch.empty(C, I, dtype=torch.bfloat16, device=dev),
                "y": torch.empty(C, H, dtype=torch.bfloat16, device=dev)}

    if fp8:
        x_q = (torch.empty(C, H, dtype=torch.uint8, device=dev), torch.empty(C, dtype=torch.float32, device=dev))
    stream = torch.cuda.current_stream()
    ev = lambda: torch.cuda.Event(enable_timing=True)
    # the bf16 and FP8 paths call moe_dispatch_topk(_fp8): the multihot step and
    # the dispatch in one call
    fused_topk = not gather
    mh = (torch.empty(T, E, dtype=torch.uint8, device=dev), torch.empty(T, E, dtype=torch.float32, device=dev),
          torch.empty(T, E, dtype=torch.int8, device=dev))
    bwd = cfg.backward
    stages = ["multihot", "dispatch", "experts", "combine"]
    launches_per_step = step_launches(T, H, E, C, fp8, gather, bwd)
    if bwd:
        stages += ["combine_bwd", "experts_bwd", "dispatch_bwd", "multihot_bwd"]
        bufs["o"] = torch.empty(C, H, dtype=torch.bfloat16, device=dev)
        bufs["gu"] = torch.empty(C, 2 * I, dtype=torch.bfloat16, device=dev)
        for l, L in enumerate(layers):
            L["grad_out"] = synthetic.make_grad_out(T, H, cfg.seed + 7919 * l + 104729 * rank, device=dev)

    def step(L, events=None, out_buf=None):
        rec = (lambda j: events[j].record(stream)) if events else (lambda j: None)
        o_buf = out if out_buf is None else out_buf
        rec(0)
        if fused_topk and fp8:  # the multihot step runs inside the dispatch call (its stage is 0)
            _, _, (rmap, probs, win), _ = moe.moe_dispatch_topk_fp8(L["x"], L["topk_idx"], L["topk_probs"], lay,
                                                                    host_sync=host_sync, out=x_q, multihot=mh)
            rec(2)
            moe.moe_grouped_experts_fp8(x_q[0], x_q[1], lay, L["W1q"], L["W1s"], L["W2"], out=bufs)
            rec(3)
        elif fused_topk:
            _, (rmap, probs, win), _ = moe.moe_dispatch_topk(L["x"], L["topk_idx"], L["topk_probs"], lay,
                                                             host_sync=host_sync, x_disp=x_disp, multihot=mh)
            rec(2)
            moe.moe_grouped_experts(x_disp, lay, L["W1"], L["W2"], out=bufs, save_o=bwd, save_gu=bwd)
            rec(3)
        else:
            rmap, probs, win = moe.moe_route_to_multihot(L["topk_idx"], L["topk_probs"], E, lay.status)
            rec(1)
        if fused_topk:
            pass
        elif gather:
            moe.moe_dispatch_layout(rmap, probs, lay, host_sync=host_sync)
            rec(2)
            moe.moe_grouped_experts_gather(L["x"], lay, L["W1"], L["W2"], out=bufs)
            rec(3)
        else:
            moe.moe_dispatch(L["x"], rmap, probs, lay, host_sync=host_sync, x_disp=x_disp)
            rec(2)
            moe.moe_grouped_experts(x_disp, lay, L["W1"], L["W2"], out=bufs, save_o=bwd, save_gu=bwd)
            rec(3)
        moe.moe_combine(bufs["y"], lay, out=o_buf)
        rec(4)
        if bwd:
            # the routing weight goes onto the gradient in the combine backward's
            # scatter (G_o = w * grad_y), so the experts' backward needs no scaling pass
            g_o, grad_w = moe.moe_combine_backward(L["grad_out"], lay, o_save=bufs["o"], scaled=True)
            rec(5)
            gxd, dW1, dW2 = moe.moe_grouped_experts_backward(g_o, x_disp, bufs["h"], bufs["gu"], lay,
                                                             L["W1"], L["W2"], scaled=True)
            rec(6)
            grad_x, grad_probs = moe.moe_dispatch_backward(gxd, lay, grad_w)
            rec(7)
            moe.moe_route_to_multihot_backward(grad_probs, L["topk_idx"], win)
            rec(8)
            return grad_x
        return None

    for i in range(args.warmup):
        step(layers[i % n_layers])
    torch.cuda.synchronize()
    barrier(world)

    step_events = [[ev() for _ in range(len(stages) + 1)] for _ in range(args.steps)]
    t0, t1 = ev(), ev()
    # Sync-free workloads (decode) run as CUDA graphs, one per cycled layer,
    # captured after the eager warm-up and replayed in the timed loop; their
    # per-stage split comes from an eager pass of the same steps.
    graphs = None
    if cfg.sync_free:
        for i in range(args.steps):
            step(layers[i % n_layers], step_events[i])
        torch.cuda.synchronize()
        graphs = []
        graph_out = [torch.empty_like(out) for _ in layers]  # one output per graph
        for L, o in zip(layers, graph_out):
            g = torch.cuda.CUDAGraph()
            with torch.cuda.graph(g):
                step(L, out_buf=o)
            graphs.append(g)
        # the timed loop replays the cycled layers back to back as one graph
        # (a decode step runs its layers in one graph), so a step costs the
        # device's time and not one host launch per layer; a remainder of
        # steps % n_layers replays the single-layer graphs
        cycle = torch.cuda.CUDAGraph()
        with torch.cuda.graph(cycle):
            for L, o in zip(layers, graph_out):
                step(L, out_buf=o)
        for i in range(args.warmup):
            graphs[i % n_layers].replay()
        cycle.replay()
        torch.cuda.synchronize()
    # The timed steps, in N_WINDOWS consecutive windows (one CUDA event pair
    # each); the step time is the median window's, as the pages time their
    # layers (medians of windows of back-to-back layers).
    if graphs is not None:
        units = [(cycle.replay, n_layers)] * (args.steps // n_layers) + \
                [(graphs[i].replay, 1) for i in range(args.steps % n_layers)]
    else:
        # no per-stage events inside the timed windows: each event record is a
        # gap on the stream; the stage split comes from a separate pass below
        units = [((lambda i=i: step(layers[i % n_layers])), 1) for i in range(args.steps)]
    bounds = window_bounds(len(units))
    w_ev = [ev() for _ in range(len(bounds) + 1)]
    with ClockSampler(local) as clk:
        torch.cuda.synchronize()
        barrier(world)
        t0.record(stream)
        w_ev[0].record(stream)
        for wi, (a, b) in enumerate(bounds):
            for fn, _ in units[a:b]:
                fn()
            w_ev[wi + 1].record(stream)
        t1.record(stream)
        torch.cuda.synchronize()
        n_timed_samples = len(clk.lines)
        # A timed region of a few ms sees one or two clock samples; the same
        # steps, repeated untimed for about CLOCK_EXTRA_S more, give the clock
        # record a longer look at the GPU under this load (reported apart).
        t_end = time.time() + CLOCK_EXTRA_S
        while time.time() < t_end:
            for fn, _ in units:
                fn()
            torch.cuda.synchronize()
    barrier(world)
    ms = t0.elapsed_time(t1)
    windows = window_summary([w_ev[i].elapsed_time(w_ev[i + 1]) for i in range(len(bounds))],
                             [sum(n for _, n in units[a:b]) for a, b in bounds])
    ms_step_max = max_over_ranks(windows["median_ms_per_step"], world)
    ms_max = max_over_ranks(ms, world)
    if graphs is None:
        # the per-stage split: the same steps again, each stage between two events
        for i in range(args.steps):
            step(layers[i % n_layers], step_events[i])
        torch.cuda.synchronize()
    per = {k: [] for k in stages}
    for evs in step_events:
        for j, k in enumerate(stages):
            if fused_topk and j == 0:      # multihot: inside the dispatch
                per[k].append(0.0)
            elif fused_topk and j == 1:    # dispatch: from the step's first event
                per[k].append(evs[0].elapsed_time(evs[2]))
            else:
                per[k].append(evs[j].elapsed_time(evs[j + 1]))
    status = int(lay.status.item())
    if status:
        raise RuntimeError(f"device status word set: {status}")

    sf_us, e2e_ms, h2d, d2h = None, None, 0, 0
    if not leg:
        # ---- the dispatch without its host round trip: the same layers in
        # sync-free mode (worst-case capacity), outside the timed region
        lay_sf = moe.Layout(T, E, K, P, worst, device=dev)
        xd_sf = torch.empty(worst, H, dtype=torch.bfloat16, device=dev)
        xq_sf = (torch.empty(worst, H, dtype=torch.uint8, device=dev),
                 torch.empty(worst, dtype=torch.float32, device=dev)) if fp8 else None
        # The calls are queued back to back and synchronised once, so that the
        # device time of each is measured rather than the host's launch latency.
        sf_ev = []
        for i in range(args.warmup + args.steps):
            L = layers[i % n_layers]
            if not fused_topk:
                rmap, probs, _ = moe.moe_route_to_multihot(L["topk_idx"], L["topk_probs"], E, lay_sf.status)
            a, b = ev(), ev()
            a.record(stream)
            if fused_topk and fp8:
                moe.moe_dispatch_topk_fp8(L["x"], L["topk_idx"], L["topk_probs"], lay_sf, host_sync=False,
                                          out=xq_sf, multihot=mh)
            elif fused_topk:
                moe.moe_dispatch_topk(L["x"], L["topk_idx"], L["topk_probs"], lay_sf, host_sync=False,
                                      x_disp=xd_sf, multihot=mh)
            elif gather:
                moe.moe_dispatch_layout(rmap, probs, lay_sf, host_sync=False)
            else:
                moe.moe_dispatch(L["x"], rmap, probs, lay_sf, host_sync=False, x_disp=xd_sf)
            b.record(stream)
            if i >= args.warmup:
                sf_ev.append((a, b))
        torch.cuda.synchronize()
        sf_us = [1e3 * a.elapsed_time(b) for a, b in sf_ev]
        del lay_sf, xd_sf, xq_sf

        # ---- end to end through the public API with host buffers
        pin = lambda t: t.cpu().pin_memory()
        in_keys = ("x", "topk_idx", "topk_probs") + (("grad_out",) if bwd else ())
        host = [{k: pin(L[k]) for k in in_keys} for L in layers]
        out_host = torch.empty(T, H, dtype=torch.bfloat16).pin_memory()
        gx_host = torch.empty(T, H, dtype=torch.bfloat16).pin_memory() if bwd else None
        h2d = sum(v.numel() * v.element_size() for v in host[0].values())
        d2h = out_host.numel() * out_host.element_size() * (2 if bwd else 1)

        # Every step copies its inputs from pinned host memory and reads its output
        # back.  The copies run on their own streams, double-buffered, so the
        # inputs of step i + 1 and the output of step i - 1 move while step i
        # computes; events order each buffer's reuse.  Eager steps alternate two
        # buffer sets; the graphs read and write their own layer's buffers.
        h2d_stream, d2h_stream = torch.cuda.Stream(), torch.cuda.Stream()
        nbuf = n_layers if graphs is not None else 2
        d_in = [{k: torch.empty_like(layers[0][k]) for k in in_keys} for _ in range(nbuf)]
        d_out = [torch.empty_like(out) for _ in range(nbuf)]
        mk = lambda: [torch.cuda.Event() for _ in range(nbuf)]
        in_ready, in_free, out_ready, out_free = mk(), mk(), mk(), mk()

        def e2e_inputs(i):
            """Queue step i's host-to-device input copies."""
            b = i % nbuf
            dst = layers[i % n_layers] if graphs is not None else d_in[b]
            h2d_stream.wait_event(in_free[b])
            with torch.cuda.stream(h2d_stream):
                for k in in_keys:
                    dst[k].copy_(host[i % n_layers][k], non_blocking=True)
                in_ready[b].record(h2d_stream)

        def e2e_compute(i):
            """Step i on the compute stream, then its output's read-back."""
            b = i % nbuf
            stream.wait_event(in_ready[b])
            stream.wait_event(out_free[b])
            gx = None
            if graphs is not None:
                graphs[i % n_layers].replay()
                res = graph_out[i % n_layers]
            else:
                L = dict(layers[i % n_layers])
                L.update(d_in[b])
                gx = step(L, out_buf=d_out[b])
                res = d_out[b]
            in_free[b].record(stream)
            out_ready[b].record(stream)
            d2h_stream.wait_event(out_ready[b])
            with torch.cuda.stream(d2h_stream):
                out_host.copy_(res, non_blocking=True)
                if bwd:
                    gx.record_stream(d2h_stream)  # allocated per step: keep it until the copy is done
                    gx_host.copy_(gx, non_blocking=True)
                out_free[b].record(d2h_stream)

        def e2e_step_inline(i):
            """A step whose copies are too small to hide (decode): everything on the
            compute stream, with no cross-stream events."""
            hs = host[i % n_layers]
            if graphs is not None:  # the graphs read their layer's own input buffers
                for k in in_keys:
                    layers[i % n_layers][k].copy_(hs[k], non_blocking=True)
                graphs[i % n_layers].replay()
                out_host.copy_(graph_out[i % n_layers], non_blocking=True)
                return
            L = dict(layers[i % n_layers])
            for k in in_keys:
                d_in[0][k].copy_(hs[k], non_blocking=True)
            L.update(d_in[0])
            gx = step(L, out_buf=d_out[0])
            out_host.copy_(d_out[0], non_blocking=True)
            if bwd:
                gx_host.copy_(gx, non_blocking=True)

        def e2e_run(n):
            if h2d + d2h < (1 << 20):
                for i in range(n):
                    e2e_step_inline(i)
                return
            for b in range(nbuf):  # every buffer starts free
                in_free[b].record(stream)
                out_free[b].record(stream)
            e2e_inputs(0)
            for i in range(n):
                if i + 1 < n:
                    e2e_inputs(i + 1)
                e2e_compute(i)
            stream.wait_event(out_free[(n - 1) % nbuf])

        e2e_run(args.warmup)
        torch.cuda.synchronize()
        barrier(world)
        e0, e1 = ev(), ev()
        e0.record(stream)
        e2e_run(args.steps)
        e1.record(stream)
        torch.cuda.synchronize()
        e2e_ms = max_over_ranks(e0.elapsed_time(e1), world)

    # ---- roofline of the dominant step (the experts' two grouped GEMM launches)
    hbm, bf16_burst, bf16_sust, src = peaks()
    work = [algorithmic(cfg, L["counts"], r[0], r[1], C, cfg.backward, fp8, gather, fused_topk)
            for L, r in zip(layers, rows)]
    mean = lambda key: float(np.mean([w[key] for w in work]))
    # per-step averages over the timed steps (layer i % n_layers)
    steps_w = [work[i % n_layers] for i in range(args.steps)]
    ex_us = 1e3 * float(np.mean(per["experts"]))
    ex_bytes = float(np.mean([w["experts_bytes"] for w in steps_w]))
    ex_flops = float(np.mean([w["experts_flops"] for w in steps_w]))
    if bwd:  # the dominant work is the experts' forward + backward GEMMs
        ex_us += 1e3 * float(np.mean(per["experts_bwd"]))
        ex_bytes += float(np.mean([w["experts_bwd_bytes"] for w in steps_w]))
        ex_flops += float(np.mean([w["experts_bwd_flops"] for w in steps_w]))
    t_hbm = ex_bytes / (hbm * 1e9)
    # with fp8, the gate/up GEMM (2/3 of the flops) runs at twice the bf16 rate
    # (the nominal 4.5 : 2.25 PFLOP/s ratio applied to the measured bf16 peak)
    tc_peak = bf16_burst * (1.0 / (2.0 / 3.0 / 2.0 + 1.0 / 3.0)) if fp8 else bf16_burst
    t_tc = ex_flops / (tc_peak * 1e12)
    if t_hbm >= t_tc:
        roof = {"bound": "hbm", "achieved": ex_bytes / (ex_us * 1e-6) / 1e9, "peak": hbm, "unit": "GB/s"}
    else:
        roof = {"bound": "tensor", "achieved": ex_flops / (ex_us * 1e-6) / 1e12, "peak": tc_peak, "unit": "TFLOP/s"}
    roof["frac"] = roof["achieved"] / roof["peak"]
    roof["traffic"] = None if (bwd or fp8 or gather) else profiled_traffic(cfg.name)
    roof["traffic_source"] = (PROFILED_TRAFFIC[cfg.name]["profile"] + " (ncu dram__bytes_read.sum + "
                              "dram__bytes_write.sum of the two launches; reported while the kernel "
                              "sources still hash to the profiled ones)") if roof["traffic"] else None
    roof["algorithmic_bytes"] = ex_bytes
    roof["kernel"] = experts_kernel_label(cfg, fp8, gather, bwd)
    roof["peak_source"] = src
    roof["tensor_frac_of_burst"] = ex_flops / (ex_us * 1e-6) / 1e12 / bf16_burst

    disp_us = 1e3 * float(np.mean(per["dispatch"]))
    comb_us = 1e3 * float(np.mean(per["combine"]))
    kernels = {
        "multihot_us": 1e3 * float(np.mean(per["multihot"])),
        "dispatch_us": disp_us,
        "experts_us": ex_us,
        "combine_us": comb_us,
        "dispatch_GBs": float(np.mean([w["dispatch_bytes"] for w in steps_w])) / (disp_us * 1e-6) / 1e9,
        "combine_GBs": float(np.mean([w["combine_bytes"] for w in steps_w])) / (comb_us * 1e-6) / 1e9,
        "experts_TFLOPs": ex_flops / (ex_us * 1e-6) / 1e12,
        **({k + "_us": 1e3 * float(np.mean(per[k])) for k in stages[4:]} if bwd else {}),
        "rows_used": [r[0] for r in rows], "rows_valid": [r[1] for r in rows], "capacity": C,
    }
    kernels["dispatch_frac_hbm"] = kernels["dispatch_GBs"] / hbm
    if sf_us is not None:
        sf_bytes = float(np.mean([algorithmic(cfg, w_l["counts"], r[0], r[1], worst, False, fp8, gather,
                                              fused_topk)["dispatch_bytes"]
                                  for w_l, r in zip(layers, rows)]))
        kernels["dispatch_sync_free_us"] = float(np.mean(sf_us))
        kernels["dispatch_sync_free_GBs"] = sf_bytes / (kernels["dispatch_sync_free_us"] * 1e-6) / 1e9
        kernels["dispatch_sync_free_frac_hbm"] = kernels["dispatch_sync_free_GBs"] / hbm
    kernels["combine_frac_hbm"] = kernels["combine_GBs"] / hbm
    kernels["experts_frac_bf16_burst"] = kernels["experts_TFLOPs"] / bf16_burst
    kernels["experts_frac_bf16_sustained"] = kernels["experts_TFLOPs"] / bf16_sust
    kernels["multihot_dispatch_us"] = kernels["multihot_us"] + kernels["dispatch_us"]
    kernels["dispatch_includes_multihot"] = fused_topk

    tokens = T * world * args.steps
    e2e = None
    if e2e_ms is not None:
        inline = h2d + d2h < (1 << 20)
        e2e = {"value": tokens / (e2e_ms * 1e-3), "unit": "tokens/s",
               "h2d_bytes_per_step": h2d, "d2h_bytes_per_step": d2h,
               "ms_per_step": e2e_ms / args.steps,
               "copies": ("on the compute stream: each step's input copies, layer and output read-back "
                          "run one after the other, so ms_per_step is the per-call latency" if inline else
                          "own streams, double-buffered: a step's copies overlap the neighbouring steps' "
                          "compute, so ms_per_step is pipelined throughput, not the latency of one call")}
    res = {
        "metric": "MoE layer tokens/sec (dispatch+experts+combine)" + (", forward + backward" if bwd else "")
                  + (", FP8 dispatch and gate/up GEMM" if fp8 else "")
                  + (", dispatch fused into the gate/up GEMM" if gather else ""),
        "value": T * world / (ms_step_max * 1e-3),
        "unit": "tokens/s",
        "n_gpus": world, "steps": args.steps, "warmup": args.warmup,
        "ms_per_step": ms_step_max,
        "higher_is_better": True,
        "scaling": "weak",
        "vs_baseline": None,
        "dtype": "e4m3 dispatch + gate/up, bf16 down" if fp8 else "bf16",
        "data": "synthetic (seeded N(0,1) tokens, softmax top-k routing, N(0,0.02) weights)",
        "config": {"workload": cfg.name, "T": T, "H": H, "E": E, "top_k": K, "I": I,
                   "pad_multiple": P, **({"fp8": "e4m3, one fp32 scale per row (tokens, W1 channels)"} if fp8 else {}),
                   "mode": "host-synced" if host_sync else "sync-free, CUDA graph replay (the cycled layers in one graph)",
                   "layers_cycled": n_layers, "l2": "inputs larger than L2 (4 distinct layers cycled, >1.2 GB weights each)",
                   "parallelism": "replicas" if world > 1 else "single GPU"},
        "timing": {"method": f"the {args.steps} timed steps in {windows['n']} consecutive windows, one CUDA "
                             "event pair each; ms_per_step is the median window's",
                   "windows": windows, "all_steps_ms_per_step": ms_max / args.steps},
        "e2e": e2e,
        "gpu_launches": launches_per_step * args.steps,
        "roofline": roof,
        "kernels": kernels,
    }
    res["clocks"] = clk.summary(n_timed_samples)
    res["clocks_extended"] = dict(clk.summary(), window=f"the timed region and {CLOCK_EXTRA_S} s of the same "
                                                         "steps repeated right after it, untimed")
    return res


# ----------------------------------------------------------------------------- the oracle on the CPU

def oracle_sample(cfg, budget_s: float, rank: int = 0):
    """Times the CPU oracle on the first tokens of one layer of ``cfg``,
    growing the sample until it takes about ``budget_s``.  Returns
    (tokens/s, tokens sampled, seconds, threads)."""
    import oracle as O
    s = cfg.seed + 104729 * rank
    x = synthetic.make_tokens(cfg.T, cfg.H, s)
    idx, p = synthetic.make_routing(cfg.T, cfg.E, cfg.K, s, cfg.zipf_s, cfg.drop)
    W1, W2 = synthetic.make_weights(cfg.E, cfg.H, cfg.I, s)
    b = lambda t: t.contiguous().view(torch.int16).numpy().view(np.uint16)
    xb, W1b, W2b = b(x), b(W1), b(W2)
    # calibrate on a small sample, then run one sample sized to take ~budget_s
    n = min(cfg.T, 16)
    while True:
        t0 = time.perf_counter()
        O.layer_forward(xb[:n], idx[:n].numpy(), p[:n].numpy(), W1b, W2b, cfg.I, cfg.P)
        dt = time.perf_counter() - t0
        if dt >= budget_s / 8 or n >= cfg.T:
            break
        n = min(cfg.T, n * 4)
    if n < cfg.T and dt < budget_s * 0.7:
        n = min(cfg.T, max(n, int(n * budget_s / max(dt, 1e-3))))
        t0 = time.perf_counter()
        O.layer_forward(xb[:n], idx[:n].numpy(), p[:n].numpy(), W1b, W2b, cfg.I, cfg.P)
        dt = time.perf_counter() - t0
    threads = torch.get_num_threads()
    try:
        import threadpoolctl
        info = threadpoolctl.threadpool_info()
        threads = max([i.get("num_threads", 1) for i in info] + [1])
    except Exception:
        pass
    return n / dt, n, dt, threads


def run_reference(args, world, rank):
    cfg = synthetic.CONFIGS[args.config]
    if rank != 0:
        return None
    vals = []
    for i in range(args.warmup + args.steps):
        v, n, dt, threads = oracle_sample(cfg, budget_s=args.ref_budget)
        if i >= args.warmup:
            vals.append((v, n, dt))
    v = float(np.median([a for a, _, _ in vals]))
    n = vals[0][1]
    dt = float(np.mean([c for _, _, c in vals]))
    return {
        "impl": "reference",
        "metric": "MoE layer tokens/sec (dispatch+experts+combine)",
        "value": v, "unit": "tokens/s", "n_gpus": world, "steps": args.steps, "warmup": args.warmup,
        "ms_per_step": dt * 1e3, "higher_is_better": True, "scaling": "weak", "vs_baseline": None,
        "dtype": "f64", "data": "synthetic",
        "config": {"workload": cfg.name, "T": cfg.T, "H": cfg.H, "E": cfg.E, "top_k": cfg.K,
                   "I": cfg.I, "pad_multiple": cfg.P},
        "cpu_baseline": {"value": v, "unit": "tokens/s", "cores": threads, "kind": "oracle",
                         "sample": f"first {n} tokens of the {cfg.name} layer (all {cfg.E} experts' weights), per step"},
        "e2e": {"value": v, "unit": "tokens/s", "h2d_bytes_per_step": 0, "d2h_bytes_per_step": 0},
    }


def target_leg(args, world, rank, local):
    """The Qwen3-30B-A3B layer at T = 16384 (host-synced, four layers cycled,
    five windows of four steps), device-timed only: the experts' TFLOP/s and
    fractions of the measured bf16 peaks, the dispatch's and combine's GB/s and
    fractions of the measured HBM copy bandwidth."""
    a = argparse.Namespace(**vars(args))
    a.config, a.steps, a.warmup, a.layers = "qwen3_30b_a3b_16k", 20, 4, 4
    r = run_ours(a, world, rank, local, leg=True)
    k = r["kernels"]
    keep = ("multihot_us", "dispatch_us", "experts_us", "combine_us", "dispatch_GBs", "dispatch_frac_hbm",
            "combine_GBs", "combine_frac_hbm", "experts_TFLOPs", "experts_frac_bf16_burst",
            "experts_frac_bf16_sustained", "multihot_dispatch_us")
    return {"workload": r["config"]["workload"], "T": r["config"]["T"], "tokens_per_s": r["value"],
            "ms_per_step": r["ms_per_step"], "steps": a.steps, "windows_spread": r["timing"]["windows"]["spread"],
            **{x: k[x] for x in keep}, "experts_roofline": r["roofline"], "clocks": r["clocks"]}


def main():
    ap = argparse.ArgumentParser()
    ap.add_argument("--gpus", type=int, default=1)
    ap.add_argument("--steps", type=int, default=40)
    ap.add_argument("--warmup", type=int, default=5)
    ap.add_argument("--impl", choices=["ours", "reference"], default="ours")
    ap.add_argument("--config", default="qwen3_30b_a3b", choices=sorted(synthetic.CONFIGS))
    ap.add_argument("--layers", type=int, default=4)
    ap.add_argument("--gather", action="store_true",
                    help="fuse the dispatch copy into the gate/up GEMM (the layout alone, then "
                         "A rows gathered from the tokens)")
    ap.add_argument("--fp8", action="store_true",
                    help="run the FP8 dispatch and e4m3 gate/up GEMM instead of the bf16 ones")
    ap.add_argument("--cpu-budget", type=float, default=15.0, help="seconds of oracle work for cpu_baseline")
    ap.add_argument("--ref-budget", type=float, default=8.0, help="seconds of oracle work per reference step")
    ap.add_argument("--no-cpu-baseline", action="store_true")
    ap.add_argument("--no-target-leg", action="store_true",
                    help="skip the Qwen3-30B-A3B T=16384 leg of the default run")
    args = ap.parse_args()
    assert args.warmup >= 3 or args.impl == "reference", "at least 3 warm-up steps"
    world, rank, local = dist_setup(args.gpus)
    if args.impl == "reference":
        res = run_reference(args, world, rank)
    else:
        res = run_ours(args, world, rank, local)
        if args.config == "qwen3_30b_a3b" and not (args.fp8 or args.gather or args.no_target_leg):
            # the same shape at T = 16384, where the experts are tensor-bound
            # and the targets for the tensor and HBM fractions are set
            res["kernels"]["target_layer_T16384"] = target_leg(args, world, rank, local)
        if rank == 0 and world == 1 and not args.no_cpu_baseline:
            cfg = synthetic.CONFIGS[args.config]
            v, n, dt, threads = oracle_sample(cfg, budget_s=args.cpu_budget)
            res["cpu_baseline"] = {"value": v, "unit": "tokens/s", "cores": threads, "kind": "oracle",
                                   "sample": f"first {n} tokens of the {cfg.name} layer, all {cfg.E} experts' weights, {dt:.1f} s"}
    if rank == 0 and res is not None:
        print(json.dumps(res))
    if world > 1:
        import torch.distributed as dist
        dist.destroy_process_group()


if __name__ == "__main__":
    main()
