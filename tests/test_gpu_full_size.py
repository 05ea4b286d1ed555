"""Full-size forward parity on the large layers, in the benchmark's launch
configuration (host-synced dispatch, the same tile shapes the bench runs).

Layers ("Add the deepep expert-parallel implementation (huggingface/transformers
#49638)", Benchmarks: the 30b and h4096 shapes; the skewed routing of the
workload set):
  * skewed: T 16384, H 2048, E 128, top-8, I 768, a log-Zipf router bias and
    5 % dropped slots -- expert 0 receives about 15 k rows (120 tiles of 128)
    and one expert none;
  * qwen3_30b_a3b_16k: the 30b shape at T 16384, where the tensor-peak target
    applies;
  * h4096: T 16384, H 4096, E 128, top-8, I 1536, forward as its training
    step runs it (gate/up values and o saved).

Each check: every row of the largest expert and of the smallest non-empty
one, plus 512 seeded random rows, against the oracle (h and y within the GEMM
tolerance, x_disp bit for bit); the layer output of 256 random tokens against
the oracle's (all of their rows computed by the oracle); the whole combine bit
for bit against the oracle's combine of the GPU's y; and the rows that must not
be written (pad rows in inference, spare rows) still holding the NaN they were
filled with, while pad rows come out zero when the forward saves for the
backward.
"""
import numpy as np
import pytest
import torch

import oracle as O
import synthetic
from tests._util import assert_gemm_close, bits

pytestmark = pytest.mark.gpu
DEV = "cuda"
BF = torch.bfloat16


@pytest.fixture(scope="module")
def moe():
    assert torch.cuda.is_available(), "GPU tests need a GPU"
    import combine_topk_multihot_gb300 as m
    return m


def _forward(moe, cfg, save: bool):
    inp = synthetic.make_layer_inputs(cfg, device=DEV)
    T, H, E, K, I, P = cfg.T, cfg.H, cfg.E, cfg.K, cfg.I, cfg.P
    C = moe.worst_case_rows(T, E, K, P)
    lay = moe.Layout(T, E, K, P, C, device=DEV)
    rmap, probs, _ = moe.moe_route_to_multihot(inp["topk_idx"], inp["topk_probs"], E, lay.status)
    x_disp, rows = moe.moe_dispatch(inp["x"], rmap, probs, lay, host_sync=True)
    nan = lambda n: torch.full((C, n), float("nan"), dtype=BF, device=DEV)
    bufs = {"h": nan(I), "y": nan(H)}
    if save:
        bufs["o"], bufs["gu"] = nan(H), nan(2 * I)
    ex = moe.moe_grouped_experts(x_disp, lay, inp["W1"], inp["W2"], save_o=save, save_gu=save, out=bufs)
    out = moe.moe_combine(ex["y"], lay)
    torch.cuda.synchronize()
    assert int(lay.status.item()) == 0
    return inp, lay, x_disp, ex, out, rows


@pytest.mark.parametrize("name,save", [("skewed", False), ("qwen3_30b_a3b_16k", False), ("h4096", True)])
def test_forward_full_size_sampled(moe, name, save):
    cfg = synthetic.CONFIGS[name]
    T, H, E, K, I = cfg.T, cfg.H, cfg.E, cfg.K, cfg.I
    inp, L, x_disp, ex, out, (R, N) = _forward(moe, cfg, save)
    counts = L.tokens_per_expert.cpu().numpy()
    offs = L.offsets.cpu().numpy()
    rt = L.row_token.cpu().numpy()
    re = L.row_expert.cpu().numpy()
    tr = L.token_row.cpu().numpy().reshape(T, K)
    assert (R, N) == (int(offs[E]), int(counts.sum()))
    nz = np.flatnonzero(counts)
    big, small = int(nz[np.argmax(counts[nz])]), int(nz[np.argmin(counts[nz])])
    if name == "skewed":
        # the bias makes expert 0 the overloaded one; some expert gets nothing
        assert big == 0 and counts[0] > 100 * 128 and (counts == 0).any()
    rng = np.random.default_rng(17)
    toks = np.sort(rng.choice(T, 256, replace=False))
    tok_rows = tr[toks][tr[toks] >= 0]
    rows = np.unique(np.concatenate([np.arange(offs[big], offs[big] + counts[big]),
                                     np.arange(offs[small], offs[small] + counts[small]),
                                     rng.choice(np.flatnonzero(rt >= 0), 512, replace=False),
                                     tok_rows]))
    xd = bits(x_disp[torch.as_tensor(rows)])
    assert np.array_equal(xd, bits(inp["x"])[rt[rows]])
    # the oracle on the sampled rows (a compact copy, so it touches only them)
    y, h, _ = O.grouped_experts(xd, re[rows], L.row_weight.cpu().numpy()[rows], bits(inp["W1"]),
                                bits(inp["W2"]), I)
    sel = torch.as_tensor(rows)
    assert_gemm_close(bits(ex["h"][sel]), h, f"{name} h", intermediate=True)
    assert_gemm_close(bits(ex["y"][sel]), y, f"{name} y")
    # the layer output of the sampled tokens: the oracle's combine of its own y
    y_full = np.zeros((L.capacity, H), np.uint16)
    y_full[rows] = y
    assert_gemm_close(bits(out)[toks], O.combine(y_full, tr[toks]), f"{name} out")
    # the whole combine, bit for bit, on the GPU's y
    y_gpu = bits(ex["y"]).copy()
    y_gpu[rt < 0] = 0
    assert np.array_equal(bits(out), O.combine(y_gpu, tr))
    # rows that are not valid: pad rows inside the groups, spare rows after R
    pad = (re == E) & (np.arange(L.capacity) < R)
    spare = np.arange(L.capacity) >= R
    yv, hv = ex["y"].float(), ex["h"].float()
    assert torch.isnan(yv[torch.as_tensor(spare)]).all() and torch.isnan(hv[torch.as_tensor(spare)]).all()
    padt = torch.as_tensor(pad)
    if save:
        for k in ("y", "h", "o", "gu"):
            assert (ex[k][padt] == 0).all(), f"{name}: pad rows of {k} are not zero"
    else:
        assert torch.isnan(yv[padt]).all() and torch.isnan(hv[padt]).all()
    assert not torch.isnan(yv[torch.as_tensor(rt >= 0)]).any()
