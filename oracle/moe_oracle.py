"""The MoE layer's hot path, step by step, on the CPU.  Test infrastructure only.

Notation: T tokens, H hidden, E experts, K top-k slots, I SwiGLU intermediate
size, P pad_multiple, C buffer rows.  The sentinel expert id is E.

Page citations:
  [HEP]  "feat: add hybridep (NVIDIA-NeMo/Automodel #1333)"
  [DEP]  "Add the deepep expert-parallel implementation (huggingface/transformers #49638)"

Readings taken where the pages are silent (each is pinned by a test):
  * a duplicate expert index in one token's top-k sets the multihot entry once;
    the slots are visited in order, so the prob (and the slot that receives the
    gradient) is the last valid duplicate's;
  * an index outside [-1, E) is an error, not a silent drop;
  * tokens_per_expert are exact counts; each expert's group is padded up to a
    multiple of P (an empty expert gets no rows); offsets are the prefix sum of
    the padded counts;
  * inside an expert's group the rows are in ascending token order; pad rows
    and spare rows hold token -1, the sentinel expert, weight 0 and x = 0;
  * a token's rows are summed in ascending expert order (= ascending row), in
    fp32 from +0.0, then rounded once to bf16;
  * the routing weight multiplies the fp32 down-projection accumulator, and the
    product is rounded once to bf16; the SwiGLU activation h is rounded to bf16
    between the two expert GEMMs;
  * W1 is [E, 2I, H] with the gate rows first, W2 is [E, H, I];
  * weight gradients are accumulated and returned in fp32.
"""
from __future__ import annotations

import numpy as np

from .bf16 import (bf16_bits_to_f32, bf16_bits_to_f64, bf16_round_f64,
                   f32_to_bf16_bits, f64_to_bf16_bits)


class OracleIndexError(ValueError):
    """An expert index outside [-1, E)."""


class OracleCapacityError(ValueError):
    """The rows the layout needs exceed the buffer's capacity."""


def sentinel_expert(E: int) -> int:
    """Spare and pad rows are routed to expert id E, which the experts skip
    ([DEP] What this adds, Eager vs captured)."""
    return E


def worst_case_capacity(T: int, E: int, K: int, P: int) -> int:
    """Rows a sync-free buffer needs for any routing: all T*K slots valid, and
    every expert's group padded by at most P-1 rows ([DEP] Eager vs captured:
    the sync-free buffer holds enough rows for any routing)."""
    return T * K + E * (P - 1)


# --------------------------------------------------------------------------
# a1: top-k -> multihot   ([HEP] Changelog: the HybridEP preprocessing step
# that maps top-k indices to multihot routing data; review of dispatch():
# probs are fp32)
# --------------------------------------------------------------------------
def route_to_multihot(topk_idx: np.ndarray, topk_probs: np.ndarray, E: int):
    """Returns routing_map uint8 [T, E], probs fp32 [T, E], winner_slot int8 [T, E].

    Slots are visited in order k = 0..K-1; a -1 slot is dropped; a valid slot
    sets routing_map[t, e] = 1, probs[t, e] = its prob and winner_slot[t, e] = k,
    so a later duplicate of the same expert overwrites an earlier one.
    winner_slot is -1 where routing_map is 0.
    """
    idx = np.asarray(topk_idx, dtype=np.int64)
    p = np.asarray(topk_probs, dtype=np.float32)
    T, K = idx.shape
    if ((idx < -1) | (idx >= E)).any():
        raise OracleIndexError("expert index outside [-1, E)")
    routing_map = np.zeros((T, E), dtype=np.uint8)
    probs = np.zeros((T, E), dtype=np.float32)
    winner = np.full((T, E), -1, dtype=np.int8)
    tokens = np.arange(T)
    for k in range(K):
        e = idx[:, k]
        ok = e >= 0
        routing_map[tokens[ok], e[ok]] = 1
        probs[tokens[ok], e[ok]] = p[ok, k]
        winner[tokens[ok], e[ok]] = k
    return routing_map, probs, winner


# --------------------------------------------------------------------------
# a2: tokens_per_expert, padded offsets   ([HEP] review of dispatch():
# tokens_per_expert, num_permuted_tokens = tokens_per_expert.sum(), pad_multiple)
# --------------------------------------------------------------------------
def counts_and_offsets(routing_map: np.ndarray, P: int):
    """Returns (tokens_per_expert int64 [E], offsets int64 [E+1]).

    tokens_per_expert[e] = number of tokens routed to e (exact);
    padded[e] = the smallest multiple of P that is >= tokens_per_expert[e];
    offsets[0] = 0, offsets[e+1] = offsets[e] + padded[e].
    """
    if P < 1:
        raise ValueError("pad_multiple must be >= 1")
    counts = np.asarray(routing_map, dtype=np.int64).sum(axis=0)
    padded = ((counts + P - 1) // P) * P
    offsets = np.zeros(counts.shape[0] + 1, dtype=np.int64)
    offsets[1:] = np.cumsum(padded)
    return counts, offsets


# --------------------------------------------------------------------------
# a3: the expanded layout   ([DEP] What this adds, Expanded layout; Eager vs
# captured for the spare rows and the sentinel expert)
# --------------------------------------------------------------------------
def build_layout(routing_map: np.ndarray, probs: np.ndarray, K: int, P: int,
                 capacity: int | None = None):
    """The expanded layout: one row per (token, expert) pair, grouped by expert.

    Returns a dict with
      tokens_per_expert [E], offsets [E+1], rows_used R = offsets[E],
      rows_valid N = sum(tokens_per_expert), capacity C,
      row_token int32 [C]   (-1 on pad / spare rows),
      row_expert int32 [C]  (the sentinel E on pad / spare rows),
      row_weight fp32 [C]   (probs[t, e]; 0 on pad / spare rows),
      token_row int32 [T, K] (token t's rows in ascending expert order, then -1).
    With ``capacity=None`` the buffer is exactly R rows (host-synced mode).
    """
    routing_map = np.asarray(routing_map, dtype=np.uint8)
    probs = np.asarray(probs, dtype=np.float32)
    T, E = routing_map.shape
    counts, offsets = counts_and_offsets(routing_map, P)
    R = int(offsets[E])
    C = R if capacity is None else int(capacity)
    if R > C:
        raise OracleCapacityError(f"layout needs {R} rows, capacity is {C}")
    SENT = sentinel_expert(E)
    row_token = np.full(C, -1, dtype=np.int32)
    row_expert = np.full(C, SENT, dtype=np.int32)
    row_weight = np.zeros(C, dtype=np.float32)
    row_of = np.full((T, E), -1, dtype=np.int64)      # row of the pair (t, e)
    for e in range(E):
        toks = np.flatnonzero(routing_map[:, e])       # ascending token order
        rows = offsets[e] + np.arange(toks.size)
        row_token[rows] = toks
        row_expert[rows] = e
        row_weight[rows] = probs[toks, e]
        row_of[toks, e] = rows
    token_row = np.full((T, K), -1, dtype=np.int32)
    for t in range(T):
        experts = np.flatnonzero(routing_map[t])        # ascending expert order
        if experts.size > K:
            raise ValueError("a token cannot have more experts than top-k slots")
        token_row[t, :experts.size] = row_of[t, experts]
    return {
        "tokens_per_expert": counts, "offsets": offsets, "rows_used": R,
        "rows_valid": int(counts.sum()), "capacity": C,
        "row_token": row_token, "row_expert": row_expert,
        "row_weight": row_weight, "token_row": token_row,
    }


# --------------------------------------------------------------------------
# a4 / a7: dispatch (and the combine's backward, which is the same gather)
# --------------------------------------------------------------------------
def dispatch(x_bits: np.ndarray, row_token: np.ndarray) -> np.ndarray:
    """x_disp[r] = x[row_token[r]] bit for bit; rows with token -1 are zero.
    ([DEP] Expanded layout; Eager vs captured: spare rows hold zeros)."""
    x_bits = np.asarray(x_bits, dtype=np.uint16)
    row_token = np.asarray(row_token)
    out = np.zeros((row_token.shape[0], x_bits.shape[1]), dtype=np.uint16)
    ok = row_token >= 0
    out[ok] = x_bits[row_token[ok]]
    return out


# --------------------------------------------------------------------------
# a5: SwiGLU experts that apply the routing weight   ([DEP] Expanded layout:
# the routing weight is applied inside the experts; Benchmarks: the experts
# are bf16 grouped GEMMs)
# --------------------------------------------------------------------------
def _silu(z: np.ndarray) -> np.ndarray:
    with np.errstate(over="ignore"):
        return z / (1.0 + np.exp(-z))


def expert_forward_f64(X, W1e, W2e, w, I, rnd=bf16_round_f64):
    """One expert on its rows, in fp64.

    X [n, H], W1e [2I, H] (gate rows 0..I-1, up rows I..2I-1), W2e [H, I],
    w [n] routing weights.  g = X W_gate^T, u = X W_up^T, h = rnd(silu(g) * u),
    o = h W2e^T, y = rnd(w * o).  Returns (y, h, o) in fp64, o unrounded.
    ``rnd`` is the rounding the layer applies (bf16); pass the identity to get
    the exact real-valued function.
    """
    g = X @ W1e[:I].T
    u = X @ W1e[I:].T
    h = rnd(_silu(g) * u)
    o = h @ W2e.T
    y = rnd(np.asarray(w, dtype=np.float64)[:, None] * o)
    return y, h, o


def grouped_experts(x_disp_bits, row_expert, row_weight, W1_bits, W2_bits, I,
                    rows=None):
    """Apply each row's expert.  Returns (y_bits [C, H], h_bits [C, I],
    o_bits [C, H]); sentinel rows are skipped and stay zero.  ``rows``
    optionally restricts the work to a subset of row indices."""
    x_disp_bits = np.asarray(x_disp_bits, dtype=np.uint16)
    row_expert = np.asarray(row_expert)
    C, H = x_disp_bits.shape
    E = W1_bits.shape[0]
    y = np.zeros((C, H), dtype=np.uint16)
    hb = np.zeros((C, I), dtype=np.uint16)
    ob = np.zeros((C, H), dtype=np.uint16)
    sel = np.zeros(C, dtype=bool)
    if rows is None:
        sel[:] = True
    else:
        sel[np.asarray(rows)] = True
    for e in range(E):
        R_e = np.flatnonzero((row_expert == e) & sel)
        if R_e.size == 0:
            continue
        ye, he, oe = expert_forward_f64(bf16_bits_to_f64(x_disp_bits[R_e]),
                                        bf16_bits_to_f64(W1_bits[e]),
                                        bf16_bits_to_f64(W2_bits[e]),
                                        np.asarray(row_weight)[R_e], I)
        y[R_e] = f64_to_bf16_bits(ye)
        hb[R_e] = f64_to_bf16_bits(he)
        ob[R_e] = f64_to_bf16_bits(oe)
    return y, hb, ob


# --------------------------------------------------------------------------
# a6 / a10: combine (and the dispatch's backward)   ([DEP] Expanded layout:
# the combine is a plain sum, with no weights)
# --------------------------------------------------------------------------
def combine(y_bits: np.ndarray, token_row: np.ndarray) -> np.ndarray:
    """out[t] = bf16( ((0 + y[r_0]) + y[r_1]) + ... ) with fp32 adds over the
    token's rows r_j = token_row[t, j] in order j = 0, 1, ...; no weights.
    A token with no rows gives +0."""
    y_bits = np.asarray(y_bits, dtype=np.uint16)
    token_row = np.asarray(token_row)
    T, K = token_row.shape
    acc = np.zeros((T, y_bits.shape[1]), dtype=np.float32)
    for j in range(K):
        r = token_row[:, j]
        ok = r >= 0
        acc[ok] = acc[ok] + bf16_bits_to_f32(y_bits[r[ok]])
    return f32_to_bf16_bits(acc)


def combine_backward(grad_out_bits: np.ndarray, row_token: np.ndarray) -> np.ndarray:
    """d out / d y: grad_y[r] = grad_out[row_token[r]], zero on pad / spare
    rows ([DEP] Training: the combine's gradient is a dispatch that follows
    the forward's layout)."""
    return dispatch(grad_out_bits, row_token)


# --------------------------------------------------------------------------
# a8: routing-weight gradient   ([DEP] Training: the routing weights receive
# gradients too)
# --------------------------------------------------------------------------
def routing_weight_grad(grad_y_bits, o_bits, row_expert, E) -> np.ndarray:
    """y_r = w_r * o_r, so dL/dw_r = sum_h grad_y[r, h] * o[r, h] (fp64 sum,
    returned as fp32); zero on sentinel rows.  o is the saved pre-weight
    down-projection output."""
    gy = bf16_bits_to_f64(grad_y_bits)
    o = bf16_bits_to_f64(o_bits)
    gw = np.sum(gy * o, axis=1)
    gw[np.asarray(row_expert) >= E] = 0.0
    return gw.astype(np.float32)


# --------------------------------------------------------------------------
# a9: expert backward   ([DEP] What this adds, Training: the gradients reach
# the tokens and the weights through the experts).  The chain rule of the
# forward above, written out in fp64 with no rounding anywhere: the forward's
# bf16 roundings (h, y) are steps of a rounding function whose derivative is
# taken as one, as autograd does, and the forward's saved bf16 h enters
# dW2 as the value the forward produced.
# --------------------------------------------------------------------------
def backward_scale(GY, w):
    """G_o = w * GY: y = w o, so dL/do = w dL/dy."""
    return np.asarray(w, dtype=np.float64)[:, None] * GY


def backward_gate_up(X, W1e, I):
    """The forward's gate and up pre-activations: g = X Wg^T, u = X Wu^T."""
    return X @ W1e[:I].T, X @ W1e[I:].T


def _sigmoid(z):
    with np.errstate(over="ignore"):
        return 1.0 / (1.0 + np.exp(-z))


def backward_swiglu(G_o, W2e, g, u):
    """G_h = G_o W2;  G_g = G_h * u * silu'(g),  G_u = G_h * silu(g) with
    silu'(g) = s (1 + g (1 - s)), s = sigmoid(g).  Returns [G_g | G_u]."""
    return expert_backward_steps_from(G_o, W2e, g, u)["G_gu"]


def expert_backward_steps_from(G_o, W2e, g, u):
    """The SwiGLU part of the chain rule, every intermediate kept."""
    G_h = G_o @ W2e
    s = _sigmoid(g)
    silu = g * s
    dsilu = s * (1.0 + g * (1.0 - s))
    G_gu = np.concatenate([G_h * u * dsilu, G_h * silu], axis=1)
    return dict(G_h=G_h, s=s, silu=silu, dsilu=dsilu, G_gu=G_gu)


def backward_gemms(G_o, G_gu, X, h, W1e):
    """dX = G_gu W1;  dW1 = G_gu^T X;  dW2 = G_o^T h (exact fp64)."""
    return G_gu @ W1e, G_gu.T @ X, G_o.T @ h


def expert_backward_steps(X, h, GY, w, W1e, W2e, I):
    """Every step of one expert's chain rule, in fp64: G_o, g, u, G_h, the
    SwiGLU derivative terms, G_gu = [G_g | G_u], and dX, dW1, dW2."""
    G_o = backward_scale(GY, w)
    g, u = backward_gate_up(X, W1e, I)
    st = expert_backward_steps_from(G_o, W2e, g, u)
    dX, dW1, dW2 = backward_gemms(G_o, st["G_gu"], X, h, W1e)
    st.update(G_o=G_o, g=g, u=u, dX=dX, dW1=dW1, dW2=dW2)
    return st


def expert_backward_f64(X, h, GY, w, W1e, W2e, I):
    """Gradients of one expert's rows, in fp64.

    Forward: g = X Wg^T, u = X Wu^T, h = silu(g) u, o = h W2^T, y = w o.
    Given dL/dy = GY and the forward's h, the chain rule in four steps:
    backward_scale (G_o), backward_gate_up (g, u), backward_swiglu (G_gu =
    [G_g | G_u]), backward_gemms (dX, dW1, dW2); every product and sum is
    exact fp64.  Returns (dX [n, H], dW1 [2I, H], dW2 [H, I]).
    """
    st = expert_backward_steps(X, h, GY, w, W1e, W2e, I)
    return st["dX"], st["dW1"], st["dW2"]


def grouped_experts_backward(grad_y_bits, x_disp_bits, h_bits, row_expert,
                             row_weight, W1_bits, W2_bits, I):
    """Returns (grad_x_disp bits [C, H], dW1 fp32 [E, 2I, H], dW2 fp32 [E, H, I]).
    Sentinel rows get zero gradient and add nothing to dW."""
    grad_y_bits = np.asarray(grad_y_bits, dtype=np.uint16)
    row_expert = np.asarray(row_expert)
    C, H = grad_y_bits.shape
    E = W1_bits.shape[0]
    gx = np.zeros((C, H), dtype=np.uint16)
    dW1 = np.zeros((E, 2 * I, H), dtype=np.float32)
    dW2 = np.zeros((E, H, I), dtype=np.float32)
    for e in range(E):
        R_e = np.flatnonzero(row_expert == e)
        if R_e.size == 0:
            continue
        dX, d1, d2 = expert_backward_f64(bf16_bits_to_f64(x_disp_bits[R_e]),
                                         bf16_bits_to_f64(h_bits[R_e]),
                                         bf16_bits_to_f64(grad_y_bits[R_e]),
                                         np.asarray(row_weight)[R_e],
                                         bf16_bits_to_f64(W1_bits[e]),
                                         bf16_bits_to_f64(W2_bits[e]), I)
        gx[R_e] = f64_to_bf16_bits(dX)
        dW1[e] = d1.astype(np.float32)
        dW2[e] = d2.astype(np.float32)
    return gx, dW1, dW2


# --------------------------------------------------------------------------
# a10 + scatter of the weight gradient back to [T, E]
# --------------------------------------------------------------------------
def dispatch_backward(grad_x_disp_bits, token_row, grad_w=None, row_token=None,
                      row_expert=None, E=None):
    """grad_x[t] = sum of grad_x_disp over t's rows (the combine, applied to the
    gradient).  With grad_w given, also returns grad_probs fp32 [T, E]:
    grad_probs[t, e] = grad_w[row of (t, e)], 0 where t is not routed to e."""
    grad_x = combine(grad_x_disp_bits, token_row)
    if grad_w is None:
        return grad_x
    T = np.asarray(token_row).shape[0]
    grad_probs = np.zeros((T, E), dtype=np.float32)
    rt = np.asarray(row_token)
    ok = rt >= 0
    grad_probs[rt[ok], np.asarray(row_expert)[ok]] = np.asarray(grad_w, dtype=np.float32)[ok]
    return grad_x, grad_probs


def route_to_multihot_backward(grad_probs, topk_idx, winner_slot):
    """grad_topk_probs[t, k] = grad_probs[t, topk_idx[t, k]] when that slot is
    valid and is the slot that set the multihot entry, else 0."""
    idx = np.asarray(topk_idx, dtype=np.int64)
    gp = np.asarray(grad_probs, dtype=np.float32)
    win = np.asarray(winner_slot)
    T, K = idx.shape
    out = np.zeros((T, K), dtype=np.float32)
    tokens = np.arange(T)
    for k in range(K):
        e = idx[:, k]
        ok = e >= 0
        ok[ok] = win[tokens[ok], e[ok]] == k
        out[tokens[ok], k] = gp[tokens[ok], e[ok]]
    return out


# --------------------------------------------------------------------------
# The whole layer
# --------------------------------------------------------------------------
def layer_forward(x_bits, topk_idx, topk_probs, W1_bits, W2_bits, I, P,
                  capacity=None):
    """a1..a6 composed.  Returns a dict with every intermediate."""
    E = W1_bits.shape[0]
    K = np.asarray(topk_idx).shape[1]
    rmap, probs, winner = route_to_multihot(topk_idx, topk_probs, E)
    L = build_layout(rmap, probs, K, P, capacity)
    x_disp = dispatch(x_bits, L["row_token"])
    y, h, o = grouped_experts(x_disp, L["row_expert"], L["row_weight"], W1_bits, W2_bits, I)
    out = combine(y, L["token_row"])
    return dict(routing_map=rmap, probs=probs, winner_slot=winner, layout=L,
                x_disp=x_disp, y=y, h=h, o=o, out=out)


def layer_backward(fwd, grad_out_bits, W1_bits, W2_bits, topk_idx, I):
    """a7..a10 and the multihot backward, given ``layer_forward``'s dict."""
    L = fwd["layout"]
    E = W1_bits.shape[0]
    grad_y = combine_backward(grad_out_bits, L["row_token"])
    grad_w = routing_weight_grad(grad_y, fwd["o"], L["row_expert"], E)
    gxd, dW1, dW2 = grouped_experts_backward(grad_y, fwd["x_disp"], fwd["h"],
                                             L["row_expert"], L["row_weight"],
                                             W1_bits, W2_bits, I)
    grad_x, grad_probs = dispatch_backward(gxd, L["token_row"], grad_w,
                                           L["row_token"], L["row_expert"], E)
    grad_topk = route_to_multihot_backward(grad_probs, topk_idx, fwd["winner_slot"])
    return dict(grad_y=grad_y, grad_w=grad_w, grad_x_disp=gxd, dW1=dW1, dW2=dW2,
                grad_x=grad_x, grad_probs=grad_probs, grad_topk_probs=grad_topk)
