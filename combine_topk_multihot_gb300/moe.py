"""Python binding of the C ABI: argument marshalling only.

Every step of the path runs in the CUDA library; PyTorch only allocates the
device buffers and supplies the current stream.  The function names are the
C entry points' names.  Pages cited:

  [HEP] "feat: add hybridep (NVIDIA-NeMo/Automodel #1333)"
  [DEP] "Add the deepep expert-parallel implementation (huggingface/transformers #49638)"
"""
from __future__ import annotations

import ctypes
from dataclasses import dataclass
from typing import Optional

import torch

from . import _native as N


class MoEError(RuntimeError):
    def __init__(self, code: int, where: str):
        self.code = code
        super().__init__(f"{where}: {N.status_string(code)}: {N.last_error()}")


def _check(code: int, where: str):
    if code != N.MOE_OK:
        raise MoEError(code, where)


def _ptr(t: Optional[torch.Tensor]):
    if t is None:
        return None
    if not t.is_contiguous():
        raise ValueError("tensors passed to the library must be contiguous")
    return ctypes.c_void_p(t.data_ptr()) if t.numel() else None


def _stream(stream=None):
    s = stream if stream is not None else torch.cuda.current_stream()
    return ctypes.c_void_p(s.cuda_stream)


def _bf16(t: torch.Tensor, name: str) -> torch.Tensor:
    if t.dtype != torch.bfloat16:
        raise TypeError(f"{name} must be bfloat16")
    return t


def worst_case_rows(T: int, E: int, K: int, pad_multiple: int) -> int:
    return int(N.lib.moe_worst_case_rows(T, E, K, pad_multiple))


class Layout:
    """The expanded layout of one forward + backward, in caller-owned device
    buffers ([HEP]'s dispatch handle, made explicit; [DEP] Custom ops)."""

    def __init__(self, T: int, E: int, K: int, pad_multiple: int, capacity: int,
                 device="cuda", status: Optional[torch.Tensor] = None):
        dev = torch.device(device)
        i32 = dict(dtype=torch.int32, device=dev)
        self.T, self.E, self.K, self.pad_multiple, self.capacity = T, E, K, pad_multiple, capacity
        self.tokens_per_expert = torch.empty(E, **i32)
        self.offsets = torch.empty(E + 1, **i32)
        self.totals = torch.empty(2, **i32)
        self.row_token = torch.empty(capacity, **i32)
        self.row_expert = torch.empty(capacity, **i32)
        self.row_weight = torch.empty(capacity, dtype=torch.float32, device=dev)
        self.token_row = torch.empty(T * K, **i32)
        self.status = status if status is not None else torch.zeros(1, **i32)
        nbytes = ctypes.c_size_t(0)
        _check(N.lib.moe_layout_workspace_bytes(T, E, ctypes.byref(nbytes)), "moe_layout_workspace_bytes")
        self.workspace = torch.empty(nbytes.value, dtype=torch.uint8, device=dev)
        self.c = N.MoeLayout(
            T, E, K, pad_multiple, capacity,
            self.tokens_per_expert.data_ptr(), self.offsets.data_ptr(), self.totals.data_ptr(),
            self.row_token.data_ptr() if capacity else None,
            self.row_expert.data_ptr() if capacity else None,
            self.row_weight.data_ptr() if capacity else None,
            self.token_row.data_ptr() if T * K else None,
            self.status.data_ptr(), self.workspace.data_ptr())

    @property
    def ref(self):
        return ctypes.byref(self.c)

    # The buffers that later steps read.  The workspace is scratch for the
    # dispatch alone and is not part of this list.
    TENSOR_FIELDS = ("tokens_per_expert", "offsets", "totals", "row_token", "row_expert",
                     "row_weight", "token_row", "status")

    def tensors(self):
        """The layout's buffers in TENSOR_FIELDS order, to pass it between ops."""
        return tuple(getattr(self, f) for f in self.TENSOR_FIELDS)

    @classmethod
    def from_tensors(cls, T: int, E: int, K: int, pad_multiple: int, tensors,
                     workspace: Optional[torch.Tensor] = None) -> "Layout":
        """Rebuild a layout around the buffers of ``tensors()``.  Without a
        ``workspace`` it gets a 256-byte placeholder: enough for every call
        except moe_dispatch, which needs ``moe_layout_workspace_bytes``."""
        self = cls.__new__(cls)
        for f, t in zip(cls.TENSOR_FIELDS, tensors):
            setattr(self, f, t)
        self.workspace = (workspace if workspace is not None else
                          torch.empty(256, dtype=torch.uint8, device=self.status.device))
        self.T, self.E, self.K, self.pad_multiple = T, E, K, pad_multiple
        self.capacity = self.row_token.numel()
        C = self.capacity
        self.c = N.MoeLayout(
            T, E, K, pad_multiple, C,
            self.tokens_per_expert.data_ptr(), self.offsets.data_ptr(), self.totals.data_ptr(),
            self.row_token.data_ptr() if C else None, self.row_expert.data_ptr() if C else None,
            self.row_weight.data_ptr() if C else None,
            self.token_row.data_ptr() if T * K else None,
            self.status.data_ptr(), self.workspace.data_ptr())
        return self


def moe_router_topk(logits: torch.Tensor, K: int, multihot: bool = False, stream=None):
    """r0: softmax -> top-K -> renormalise.  Returns (topk_idx int64 [T, K],
    topk_probs fp32 [T, K]), plus (routing_map, probs, winner_slot) of the
    multihot step when ``multihot`` (written by the same kernel)."""
    T, E = logits.shape
    if logits.dtype != torch.float32:
        raise TypeError("logits must be float32")
    dev = logits.device
    idx = torch.empty(T, K, dtype=torch.int64, device=dev)
    w = torch.empty(T, K, dtype=torch.float32, device=dev)
    mh = (torch.empty(T, E, dtype=torch.uint8, device=dev), torch.empty(T, E, dtype=torch.float32, device=dev),
          torch.empty(T, E, dtype=torch.int8, device=dev)) if multihot else (None, None, None)
    _check(N.lib.moe_router_topk(_ptr(logits), T, E, K, _ptr(idx), _ptr(w), _ptr(mh[0]), _ptr(mh[1]),
                                 _ptr(mh[2]), _stream(stream)), "moe_router_topk")
    return (idx, w) + (mh if multihot else ())


def moe_router_topk_backward(grad_topk_probs: torch.Tensor, topk_probs: torch.Tensor,
                             topk_idx: torch.Tensor, E: int, stream=None):
    """r0 backward: grad_logits fp32 [T, E]."""
    T, K = topk_idx.shape
    g = torch.empty(T, E, dtype=torch.float32, device=topk_idx.device)
    _check(N.lib.moe_router_topk_backward(_ptr(grad_topk_probs), _ptr(topk_probs), _ptr(topk_idx), T, E, K,
                                          _ptr(g), _stream(stream)), "moe_router_topk_backward")
    return g


def moe_route_to_multihot(topk_idx: torch.Tensor, topk_probs: torch.Tensor, E: int,
                          status: torch.Tensor, stream=None):
    """a1: returns (routing_map uint8 [T,E], probs fp32 [T,E], winner_slot int8 [T,E])."""
    T, K = topk_idx.shape
    assert topk_idx.dtype == torch.int64 and topk_probs.dtype == torch.float32
    dev = topk_idx.device
    routing_map = torch.empty(T, E, dtype=torch.uint8, device=dev)
    probs = torch.empty(T, E, dtype=torch.float32, device=dev)
    winner = torch.empty(T, E, dtype=torch.int8, device=dev)
    _check(N.lib.moe_route_to_multihot(_ptr(topk_idx), _ptr(topk_probs), T, K, E,
                                       _ptr(routing_map), _ptr(probs), _ptr(winner),
                                       _ptr(status), _stream(stream)), "moe_route_to_multihot")
    return routing_map, probs, winner


def moe_dispatch(x: torch.Tensor, routing_map: torch.Tensor, probs: torch.Tensor, layout: Layout,
                 host_sync: bool = True, x_disp: Optional[torch.Tensor] = None, stream=None):
    """a2-a4: fills ``layout`` and returns (x_disp [C, H], (R, N) or None)."""
    _bf16(x, "x")
    H = x.shape[1]
    if x_disp is None:
        x_disp = torch.empty(layout.capacity, H, dtype=torch.bfloat16, device=x.device)
    rows = (ctypes.c_int64 * 2)() if host_sync else None
    _check(N.lib.moe_dispatch(_ptr(x), _ptr(routing_map), _ptr(probs), H, layout.ref,
                              _ptr(x_disp), rows, _stream(stream)), "moe_dispatch")
    return x_disp, ((int(rows[0]), int(rows[1])) if host_sync else None)


def moe_dispatch_topk(x: torch.Tensor, topk_idx: torch.Tensor, topk_probs: torch.Tensor, layout: Layout,
                      host_sync: bool = True, x_disp: Optional[torch.Tensor] = None, multihot=None,
                      stream=None):
    """a1-a4 in one call: the multihot step and the dispatch from the top-k
    choices.  Returns (x_disp [C, H], (routing_map, probs, winner_slot),
    (R, N) or None); ``multihot`` optionally gives the three output buffers."""
    _bf16(x, "x")
    assert topk_idx.dtype == torch.int64 and topk_probs.dtype == torch.float32
    T, H = x.shape
    E = layout.E
    dev = x.device
    if x_disp is None:
        x_disp = torch.empty(layout.capacity, H, dtype=torch.bfloat16, device=dev)
    if multihot is None:
        multihot = (torch.empty(T, E, dtype=torch.uint8, device=dev), torch.empty(T, E, dtype=torch.float32, device=dev),
                    torch.empty(T, E, dtype=torch.int8, device=dev))
    rows = (ctypes.c_int64 * 2)() if host_sync else None
    _check(N.lib.moe_dispatch_topk(_ptr(x), _ptr(topk_idx), _ptr(topk_probs), H, layout.ref, _ptr(multihot[0]),
                                   _ptr(multihot[1]), _ptr(multihot[2]), _ptr(x_disp), rows, _stream(stream)),
           "moe_dispatch_topk")
    return x_disp, tuple(multihot), ((int(rows[0]), int(rows[1])) if host_sync else None)


def moe_dispatch_layout(routing_map: torch.Tensor, probs: torch.Tensor, layout: Layout,
                        host_sync: bool = True, stream=None):
    """a2-a3 alone (no rows copied): fills ``layout``; returns (R, N) or None."""
    rows = (ctypes.c_int64 * 2)() if host_sync else None
    _check(N.lib.moe_dispatch_layout(_ptr(routing_map), _ptr(probs), layout.ref, rows, _stream(stream)),
           "moe_dispatch_layout")
    return (int(rows[0]), int(rows[1])) if host_sync else None


def moe_grouped_experts_gather(x: torch.Tensor, layout: Layout, W1: torch.Tensor, W2: torch.Tensor,
                               save_o: bool = False, save_gu: bool = False, out=None, stream=None):
    """a4 fused into a5: the gate/up GEMM reads its rows from the tokens ``x``
    by the layout's row_token.  Returns dict(h, y, o, gu) as moe_grouped_experts."""
    _bf16(x, "x")
    E, twoI, H = W1.shape
    I = twoI // 2
    C = layout.capacity
    dev = x.device
    o = out or {}
    h = o.get("h") if o.get("h") is not None else torch.empty(C, I, dtype=torch.bfloat16, device=dev)
    y = o.get("y") if o.get("y") is not None else torch.empty(C, H, dtype=torch.bfloat16, device=dev)
    o_save = (o.get("o") if o.get("o") is not None else torch.empty(C, H, dtype=torch.bfloat16, device=dev)) if save_o else None
    gu = (o.get("gu") if o.get("gu") is not None else torch.empty(C, 2 * I, dtype=torch.bfloat16, device=dev)) if save_gu else None
    _check(N.lib.moe_grouped_experts_gather(_ptr(x), layout.ref, H, I, _ptr(W1), _ptr(W2), _ptr(h), _ptr(y),
                                            _ptr(o_save), _ptr(gu), _stream(stream)),
           "moe_grouped_experts_gather")
    return {"h": h, "y": y, "o": o_save, "gu": gu}


def moe_dispatch_fp8(x: torch.Tensor, routing_map: torch.Tensor, probs: torch.Tensor, layout: Layout,
                     host_sync: bool = True, out=None, stream=None):
    """a4 in e4m3: fills ``layout`` and returns (x_disp_q uint8 [C, H],
    x_disp_scale fp32 [C], (R, N) or None)."""
    _bf16(x, "x")
    H = x.shape[1]
    C = layout.capacity
    q = out[0] if out is not None else torch.empty(C, H, dtype=torch.uint8, device=x.device)
    sc = out[1] if out is not None else torch.empty(C, dtype=torch.float32, device=x.device)
    rows = (ctypes.c_int64 * 2)() if host_sync else None
    _check(N.lib.moe_dispatch_fp8(_ptr(x), _ptr(routing_map), _ptr(probs), H, layout.ref, _ptr(q), _ptr(sc),
                                  rows, _stream(stream)), "moe_dispatch_fp8")
    return q, sc, ((int(rows[0]), int(rows[1])) if host_sync else None)


def moe_dispatch_topk_fp8(x: torch.Tensor, topk_idx: torch.Tensor, topk_probs: torch.Tensor, layout: Layout,
                          host_sync: bool = True, out=None, multihot=None, stream=None):
    """a1-a4 in one call with e4m3 rows: the multihot step and the FP8
    dispatch from the top-k choices.  Returns (x_disp_q uint8 [C, H],
    x_disp_scale fp32 [C], (routing_map, probs, winner_slot), (R, N) or None);
    ``out`` optionally gives the two row buffers, ``multihot`` the three
    multihot outputs."""
    _bf16(x, "x")
    assert topk_idx.dtype == torch.int64 and topk_probs.dtype == torch.float32
    T, H = x.shape
    E = layout.E
    C = layout.capacity
    dev = x.device
    q = out[0] if out is not None else torch.empty(C, H, dtype=torch.uint8, device=dev)
    sc = out[1] if out is not None else torch.empty(C, dtype=torch.float32, device=dev)
    if multihot is None:
        multihot = (torch.empty(T, E, dtype=torch.uint8, device=dev), torch.empty(T, E, dtype=torch.float32, device=dev),
                    torch.empty(T, E, dtype=torch.int8, device=dev))
    rows = (ctypes.c_int64 * 2)() if host_sync else None
    _check(N.lib.moe_dispatch_topk_fp8(_ptr(x), _ptr(topk_idx), _ptr(topk_probs), H, layout.ref, _ptr(multihot[0]),
                                       _ptr(multihot[1]), _ptr(multihot[2]), _ptr(q), _ptr(sc), rows,
                                       _stream(stream)), "moe_dispatch_topk_fp8")
    return q, sc, tuple(multihot), ((int(rows[0]), int(rows[1])) if host_sync else None)


def moe_quantize_fp8(src: torch.Tensor, stream=None):
    """Rowwise e4m3 of a bf16 tensor whose last dimension is the row: returns
    (codes uint8, same shape; scales fp32, shape[:-1])."""
    _bf16(src, "src")
    cols = src.shape[-1]
    rows = src.numel() // cols
    codes = torch.empty(src.shape, dtype=torch.uint8, device=src.device)
    scales = torch.empty(src.shape[:-1], dtype=torch.float32, device=src.device)
    _check(N.lib.moe_quantize_fp8(_ptr(src), rows, cols, _ptr(codes), _ptr(scales), _stream(stream)),
           "moe_quantize_fp8")
    return codes, scales


def moe_grouped_experts_fp8(x_disp_q: torch.Tensor, x_disp_scale: torch.Tensor, layout: Layout,
                            W1_q: torch.Tensor, W1_scale: torch.Tensor, W2: torch.Tensor, out=None,
                            stream=None):
    """a5 with the e4m3 gate/up GEMM: returns dict(h, y), bf16 [C, *]."""
    E, twoI, H = W1_q.shape
    I = twoI // 2
    C = layout.capacity
    dev = x_disp_q.device
    o = out or {}
    h = o.get("h") if o.get("h") is not None else torch.empty(C, I, dtype=torch.bfloat16, device=dev)
    y = o.get("y") if o.get("y") is not None else torch.empty(C, H, dtype=torch.bfloat16, device=dev)
    _check(N.lib.moe_grouped_experts_fp8(_ptr(x_disp_q), _ptr(x_disp_scale), layout.ref, H, I, _ptr(W1_q),
                                         _ptr(W1_scale), _ptr(W2), _ptr(h), _ptr(y), _stream(stream)),
           "moe_grouped_experts_fp8")
    return {"h": h, "y": y}


def moe_grouped_experts(x_disp: torch.Tensor, layout: Layout, W1: torch.Tensor, W2: torch.Tensor,
                        save_o: bool = False, save_gu: bool = False, out=None, stream=None):
    """a5: returns dict(h, y, o (or None), gu (or None)), each [C, *] bf16."""
    E, twoI, H = W1.shape
    I = twoI // 2
    C = layout.capacity
    dev = x_disp.device
    o = out or {}
    h = o.get("h") if o.get("h") is not None else torch.empty(C, I, dtype=torch.bfloat16, device=dev)
    y = o.get("y") if o.get("y") is not None else torch.empty(C, H, dtype=torch.bfloat16, device=dev)
    o_save = (o.get("o") if o.get("o") is not None else torch.empty(C, H, dtype=torch.bfloat16, device=dev)) if save_o else None
    gu = (o.get("gu") if o.get("gu") is not None else torch.empty(C, 2 * I, dtype=torch.bfloat16, device=dev)) if save_gu else None
    _check(N.lib.moe_grouped_experts(_ptr(x_disp), layout.ref, H, I, _ptr(W1), _ptr(W2), _ptr(h),
                                     _ptr(y), _ptr(o_save), _ptr(gu), _stream(stream)),
           "moe_grouped_experts")
    return {"h": h, "y": y, "o": o_save, "gu": gu}


def moe_combine(y_disp: torch.Tensor, layout: Layout, out: Optional[torch.Tensor] = None, stream=None):
    """a6: out [T, H] bf16."""
    H = y_disp.shape[1]
    if out is None:
        out = torch.empty(layout.T, H, dtype=torch.bfloat16, device=y_disp.device)
    _check(N.lib.moe_combine(_ptr(y_disp), layout.ref, H, _ptr(out), _stream(stream)), "moe_combine")
    return out


def moe_combine_backward(grad_out: torch.Tensor, layout: Layout, o_save: Optional[torch.Tensor] = None,
                         stream=None, scaled: bool = False):
    """a7 (+a8 when o_save is given): returns (grad_y [C, H], grad_w [C] or None).
    With ``scaled`` (moe_combine_backward_scaled) the rows are G_o = bf16(w * grad_y)
    instead, for moe_grouped_experts_backward(..., scaled=True)."""
    H = grad_out.shape[1]
    grad_y = torch.empty(layout.capacity, H, dtype=torch.bfloat16, device=grad_out.device)
    grad_w = (torch.empty(layout.capacity, dtype=torch.float32, device=grad_out.device)
              if o_save is not None else None)
    fn = N.lib.moe_combine_backward_scaled if scaled else N.lib.moe_combine_backward
    _check(fn(_ptr(grad_out), _ptr(o_save), layout.ref, H, _ptr(grad_y), _ptr(grad_w), _stream(stream)),
           "moe_combine_backward_scaled" if scaled else "moe_combine_backward")
    return grad_y, grad_w


def moe_dispatch_backward(grad_x_disp: torch.Tensor, layout: Layout,
                          grad_w: Optional[torch.Tensor] = None, stream=None):
    """a10 (+ grad_w scatter): returns (grad_x [T, H], grad_probs [T, E] or None)."""
    H = grad_x_disp.shape[1]
    dev = grad_x_disp.device
    grad_x = torch.empty(layout.T, H, dtype=torch.bfloat16, device=dev)
    grad_probs = (torch.empty(layout.T, layout.E, dtype=torch.float32, device=dev)
                  if grad_w is not None else None)
    _check(N.lib.moe_dispatch_backward(_ptr(grad_x_disp), _ptr(grad_w), layout.ref, H, _ptr(grad_x),
                                       _ptr(grad_probs), _stream(stream)), "moe_dispatch_backward")
    return grad_x, grad_probs


def moe_route_to_multihot_backward(grad_probs: torch.Tensor, topk_idx: torch.Tensor,
                                   winner_slot: torch.Tensor, stream=None):
    """Multihot backward: grad_topk_probs [T, K] fp32."""
    T, K = topk_idx.shape
    E = grad_probs.shape[1]
    g = torch.empty(T, K, dtype=torch.float32, device=grad_probs.device)
    _check(N.lib.moe_route_to_multihot_backward(_ptr(grad_probs), _ptr(topk_idx), _ptr(winner_slot),
                                                T, K, E, _ptr(g), _stream(stream)),
           "moe_route_to_multihot_backward")
    return g


def moe_grouped_experts_backward(grad_y: torch.Tensor, x_disp: torch.Tensor, h: torch.Tensor,
                                 gu_save: torch.Tensor, layout: Layout, W1: torch.Tensor,
                                 W2: torch.Tensor, stream=None, return_operands: bool = False,
                                 scaled: bool = False):
    """a9: returns (grad_x_disp [C, H] bf16, dW1 [E, 2I, H] fp32, dW2 [E, H, I] fp32),
    plus, with return_operands, views of the workspace's G_o [C, H] and
    [G_g | G_u] [C, 2I] (bf16, valid rows).  With ``scaled``
    (moe_grouped_experts_backward_scaled) ``grad_y`` is G_o from
    moe_combine_backward(..., scaled=True), and the G_o returned is ``grad_y``."""
    E, twoI, H = W1.shape
    I = twoI // 2
    dev = grad_y.device
    nbytes = ctypes.c_size_t(0)
    _check(N.lib.moe_experts_backward_workspace_bytes(layout.capacity, H, I, ctypes.byref(nbytes)),
           "moe_experts_backward_workspace_bytes")
    ws = torch.empty(nbytes.value, dtype=torch.uint8, device=dev)
    grad_x_disp = torch.empty(layout.capacity, H, dtype=torch.bfloat16, device=dev)
    dW1 = torch.empty(E, 2 * I, H, dtype=torch.float32, device=dev)
    dW2 = torch.empty(E, H, I, dtype=torch.float32, device=dev)
    fn = N.lib.moe_grouped_experts_backward_scaled if scaled else N.lib.moe_grouped_experts_backward
    _check(fn(_ptr(grad_y), _ptr(x_disp), _ptr(h), _ptr(gu_save), layout.ref, H, I, _ptr(W1), _ptr(W2),
              _ptr(grad_x_disp), _ptr(dW1), _ptr(dW2), _ptr(ws), _stream(stream)),
           "moe_grouped_experts_backward_scaled" if scaled else "moe_grouped_experts_backward")
    if not return_operands:
        return grad_x_disp, dW1, dW2
    C = layout.capacity
    base = (-ws.data_ptr()) % 256
    go_bytes = C * H * 2
    gu_off = base + (go_bytes + 255) // 256 * 256
    G_o = grad_y if scaled else ws[base:base + go_bytes].view(torch.bfloat16).view(C, H)
    G_gu = ws[gu_off:gu_off + C * 2 * I * 2].view(torch.bfloat16).view(C, 2 * I)
    return grad_x_disp, dW1, dW2, G_o, G_gu


@dataclass
class ForwardResult:
    out: torch.Tensor
    layout: Layout
    routing_map: torch.Tensor
    probs: torch.Tensor
    winner_slot: torch.Tensor
    x_disp: torch.Tensor
    h: torch.Tensor
    y: torch.Tensor
    o: Optional[torch.Tensor]
    gu: Optional[torch.Tensor]
    rows: Optional[tuple]


def moe_layer_forward(x, topk_idx, topk_probs, W1, W2, pad_multiple: int, host_sync: bool = True,
                      capacity: Optional[int] = None, save_for_backward: bool = False,
                      layout: Optional[Layout] = None, stream=None) -> ForwardResult:
    """a1..a6 in order: multihot, dispatch, grouped experts, combine."""
    T, K = topk_idx.shape
    E = W1.shape[0]
    if layout is None:
        C = capacity if capacity is not None else worst_case_rows(T, E, K, pad_multiple)
        layout = Layout(T, E, K, pad_multiple, C, device=x.device)
    rmap, probs, win = moe_route_to_multihot(topk_idx, topk_probs, E, layout.status, stream)
    x_disp, rows = moe_dispatch(x, rmap, probs, layout, host_sync=host_sync, stream=stream)
    ex = moe_grouped_experts(x_disp, layout, W1, W2, save_o=save_for_backward,
                             save_gu=save_for_backward, stream=stream)
    out = moe_combine(ex["y"], layout, stream=stream)
    return ForwardResult(out, layout, rmap, probs, win, x_disp, ex["h"], ex["y"], ex["o"], ex["gu"], rows)
