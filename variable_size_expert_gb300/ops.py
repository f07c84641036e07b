"""torch-facing API over the C ABI.

PyTorch supplies device memory and the current stream; every step of the
method runs in libmgg.so's kernels.  Inputs must be CUDA tensors on an
sm_103 device; there is no CPU fallback.

Functions mirror the pages' usage ("grouped-gemm-moe", §Usage):
  moe(x, W, expert_ids, topk_weights)        differentiable fused MoE layer
  grouped_gemm(a, W, group_sizes | end_offs) bare variable-size grouped GEMM
plus the lower-level calls (route, moe_forward, moe_backward,
grouped_gemm_masked, debug_tile_schedule) and the e4m3 forms with per-row
scales (quantize_fp8, moe_forward_fp8, grouped_gemm_fp8,
grouped_gemm_masked_fp8) and per-column weight scales for the input
gradient (quantize_fp8_cols, moe_backward_dx_fp8).
"""
from __future__ import annotations

import ctypes
from dataclasses import dataclass

import torch

from . import _lib as L

__all__ = [
    "RoutingBuffers", "route", "route_noalloc", "moe_forward", "moe_backward", "moe", "grouped_gemm",
    "grouped_gemm_masked", "debug_tile_schedule", "tile_config", "workspace_bytes",
    "moe_ffn_forward", "quantize_fp8", "moe_forward_fp8", "grouped_gemm_fp8",
    "grouped_gemm_masked_fp8", "quantize_fp8_cols", "moe_backward_dx_fp8",
    "new_status", "read_status",
]


def _dtype_code(t: torch.Tensor) -> int:
    if t.dtype == torch.bfloat16:
        return L.MGG_BF16
    if t.dtype == torch.float32:
        return L.MGG_F32
    raise TypeError(f"unsupported dtype {t.dtype}: bfloat16 or float32")


def _ptr(t: torch.Tensor | None) -> int | None:
    if t is None:
        return None
    if not t.is_cuda:
        raise ValueError("tensors must live on a CUDA device")
    if not t.is_contiguous():
        raise ValueError("tensors must be contiguous")
    return t.data_ptr()


def _stream() -> int:
    return torch.cuda.current_stream().cuda_stream


def _workspace(nbytes: int, device) -> torch.Tensor:
    return torch.empty(max(int(nbytes), 256), dtype=torch.uint8, device=device)


def new_status(device) -> torch.Tensor:
    """A zeroed device status word (int32[1]) for the kernels to OR error bits into."""
    return torch.zeros(1, dtype=torch.int32, device=device)


def read_status(status: torch.Tensor) -> int:
    """Synchronising read of a status word (for tests and debugging)."""
    return int(status.item())


def _code_of(dtype: torch.dtype) -> int:
    if dtype in (torch.uint8, torch.float8_e4m3fn):
        return L.MGG_FP8_E4M3
    return L.MGG_BF16 if dtype == torch.bfloat16 else L.MGG_F32


def tile_config(op: int, dtype: torch.dtype = torch.bfloat16):
    lib = L.load()
    bm, bn, bk = ctypes.c_int(), ctypes.c_int(), ctypes.c_int()
    code = _code_of(dtype)
    L.check(lib.mgg_tile_config(op, code, ctypes.byref(bm), ctypes.byref(bn), ctypes.byref(bk)),
            "mgg_tile_config")
    return bm.value, bn.value, bk.value


def workspace_bytes(op: int, T=0, k=0, E=0, N=0, K=0, dtype=torch.bfloat16) -> int:
    code = _code_of(dtype)
    return int(L.load().mgg_workspace_bytes(op, T, k, E, N, K, code))


@dataclass
class RoutingBuffers:
    """Device routing buffers (see mgg_routing in include/mgg.h)."""
    counts: torch.Tensor
    end_offs: torch.Tensor
    start: torch.Tensor
    tile_start: torch.Tensor
    row_assign: torch.Tensor
    row_token: torch.Tensor
    row_weight: torch.Tensor
    assign_row: torch.Tensor

    @staticmethod
    def empty(T: int, k: int, E: int, device) -> "RoutingBuffers":
        S = T * k
        i32 = dict(dtype=torch.int32, device=device)
        return RoutingBuffers(
            counts=torch.empty(E, **i32), end_offs=torch.empty(E, **i32),
            start=torch.empty(E + 1, **i32), tile_start=torch.empty(E + 1, **i32),
            row_assign=torch.empty(S, **i32), row_token=torch.empty(S, **i32),
            row_weight=torch.empty(S, dtype=torch.float32, device=device),
            assign_row=torch.empty(S, **i32))

    def struct(self) -> L.Routing:
        return L.Routing(*(_ptr(getattr(self, f)) for f, _ in L.Routing._fields_))


def _ids_i32(expert_ids: torch.Tensor) -> torch.Tensor:
    # the ABI takes int32 ids; torch's usual int64 is narrowed here (marshalling)
    return expert_ids if expert_ids.dtype == torch.int32 else expert_ids.to(torch.int32)


def route(expert_ids: torch.Tensor, topk_weights: torch.Tensor, E: int, N: int,
          dtype: torch.dtype = torch.bfloat16, status: torch.Tensor | None = None,
          out: RoutingBuffers | None = None) -> RoutingBuffers:
    """Device routing: counts, offsets, stable permutation, tile prefix sums."""
    lib = L.load()
    ids = _ids_i32(expert_ids).contiguous()
    w = topk_weights.contiguous().float()
    T, k = ids.shape
    dev = ids.device
    r = out or RoutingBuffers.empty(T, k, E, dev)
    st = status if status is not None else new_status(dev)
    code = L.MGG_BF16 if dtype == torch.bfloat16 else L.MGG_F32
    nbytes = lib.mgg_workspace_bytes(L.MGG_OP_ROUTE, T, k, E, N, 0, code)
    ws = _workspace(nbytes, dev)
    rs = r.struct()
    L.check(lib.mgg_route(_ptr(ids), _ptr(w), T, k, E, N, code, ctypes.byref(rs), _ptr(st),
                          _ptr(ws), ws.numel(), _stream()), "mgg_route")
    return r


def route_noalloc(expert_ids: torch.Tensor, topk_weights: torch.Tensor, E: int, N: int,
                  dtype: torch.dtype = torch.bfloat16, status: torch.Tensor | None = None,
                  out: RoutingBuffers | None = None) -> RoutingBuffers:
    """``route`` without a workspace: the library's fixed device scratch
    serves the histogram (mgg_route_noalloc; results as mgg_route)."""
    lib = L.load()
    ids = _ids_i32(expert_ids).contiguous()
    w = topk_weights.contiguous().float()
    T, k = ids.shape
    dev = ids.device
    r = out or RoutingBuffers.empty(T, k, E, dev)
    st = status if status is not None else new_status(dev)
    code = L.MGG_BF16 if dtype == torch.bfloat16 else L.MGG_F32
    rs = r.struct()
    L.check(lib.mgg_route_noalloc(_ptr(ids), _ptr(w), T, k, E, N, code, ctypes.byref(rs),
                                  _ptr(st), _stream()), "mgg_route_noalloc")
    return r


def moe_forward(x: torch.Tensor, W: torch.Tensor, expert_ids: torch.Tensor,
                topk_weights: torch.Tensor, status: torch.Tensor | None = None,
                out: torch.Tensor | None = None, routing: RoutingBuffers | None = None,
                workspace: torch.Tensor | None = None):
    """Fused MoE forward.  Returns (y [T, N] float32, routing)."""
    lib = L.load()
    code = _dtype_code(x)
    if W.dtype != x.dtype:
        raise TypeError("x and W must share a dtype")
    T, K = x.shape
    E, N, K2 = W.shape
    if K2 != K:
        raise ValueError("W must be [E, N, K] with the K of x")
    ids = _ids_i32(expert_ids).contiguous()
    w = topk_weights.detach().contiguous().float()
    k = ids.shape[1]
    dev = x.device
    y = out if out is not None else torch.empty(T, N, dtype=torch.float32, device=dev)
    r = routing or RoutingBuffers.empty(T, k, E, dev)
    st = status if status is not None else new_status(dev)
    nbytes = lib.mgg_workspace_bytes(L.MGG_OP_FORWARD, T, k, E, N, K, code)
    ws = workspace if workspace is not None and workspace.numel() >= nbytes else _workspace(nbytes, dev)
    rs = r.struct()
    L.check(lib.mgg_moe_forward(_ptr(x), _ptr(W), _ptr(ids), _ptr(w), T, K, N, E, k, code,
                                _ptr(y), ctypes.byref(rs), _ptr(st), _ptr(ws), ws.numel(),
                                _stream()), "mgg_moe_forward")
    return y, r


def moe_ffn_forward(x: torch.Tensor, Wg: torch.Tensor, Wu: torch.Tensor, Wd: torch.Tensor,
                    expert_ids: torch.Tensor, topk_weights: torch.Tensor,
                    status: torch.Tensor | None = None, out: torch.Tensor | None = None,
                    h: torch.Tensor | None = None, routing: RoutingBuffers | None = None,
                    workspace: torch.Tensor | None = None, gu: torch.Tensor | bool | None = None):
    """Gated expert FFN forward (bf16).  Returns (y [T, H] float32, h [T*k, F]
    bf16 in expert-sorted row order, routing), and with ``gu`` (True, or a
    float32 [T*k, 2F] buffer) also gu, the gate and up projections the
    backward needs: (y, h, routing, gu)."""
    lib = L.load()
    if x.dtype != torch.bfloat16 or not (Wg.dtype == Wu.dtype == Wd.dtype == torch.bfloat16):
        raise TypeError("the gated FFN path takes bfloat16 x and weights")
    T, H = x.shape
    E, F, H2 = Wg.shape
    if H2 != H or tuple(Wu.shape) != (E, F, H) or tuple(Wd.shape) != (E, H, F):
        raise ValueError("expected Wg, Wu [E, F, H] and Wd [E, H, F] with the H of x")
    ids = _ids_i32(expert_ids).contiguous()
    w = topk_weights.detach().contiguous().float()
    k = ids.shape[1]
    dev = x.device
    y = out if out is not None else torch.empty(T, H, dtype=torch.float32, device=dev)
    hb = h if h is not None else torch.empty(T * k, F, dtype=torch.bfloat16, device=dev)
    r = routing or RoutingBuffers.empty(T, k, E, dev)
    st = status if status is not None else new_status(dev)
    nbytes = lib.mgg_workspace_bytes(L.MGG_OP_FFN_FORWARD, T, k, E, H, F, L.MGG_BF16)
    ws = workspace if workspace is not None and workspace.numel() >= nbytes else _workspace(nbytes, dev)
    rs = r.struct()
    gub = None
    if gu is not None and gu is not False:
        gub = gu if isinstance(gu, torch.Tensor) else torch.empty(T * k, 2 * F, dtype=torch.float32,
                                                                  device=dev)
    L.check(lib.mgg_moe_ffn_forward(_ptr(x), _ptr(Wg), _ptr(Wu), _ptr(Wd), _ptr(ids), _ptr(w), T,
                                    H, F, E, k, L.MGG_BF16, _ptr(y), _ptr(hb),
                                    _ptr(gub) if gub is not None else None, ctypes.byref(rs),
                                    _ptr(st), _ptr(ws), ws.numel(), _stream()),
            "mgg_moe_ffn_forward")
    return (y, hb, r) if gub is None else (y, hb, r, gub)


def moe_ffn_backward(dy: torch.Tensor, x: torch.Tensor, Wg: torch.Tensor, Wu: torch.Tensor,
                     Wd: torch.Tensor, h: torch.Tensor, gu: torch.Tensor, routing: RoutingBuffers,
                     k: int, status: torch.Tensor | None = None, dx=None, dWg=None, dWu=None,
                     dWd=None, dtopk=None, workspace: torch.Tensor | None = None):
    """Gated expert FFN backward (bf16) from the training forward's h and gu.
    Returns (dx [T, H], dWg [E, F, H], dWu [E, F, H], dWd [E, H, F],
    dtopk [T, k]), all float32."""
    lib = L.load()
    T, H = x.shape
    E, F, _ = Wg.shape
    dev = x.device
    dy = dy.contiguous().float()
    f32 = dict(dtype=torch.float32, device=dev)
    dx = dx if dx is not None else torch.empty(T, H, **f32)
    dWg = dWg if dWg is not None else torch.empty(E, F, H, **f32)
    dWu = dWu if dWu is not None else torch.empty(E, F, H, **f32)
    dWd = dWd if dWd is not None else torch.empty(E, H, F, **f32)
    dtopk = dtopk if dtopk is not None else torch.empty(T, k, **f32)
    st = status if status is not None else new_status(dev)
    nbytes = lib.mgg_workspace_bytes(L.MGG_OP_FFN_BACKWARD, T, k, E, H, F, L.MGG_BF16)
    ws = workspace if workspace is not None and workspace.numel() >= nbytes else _workspace(nbytes, dev)
    rs = routing.struct()
    L.check(lib.mgg_moe_ffn_backward(_ptr(dy), _ptr(x), _ptr(Wg), _ptr(Wu), _ptr(Wd), _ptr(h),
                                     _ptr(gu), ctypes.byref(rs), T, H, F, E, k, L.MGG_BF16,
                                     _ptr(dx), _ptr(dWg), _ptr(dWu), _ptr(dWd), _ptr(dtopk),
                                     _ptr(st), _ptr(ws), ws.numel(), _stream()),
            "mgg_moe_ffn_backward")
    return dx, dWg, dWu, dWd, dtopk


def moe_backward(dy: torch.Tensor, x: torch.Tensor, W: torch.Tensor, routing: RoutingBuffers,
                 k: int, status: torch.Tensor | None = None, dx=None, dW=None, dtopk=None,
                 workspace: torch.Tensor | None = None):
    """Fused MoE backward.  Returns (dx [T,K], dW [E,N,K], dtopk [T,k]), all float32."""
    lib = L.load()
    code = _dtype_code(x)
    T, K = x.shape
    E, N, _ = W.shape
    dev = x.device
    dy = dy.contiguous().float()
    dx = dx if dx is not None else torch.empty(T, K, dtype=torch.float32, device=dev)
    dW = dW if dW is not None else torch.empty(E, N, K, dtype=torch.float32, device=dev)
    dtopk = dtopk if dtopk is not None else torch.empty(T, k, dtype=torch.float32, device=dev)
    st = status if status is not None else new_status(dev)
    nbytes = lib.mgg_workspace_bytes(L.MGG_OP_BACKWARD, T, k, E, N, K, code)
    ws = workspace if workspace is not None and workspace.numel() >= nbytes else _workspace(nbytes, dev)
    rs = routing.struct()
    L.check(lib.mgg_moe_backward(_ptr(dy), _ptr(x), _ptr(W), ctypes.byref(rs), T, K, N, E, k, code,
                                 _ptr(dx), _ptr(dW), _ptr(dtopk), _ptr(st), _ptr(ws), ws.numel(),
                                 _stream()), "mgg_moe_backward")
    return dx, dW, dtopk


class _MoEFunction(torch.autograd.Function):
    @staticmethod
    def forward(ctx, x, W, expert_ids, topk_weights):
        y, r = moe_forward(x.detach(), W.detach(), expert_ids, topk_weights.detach())
        ctx.save_for_backward(x.detach(), W.detach())
        ctx.routing = r
        ctx.k = expert_ids.shape[1]
        ctx.w_dtype = topk_weights.dtype
        return y

    @staticmethod
    def backward(ctx, dy):
        x, W = ctx.saved_tensors
        dx, dW, dtopk = moe_backward(dy, x, W, ctx.routing, ctx.k)
        return dx.to(x.dtype), dW.to(W.dtype), None, dtopk.to(ctx.w_dtype)


def moe(x: torch.Tensor, W: torch.Tensor, expert_ids: torch.Tensor,
        topk_weights: torch.Tensor) -> torch.Tensor:
    """Fused MoE layer y[t] = sum_j w[t,j] x[t] W_{ids[t,j]}^T, differentiable to
    x, W and topk_weights ("grouped-gemm-moe", §Usage)."""
    return _MoEFunction.apply(x, W, expert_ids, topk_weights)


def grouped_gemm(a: torch.Tensor, W: torch.Tensor, group_sizes: torch.Tensor | None = None,
                 end_offs: torch.Tensor | None = None, status: torch.Tensor | None = None,
                 out: torch.Tensor | None = None) -> torch.Tensor:
    """Bare grouped GEMM on pre-grouped rows: out[r] = a[r] W_e^T for the
    group e holding row r.  Give either group sizes or int32 end offsets."""
    lib = L.load()
    code = _dtype_code(a)
    rows, K = a.shape
    E, N, _ = W.shape
    if (group_sizes is None) == (end_offs is None):
        raise ValueError("give exactly one of group_sizes and end_offs")
    layout = L.MGG_LAYOUT_CONTIGUOUS_SIZES if group_sizes is not None else L.MGG_LAYOUT_CONTIGUOUS
    offs = (group_sizes if group_sizes is not None else end_offs)
    offs = offs.to(device=a.device, dtype=torch.int32).contiguous()
    dev = a.device
    C = out if out is not None else torch.empty(rows, N, dtype=torch.float32, device=dev)
    st = status if status is not None else new_status(dev)
    nbytes = lib.mgg_workspace_bytes(L.MGG_OP_GROUPED_GEMM, 0, 0, E, N, K, code)
    ws = _workspace(nbytes, dev)
    L.check(lib.mgg_grouped_gemm(_ptr(a), _ptr(W), _ptr(C), code, layout, _ptr(offs), rows, E, N, K,
                                 _ptr(st), _ptr(ws), ws.numel(), _stream()), "mgg_grouped_gemm")
    return C


def grouped_gemm_masked(x: torch.Tensor, W: torch.Tensor, masked_m: torch.Tensor,
                        status: torch.Tensor | None = None,
                        out: torch.Tensor | None = None) -> torch.Tensor:
    """Masked decode layout: out[e, i] = x[e, i] W_e^T for i < masked_m[e];
    other rows of ``out`` are left as they were."""
    lib = L.load()
    code = _dtype_code(x)
    E, M_max, K = x.shape
    _, N, _ = W.shape
    dev = x.device
    mm = masked_m.to(device=dev, dtype=torch.int32).contiguous()
    y = out if out is not None else torch.zeros(E, M_max, N, dtype=torch.float32, device=dev)
    st = status if status is not None else new_status(dev)
    L.check(lib.mgg_grouped_gemm(_ptr(x), _ptr(W), _ptr(y), code, L.MGG_LAYOUT_MASKED, _ptr(mm),
                                 M_max, E, N, K, _ptr(st), None, 0, _stream()),
            "mgg_grouped_gemm(masked)")
    return y


# ---------------------------------------------------------------- e4m3
def _codes(t: torch.Tensor) -> torch.Tensor:
    if t.dtype == torch.float8_e4m3fn:
        return t.view(torch.uint8)
    if t.dtype != torch.uint8:
        raise TypeError("e4m3 operands are uint8 codes (or float8_e4m3fn)")
    return t


def quantize_fp8(src: torch.Tensor):
    """Per-row e4m3 quantisation of a bfloat16/float32 tensor [..., C]:
    returns (codes uint8 [..., C], scale float32 [...]) with
    src ~ decode(codes) * scale[..., None] (mgg_quantize_fp8)."""
    lib = L.load()
    code = _dtype_code(src)
    src = src.contiguous()
    cols = src.shape[-1]
    rows = src.numel() // max(cols, 1)
    q = torch.empty(src.shape, dtype=torch.uint8, device=src.device)
    scale = torch.empty(src.shape[:-1], dtype=torch.float32, device=src.device)
    L.check(lib.mgg_quantize_fp8(_ptr(src), code, rows, cols, _ptr(q), _ptr(scale), _stream()),
            "mgg_quantize_fp8")
    return q, scale


def moe_forward_fp8(xq: torch.Tensor, x_scale: torch.Tensor, Wq: torch.Tensor,
                    w_scale: torch.Tensor, expert_ids: torch.Tensor, topk_weights: torch.Tensor,
                    status: torch.Tensor | None = None, out: torch.Tensor | None = None,
                    routing: RoutingBuffers | None = None, workspace: torch.Tensor | None = None):
    """Fused MoE forward on e4m3 codes with per-token (x_scale [T]) and
    per-(expert, channel) (w_scale [E, N]) scales.  Returns (y, routing)."""
    lib = L.load()
    xq, Wq = _codes(xq), _codes(Wq)
    T, K = xq.shape
    E, N, K2 = Wq.shape
    if K2 != K:
        raise ValueError("W must be [E, N, K] with the K of x")
    ids = _ids_i32(expert_ids).contiguous()
    w = topk_weights.detach().contiguous().float()
    k = ids.shape[1]
    dev = xq.device
    y = out if out is not None else torch.empty(T, N, dtype=torch.float32, device=dev)
    r = routing or RoutingBuffers.empty(T, k, E, dev)
    st = status if status is not None else new_status(dev)
    nbytes = lib.mgg_workspace_bytes(L.MGG_OP_FORWARD, T, k, E, N, K, L.MGG_FP8_E4M3)
    ws = workspace if workspace is not None and workspace.numel() >= nbytes else _workspace(nbytes, dev)
    rs = r.struct()
    L.check(lib.mgg_moe_forward_fp8(_ptr(xq), _ptr(x_scale.contiguous()), _ptr(Wq),
                                    _ptr(w_scale.contiguous()), _ptr(ids), _ptr(w), T, K, N, E, k,
                                    _ptr(y), ctypes.byref(rs), _ptr(st), _ptr(ws), ws.numel(),
                                    _stream()), "mgg_moe_forward_fp8")
    return y, r


def quantize_fp8_cols(W: torch.Tensor):
    """Per-(expert, input column) e4m3 quantisation of W [E, N, K] (bfloat16),
    stored transposed: returns (codes uint8 [E, K, N], scale float32 [E, K])
    with W[e, n, k] ~ decode(codes[e, k, n]) * scale[e, k]
    (mgg_quantize_fp8_cols)."""
    lib = L.load()
    if W.dtype != torch.bfloat16 or W.dim() != 3:
        raise TypeError("W must be a bfloat16 [E, N, K] tensor")
    W = W.contiguous()
    E, N, K = W.shape
    q = torch.empty(E, K, N, dtype=torch.uint8, device=W.device)
    scale = torch.empty(E, K, dtype=torch.float32, device=W.device)
    L.check(lib.mgg_quantize_fp8_cols(_ptr(W), E, N, K, _ptr(q), _ptr(scale), _stream()),
            "mgg_quantize_fp8_cols")
    return q, scale


def moe_backward_dx_fp8(dyq: torch.Tensor, dy_scale: torch.Tensor, Wtq: torch.Tensor,
                        wt_scale: torch.Tensor, x: torch.Tensor, routing: RoutingBuffers, k: int,
                        status: torch.Tensor | None = None, dx=None, dtopk=None,
                        workspace: torch.Tensor | None = None):
    """Input and routing-weight gradients on e4m3 operands: dy quantised per
    token (dyq [T, N], dy_scale [T]) and W per input column (Wtq [E, K, N],
    wt_scale [E, K], from quantize_fp8_cols); x [T, K] bfloat16.  Returns
    (dx [T, K], dtopk [T, k]), float32 (mgg_moe_backward_dx_fp8)."""
    lib = L.load()
    dyq, Wtq = _codes(dyq), _codes(Wtq)
    T, N = dyq.shape
    E, K, N2 = Wtq.shape
    if N2 != N or tuple(x.shape) != (T, K):
        raise ValueError("dyq [T, N], Wtq [E, K, N] and x [T, K] must agree")
    if x.dtype != torch.bfloat16:
        raise TypeError("x must be bfloat16")
    dev = dyq.device
    x = x.contiguous()
    dx = dx if dx is not None else torch.empty(T, K, dtype=torch.float32, device=dev)
    dtopk = dtopk if dtopk is not None else torch.empty(T, k, dtype=torch.float32, device=dev)
    st = status if status is not None else new_status(dev)
    nbytes = lib.mgg_workspace_bytes(L.MGG_OP_BACKWARD, T, k, E, N, K, L.MGG_FP8_E4M3)
    ws = workspace if workspace is not None and workspace.numel() >= nbytes else _workspace(nbytes, dev)
    rs = routing.struct()
    L.check(lib.mgg_moe_backward_dx_fp8(_ptr(dyq.contiguous()), _ptr(dy_scale.contiguous()),
                                        _ptr(Wtq.contiguous()), _ptr(wt_scale.contiguous()), _ptr(x),
                                        ctypes.byref(rs), T, K, N, E, k, _ptr(dx), _ptr(dtopk),
                                        _ptr(st), _ptr(ws), ws.numel(), _stream()),
            "mgg_moe_backward_dx_fp8")
    return dx, dtopk


def grouped_gemm_fp8(aq: torch.Tensor, a_scale: torch.Tensor, Wq: torch.Tensor,
                     w_scale: torch.Tensor, group_sizes: torch.Tensor | None = None,
                     end_offs: torch.Tensor | None = None, status: torch.Tensor | None = None,
                     out: torch.Tensor | None = None) -> torch.Tensor:
    """Bare grouped GEMM on e4m3 codes: out[r] = a_scale[r] w_scale[e] * (a[r] W_e^T)."""
    lib = L.load()
    aq, Wq = _codes(aq), _codes(Wq)
    rows, K = aq.shape
    E, N, _ = Wq.shape
    if (group_sizes is None) == (end_offs is None):
        raise ValueError("give exactly one of group_sizes and end_offs")
    layout = L.MGG_LAYOUT_CONTIGUOUS_SIZES if group_sizes is not None else L.MGG_LAYOUT_CONTIGUOUS
    offs = (group_sizes if group_sizes is not None else end_offs)
    offs = offs.to(device=aq.device, dtype=torch.int32).contiguous()
    dev = aq.device
    C = out if out is not None else torch.empty(rows, N, dtype=torch.float32, device=dev)
    st = status if status is not None else new_status(dev)
    nbytes = lib.mgg_workspace_bytes(L.MGG_OP_GROUPED_GEMM, 0, 0, E, N, K, L.MGG_FP8_E4M3)
    ws = _workspace(nbytes, dev)
    L.check(lib.mgg_grouped_gemm_fp8(_ptr(aq), _ptr(a_scale.contiguous()), _ptr(Wq),
                                     _ptr(w_scale.contiguous()), _ptr(C), layout, _ptr(offs), rows,
                                     E, N, K, _ptr(st), _ptr(ws), ws.numel(), _stream()),
            "mgg_grouped_gemm_fp8")
    return C


def grouped_gemm_masked_fp8(xq: torch.Tensor, x_scale: torch.Tensor, Wq: torch.Tensor,
                            w_scale: torch.Tensor, masked_m: torch.Tensor,
                            status: torch.Tensor | None = None,
                            out: torch.Tensor | None = None) -> torch.Tensor:
    """Masked decode layout on e4m3 codes: out[e, i] = x_scale[e, i] w_scale[e] *
    (x[e, i] W_e^T) for i < masked_m[e]; other rows of ``out`` are left as they were."""
    lib = L.load()
    xq, Wq = _codes(xq), _codes(Wq)
    E, M_max, K = xq.shape
    _, N, _ = Wq.shape
    dev = xq.device
    mm = masked_m.to(device=dev, dtype=torch.int32).contiguous()
    y = out if out is not None else torch.zeros(E, M_max, N, dtype=torch.float32, device=dev)
    st = status if status is not None else new_status(dev)
    L.check(lib.mgg_grouped_gemm_fp8(_ptr(xq), _ptr(x_scale.contiguous()), _ptr(Wq),
                                     _ptr(w_scale.contiguous()), _ptr(y), L.MGG_LAYOUT_MASKED,
                                     _ptr(mm), M_max, E, N, K, _ptr(st), None, 0, _stream()),
            "mgg_grouped_gemm_fp8(masked)")
    return y


def debug_tile_schedule(routing: RoutingBuffers, E: int, N: int, max_tiles: int,
                        dtype: torch.dtype = torch.bfloat16) -> torch.Tensor:
    """The (e, mb, nb, row0, rows) the GEMM kernel decodes for each tile index;
    rows past the device tile count stay -1."""
    lib = L.load()
    out = torch.full((max(max_tiles, 1), 5), -1, dtype=torch.int32, device=routing.counts.device)
    code = L.MGG_BF16 if dtype == torch.bfloat16 else L.MGG_F32
    rs = routing.struct()
    L.check(lib.mgg_debug_tile_schedule(ctypes.byref(rs), E, N, code, max_tiles, _ptr(out), _stream()),
            "mgg_debug_tile_schedule")
    return out[:max_tiles]
