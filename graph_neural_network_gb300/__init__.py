"""IO-aware fused GAT neighbour aggregation on GB300 (sm_103a).

Python front end of the C-ABI library ``libgnnagg.so`` (``include/gnnagg.h``).
torch supplies device memory and the current stream; the library's CUDA
kernels do all the work.

    g = Graph(row_ptr, col_idx)                    # once per graph (CSR, int32, cuda)
    out, lse = gat_forward(g, h, a_src, a_dst, 0.2)
    dh, da_src, da_dst = gat_backward(g, h, a_src, a_dst, 0.2, lse, dout)

``GATAggregate`` wraps the pair as a torch.autograd.Function.

The SpMM-family propagation of GCN / GraphConv layers (out = A~ x, norm
"sum", "mean" or "sym") runs on the same prepared graph:

    out = gcn_forward(g, x, "sym")                 # x [N, F]
    dx = gcn_backward(g, dout, "sym")              # A~^T dout over the cached CSC

the GATv2 attention (score att . LeakyReLU(xr_i + xl_j), value xl_j):

    out, lse = gatv2_forward(g, xl, xr, att, 0.2)
    dxl, dxr, datt = gatv2_backward(g, xl, xr, att, 0.2, lse, dout)

the graph-transformer attention (score scale * q_i . key_j, value val_j):

    out, lse = transformer_forward(g, q, key, val)     # scale defaults to 1/sqrt(D)
    dq, dkey, dval = transformer_backward(g, q, key, val, lse, dout)

and the max / min neighbourhood reduction with its winners:

    out, arg = reduce_forward(g, x, "max")         # arg [N, F] int32, -1 if no in-edges
    dx = reduce_backward(g, arg, dout)
"""
from __future__ import annotations

import ctypes

import torch

from . import _native
from ._native import GnnError, Tiling

__all__ = ["Graph", "gat_forward", "gat_backward", "GATAggregate", "GnnError", "Tiling",
           "check_device_error", "default_tiling", "gcn_forward", "gcn_backward",
           "GCNAggregate", "reduce_forward", "reduce_backward", "ReduceAggregate",
           "gatv2_forward", "gatv2_backward", "GATv2Aggregate", "transformer_forward",
           "transformer_backward", "TransformerAggregate"]


def _ptr(t):
    return None if t is None else ctypes.c_void_p(t.data_ptr())


def _stream(stream, device):
    s = stream if stream is not None else torch.cuda.current_stream(device)
    return ctypes.c_void_p(s.cuda_stream)


def _dtype_code(dt):
    if dt == torch.float32:
        return _native.F32
    if dt == torch.bfloat16:
        return _native.BF16
    raise TypeError(f"features must be float32 or bfloat16, got {dt}")


def default_tiling() -> Tiling:
    return _native.default_tiling()


class Graph:
    """A CSR graph prepared for aggregation (CSC transpose and degree buckets).

    row_ptr [N+1] and col_idx [E] are int32 CUDA tensors; row i lists the
    sources j of the edges j -> i.  They are referenced, not copied, and kept
    alive by this object.
    """

    def __init__(self, row_ptr: torch.Tensor, col_idx: torch.Tensor, tiling: Tiling | None = None,
                 stream=None):
        lib = _native.load()
        if row_ptr.dtype != torch.int32 or col_idx.dtype != torch.int32:
            raise TypeError("row_ptr and col_idx must be int32")
        if not (row_ptr.is_cuda and col_idx.is_cuda):
            raise ValueError("row_ptr and col_idx must be CUDA tensors")
        self.row_ptr = row_ptr.contiguous()
        self.col_idx = col_idx.contiguous()
        self.device = row_ptr.device
        self.n = self.row_ptr.numel() - 1
        self.e = self.col_idx.numel()
        self.tiling = tiling if tiling is not None else default_tiling()
        tref = ctypes.byref(self.tiling)
        nb = lib.gnn_graph_buffer_bytes(self.n, self.e, tref)
        ns = lib.gnn_graph_scratch_bytes(self.n, self.e)
        if nb == 0 or ns == 0:
            raise GnnError(_native.ERR_INVALID_ARG, "graph sizes or tiling")
        self.buffer = torch.empty(nb, dtype=torch.uint8, device=self.device)
        scratch = torch.empty(ns, dtype=torch.uint8, device=self.device)
        handle = ctypes.c_void_p()
        col = self.col_idx if self.e > 0 else torch.empty(4, dtype=torch.int32, device=self.device)
        rc = lib.gnn_graph_prepare(self.n, self.e, _ptr(self.row_ptr), _ptr(col),
                                   _ptr(self.buffer), nb, _ptr(scratch), ns, tref,
                                   _stream(stream, self.device), ctypes.byref(handle))
        _native.check(rc, "gnn_graph_prepare")
        self._col_keepalive = col
        self.handle = handle
        self._lib = lib

    def __del__(self):
        h = getattr(self, "handle", None)
        if h is not None and h.value:
            self._lib.gnn_graph_destroy(h)
            self.handle = None

    def stats(self) -> dict:
        arr = (ctypes.c_int64 * 16)()
        _native.check(self._lib.gnn_graph_stats(self.handle, arr, 16), "gnn_graph_stats")
        v = list(arr)
        keys = ["light", "items", "hubs", "hub_chunks", "max_deg", "max_item"]
        return dict(n=v[0], e=v[1], csr=dict(zip(keys, v[2:8])), csc=dict(zip(keys, v[8:14])),
                    light_max_deg=v[14], cta_max_deg=v[15])

    def arrays(self) -> dict:
        """Views (into this graph's buffer) of the prepared structures."""
        ptrs = (ctypes.c_void_p * 8)()
        _native.check(self._lib.gnn_graph_arrays(self.handle, ptrs, 8), "gnn_graph_arrays")
        st = self.stats()
        base = self.buffer.data_ptr()

        def view(p, count, width):
            off = p - base
            assert 0 <= off and off + 4 * width * count <= self.buffer.numel()
            return self.buffer[off:off + 4 * width * count].view(torch.int32).view(count, width) \
                if width > 1 else self.buffer[off:off + 4 * count].view(torch.int32)

        def nitems(d):
            return d["items"]
        return dict(
            col_ptr=view(ptrs[0], self.n + 1, 1), row_idx=view(ptrs[1], self.e, 1),
            csr_light=view(ptrs[2], st["csr"]["light"], 1),
            csr_items=view(ptrs[3], nitems(st["csr"]), 4),
            csr_hubs=view(ptrs[4], st["csr"]["hubs"], 4),
            csc_light=view(ptrs[5], st["csc"]["light"], 1),
            csc_items=view(ptrs[6], nitems(st["csc"]), 4),
            csc_hubs=view(ptrs[7], st["csc"]["hubs"], 4))

    def workspace_bytes(self, H: int, D: int, dtype: torch.dtype) -> int:
        return int(self._lib.gat_agg_workspace_bytes(self.handle, H, D, _dtype_code(dtype)))

    def workspace(self, H: int, D: int, dtype: torch.dtype) -> torch.Tensor:
        n = self.workspace_bytes(H, D, dtype)
        if n == 0:
            raise GnnError(_native.ERR_UNSUPPORTED, f"(H={H}, D={D}, {dtype})")
        return torch.empty(n, dtype=torch.uint8, device=self.device)


def _check_tensor(g: Graph, t, name: str, shape, dtype=None, floating=False):
    """Raise before any pointer reaches the library unless t is a contiguous
    tensor of the given shape (and dtype) on the graph's CUDA device."""
    if not isinstance(t, torch.Tensor):
        raise TypeError(f"{name} must be a torch.Tensor, got {type(t).__name__}")
    if shape is not None and tuple(t.shape) != tuple(shape):
        raise ValueError(f"{name} must have shape {tuple(shape)}, got {tuple(t.shape)}")
    if dtype is not None and t.dtype != dtype:
        raise TypeError(f"{name} must be {dtype}, got {t.dtype}")
    if floating and not t.is_floating_point():
        raise TypeError(f"{name} must be a floating-point tensor, got {t.dtype}")
    if not t.is_cuda or t.device != g.device:
        raise ValueError(f"{name} must be on the graph's device {g.device}, got {t.device}")
    if not t.is_contiguous():
        raise ValueError(f"{name} must be contiguous")
    return t


def _check_features(g: Graph, x: torch.Tensor, name: str):
    if not isinstance(x, torch.Tensor) or x.dim() != 3 or x.shape[0] != g.n:
        raise ValueError(f"{name} must be [N, H, D] with N = {g.n}")
    _dtype_code(x.dtype)
    _check_tensor(g, x, name, None)


def _att(g: Graph, a, name: str, H: int, D: int) -> torch.Tensor:
    """An attention vector [H, D] on the graph's device, widened to float32."""
    _check_tensor(g, a, name, (H, D), floating=True)
    return a.to(torch.float32).contiguous()


def _given(g: Graph, t, name: str, shape, dtype, make):
    """A caller-supplied output (checked) or a new one."""
    return make() if t is None else _check_tensor(g, t, name, shape, dtype)


def _check_ws(g: Graph, ws):
    if ws is not None:
        _check_tensor(g, ws, "ws", None, torch.uint8)
        if ws.dim() != 1:
            raise ValueError("ws must be a one-dimensional uint8 tensor")
    return ws


def gat_forward(g: Graph, h: torch.Tensor, a_src: torch.Tensor, a_dst: torch.Tensor,
                slope: float = 0.2, out=None, lse=None, ws=None, stream=None):
    """out [N,H,D] (h's dtype) and lse [N,H] float32."""
    _check_features(g, h, "h")
    N, H, D = h.shape
    dt = _dtype_code(h.dtype)
    a_src = _att(g, a_src, "a_src", H, D)
    a_dst = _att(g, a_dst, "a_dst", H, D)
    out = _given(g, out, "out", h.shape, h.dtype, lambda: torch.empty_like(h))
    lse = _given(g, lse, "lse", (N, H), torch.float32,
                 lambda: torch.empty((N, H), dtype=torch.float32, device=h.device))
    if _check_ws(g, ws) is None:
        ws = g.workspace(H, D, h.dtype)
    rc = g._lib.gat_agg_forward(g.handle, H, D, dt, _ptr(h), _ptr(a_src), _ptr(a_dst),
                                float(slope), _ptr(out), _ptr(lse), _ptr(ws), ws.numel(),
                                _stream(stream, h.device))
    _native.check(rc, "gat_agg_forward")
    return out, lse


def gat_backward(g: Graph, h: torch.Tensor, a_src: torch.Tensor, a_dst: torch.Tensor,
                 slope: float, lse: torch.Tensor, dout: torch.Tensor, dh=None, da_src=None,
                 da_dst=None, ws=None, stream=None, reuse_scores=False):
    """dh [N,H,D] (h's dtype), da_src and da_dst [H,D] float32.

    reuse_scores: ws is the workspace the gat_forward call on the same h,
    a_src, a_dst used, untouched since; the backward then takes the per-node
    scores that call left there instead of computing them again."""
    _check_features(g, h, "h")
    _check_features(g, dout, "dout")
    if dout.dtype != h.dtype:
        raise TypeError("dout must have h's dtype")
    N, H, D = h.shape
    dt = _dtype_code(h.dtype)
    a_src = _att(g, a_src, "a_src", H, D)
    a_dst = _att(g, a_dst, "a_dst", H, D)
    _check_tensor(g, lse, "lse", (N, H), torch.float32)
    dh = _given(g, dh, "dh", h.shape, h.dtype, lambda: torch.empty_like(h))
    da_src = _given(g, da_src, "da_src", (H, D), torch.float32,
                    lambda: torch.empty((H, D), dtype=torch.float32, device=h.device))
    da_dst = _given(g, da_dst, "da_dst", (H, D), torch.float32,
                    lambda: torch.empty((H, D), dtype=torch.float32, device=h.device))
    if _check_ws(g, ws) is None:
        if reuse_scores:
            raise ValueError("reuse_scores needs the forward call's workspace")
        ws = g.workspace(H, D, h.dtype)
    if reuse_scores:
        rc = g._lib.gat_agg_backward_reuse(g.handle, H, D, dt, _ptr(h), _ptr(a_src), _ptr(a_dst),
                                           float(slope), _ptr(lse), _ptr(dout), _ptr(dh),
                                           _ptr(da_src), _ptr(da_dst), _ptr(ws), ws.numel(),
                                           _stream(stream, h.device), None, 0)
    else:
        rc = g._lib.gat_agg_backward(g.handle, H, D, dt, _ptr(h), _ptr(a_src), _ptr(a_dst),
                                     float(slope), _ptr(lse), _ptr(dout), _ptr(dh), _ptr(da_src),
                                     _ptr(da_dst), _ptr(ws), ws.numel(), _stream(stream, h.device))
    _native.check(rc, "gat_agg_backward")
    return dh, da_src, da_dst


def _row_width(g: Graph, x: torch.Tensor, name: str) -> int:
    if not isinstance(x, torch.Tensor) or x.dim() < 2 or x.shape[0] != g.n:
        raise ValueError(f"{name} must be a tensor [N, ...] with N = {g.n}")
    _check_tensor(g, x, name, None)
    F = 1
    for d in x.shape[1:]:
        F *= d
    return F


def _gcn_call(fname, g, x, norm, out, ws, stream, what):
    F = _row_width(g, x, "features")
    dt = _dtype_code(x.dtype)
    if norm not in _native.NORMS:
        raise ValueError(f"norm must be one of {sorted(_native.NORMS)}")
    out = _given(g, out, "out", x.shape, x.dtype, lambda: torch.empty_like(x))
    if _check_ws(g, ws) is None:
        n = g._lib.gcn_agg_workspace_bytes(g.handle, F, dt)
        if n == 0:
            raise GnnError(_native.ERR_UNSUPPORTED, f"(F={F}, {x.dtype})")
        ws = torch.empty(n, dtype=torch.uint8, device=x.device)
    fn = getattr(g._lib, fname)
    rc = fn(g.handle, F, dt, _native.NORMS[norm], _ptr(x), _ptr(out), _ptr(ws), ws.numel(),
            _stream(stream, x.device))
    _native.check(rc, what)
    return out


def gcn_forward(g: Graph, x: torch.Tensor, norm: str = "sym", out=None, ws=None, stream=None):
    """out = A~ x (x [N, ...] float32 or bfloat16, features flattened per node)."""
    return _gcn_call("gcn_agg_forward", g, x, norm, out, ws, stream, "gcn_agg_forward")


def gcn_backward(g: Graph, dout: torch.Tensor, norm: str = "sym", dx=None, ws=None, stream=None):
    """dx = A~^T dout."""
    return _gcn_call("gcn_agg_backward", g, dout, norm, dx, ws, stream, "gcn_agg_backward")


class GCNAggregate(torch.autograd.Function):
    """out = GCNAggregate.apply(graph, x, norm)."""

    @staticmethod
    def forward(ctx, g, x, norm):
        ctx.g = g
        ctx.norm = norm
        return gcn_forward(g, x.contiguous(), norm)

    @staticmethod
    def backward(ctx, dout):
        return None, gcn_backward(ctx.g, dout.contiguous(), ctx.norm), None


def _gatv2_ws(g, H, D, dtype, ws, device):
    if ws is not None:
        return ws
    n = g._lib.gatv2_agg_workspace_bytes(g.handle, H, D, _dtype_code(dtype))
    if n == 0:
        raise GnnError(_native.ERR_UNSUPPORTED, f"(H={H}, D={D}, {dtype})")
    return torch.empty(n, dtype=torch.uint8, device=device)


def gatv2_forward(g: Graph, xl: torch.Tensor, xr: torch.Tensor, att: torch.Tensor,
                  slope: float = 0.2, out=None, lse=None, ws=None, stream=None):
    """out [N,H,D] (xl's dtype) and lse [N,H] float32."""
    _check_features(g, xl, "xl")
    _check_features(g, xr, "xr")
    if xr.shape != xl.shape or xr.dtype != xl.dtype:
        raise ValueError("xr must match xl in shape and dtype")
    N, H, D = xl.shape
    att = _att(g, att, "att", H, D)
    out = _given(g, out, "out", xl.shape, xl.dtype, lambda: torch.empty_like(xl))
    lse = _given(g, lse, "lse", (N, H), torch.float32,
                 lambda: torch.empty((N, H), dtype=torch.float32, device=xl.device))
    ws = _gatv2_ws(g, H, D, xl.dtype, _check_ws(g, ws), xl.device)
    rc = g._lib.gatv2_agg_forward(g.handle, H, D, _dtype_code(xl.dtype), _ptr(xl), _ptr(xr),
                                  _ptr(att), float(slope), _ptr(out), _ptr(lse), _ptr(ws),
                                  ws.numel(), _stream(stream, xl.device))
    _native.check(rc, "gatv2_agg_forward")
    return out, lse


def gatv2_backward(g: Graph, xl: torch.Tensor, xr: torch.Tensor, att: torch.Tensor,
                   slope: float, lse: torch.Tensor, dout: torch.Tensor, dxl=None, dxr=None,
                   datt=None, ws=None, stream=None):
    """dxl, dxr [N,H,D] (xl's dtype) and datt [H,D] float32."""
    _check_features(g, xl, "xl")
    _check_features(g, xr, "xr")
    _check_features(g, dout, "dout")
    if xr.shape != xl.shape or dout.shape != xl.shape or dout.dtype != xl.dtype:
        raise ValueError("xr and dout must match xl")
    N, H, D = xl.shape
    att = _att(g, att, "att", H, D)
    _check_tensor(g, lse, "lse", (N, H), torch.float32)
    dxl = _given(g, dxl, "dxl", xl.shape, xl.dtype, lambda: torch.empty_like(xl))
    dxr = _given(g, dxr, "dxr", xl.shape, xl.dtype, lambda: torch.empty_like(xl))
    datt = _given(g, datt, "datt", (H, D), torch.float32,
                  lambda: torch.empty((H, D), dtype=torch.float32, device=xl.device))
    ws = _gatv2_ws(g, H, D, xl.dtype, _check_ws(g, ws), xl.device)
    rc = g._lib.gatv2_agg_backward(g.handle, H, D, _dtype_code(xl.dtype), _ptr(xl), _ptr(xr),
                                   _ptr(att), float(slope), _ptr(lse), _ptr(dout),
                                   _ptr(dxl), _ptr(dxr), _ptr(datt), _ptr(ws), ws.numel(),
                                   _stream(stream, xl.device))
    _native.check(rc, "gatv2_agg_backward")
    return dxl, dxr, datt


class GATv2Aggregate(torch.autograd.Function):
    """out = GATv2Aggregate.apply(graph, xl, xr, att, slope)."""

    @staticmethod
    def forward(ctx, g, xl, xr, att, slope):
        xl, xr = xl.contiguous(), xr.contiguous()
        out, lse = gatv2_forward(g, xl, xr, att, slope)
        ctx.g, ctx.slope = g, slope
        ctx.save_for_backward(xl, xr, att, lse)
        return out

    @staticmethod
    def backward(ctx, dout):
        xl, xr, att, lse = ctx.saved_tensors
        dxl, dxr, datt = gatv2_backward(ctx.g, xl, xr, att, ctx.slope, lse, dout.contiguous())
        return None, dxl, dxr, datt.to(att.dtype), None


def _gt_ws(g, H, D, dtype, ws, device):
    if ws is not None:
        return ws
    n = g._lib.transformer_agg_workspace_bytes(g.handle, H, D, _dtype_code(dtype))
    if n == 0:
        raise GnnError(_native.ERR_UNSUPPORTED, f"(H={H}, D={D}, {dtype})")
    return torch.empty(n, dtype=torch.uint8, device=device)


def _gt_inputs(g, q, key, val):
    for name, x in (("q", q), ("key", key), ("val", val)):
        _check_features(g, x, name)
        if x.shape != q.shape or x.dtype != q.dtype:
            raise ValueError("q, key and val must share shape and dtype")
    return q.shape


def transformer_forward(g: Graph, q: torch.Tensor, key: torch.Tensor, val: torch.Tensor,
                        scale: float | None = None, out=None, lse=None, ws=None, stream=None):
    """out [N,H,D] (q's dtype) and lse [N,H] float32; scale defaults to 1/sqrt(D)."""
    N, H, D = _gt_inputs(g, q, key, val)
    scale = D ** -0.5 if scale is None else float(scale)
    out = _given(g, out, "out", q.shape, q.dtype, lambda: torch.empty_like(q))
    lse = _given(g, lse, "lse", (N, H), torch.float32,
                 lambda: torch.empty((N, H), dtype=torch.float32, device=q.device))
    ws = _gt_ws(g, H, D, q.dtype, _check_ws(g, ws), q.device)
    rc = g._lib.transformer_agg_forward(g.handle, H, D, _dtype_code(q.dtype), _ptr(q), _ptr(key),
                                        _ptr(val), scale, _ptr(out), _ptr(lse), _ptr(ws),
                                        ws.numel(), _stream(stream, q.device))
    _native.check(rc, "transformer_agg_forward")
    return out, lse


def transformer_backward(g: Graph, q: torch.Tensor, key: torch.Tensor, val: torch.Tensor,
                         lse: torch.Tensor, dout: torch.Tensor, scale: float | None = None,
                         dq=None, dkey=None, dval=None, ws=None, stream=None):
    """dq, dkey, dval [N,H,D] (q's dtype)."""
    N, H, D = _gt_inputs(g, q, key, val)
    _check_features(g, dout, "dout")
    if dout.shape != q.shape or dout.dtype != q.dtype:
        raise ValueError("dout must match q")
    scale = D ** -0.5 if scale is None else float(scale)
    _check_tensor(g, lse, "lse", (N, H), torch.float32)
    dq = _given(g, dq, "dq", q.shape, q.dtype, lambda: torch.empty_like(q))
    dkey = _given(g, dkey, "dkey", q.shape, q.dtype, lambda: torch.empty_like(q))
    dval = _given(g, dval, "dval", q.shape, q.dtype, lambda: torch.empty_like(q))
    ws = _gt_ws(g, H, D, q.dtype, _check_ws(g, ws), q.device)
    rc = g._lib.transformer_agg_backward(g.handle, H, D, _dtype_code(q.dtype), _ptr(q),
                                         _ptr(key), _ptr(val), scale, _ptr(lse),
                                         _ptr(dout), _ptr(dq), _ptr(dkey), _ptr(dval), _ptr(ws),
                                         ws.numel(), _stream(stream, q.device))
    _native.check(rc, "transformer_agg_backward")
    return dq, dkey, dval


class TransformerAggregate(torch.autograd.Function):
    """out = TransformerAggregate.apply(graph, q, key, val, scale)."""

    @staticmethod
    def forward(ctx, g, q, key, val, scale):
        q, key, val = q.contiguous(), key.contiguous(), val.contiguous()
        out, lse = transformer_forward(g, q, key, val, scale)
        ctx.g, ctx.scale = g, scale
        ctx.save_for_backward(q, key, val, lse)
        return out

    @staticmethod
    def backward(ctx, dout):
        q, key, val, lse = ctx.saved_tensors
        dq, dk, dv = transformer_backward(ctx.g, q, key, val, lse, dout.contiguous(), ctx.scale)
        return None, dq, dk, dv, None


def _reduce_ws(g, F, dt, ws, device):
    if ws is not None:
        return ws
    n = g._lib.reduce_agg_workspace_bytes(g.handle, F, dt)
    if n == 0:
        raise GnnError(_native.ERR_UNSUPPORTED, f"(F={F})")
    return torch.empty(n, dtype=torch.uint8, device=device)


def reduce_forward(g: Graph, x: torch.Tensor, op: str = "max", out=None, arg=None, ws=None,
                   stream=None):
    """out [N, ...] (x's dtype) = max or min over in-neighbours, feature by
    feature; arg int32 of the same shape = the winning source (-1: none)."""
    F = _row_width(g, x, "x")
    dt = _dtype_code(x.dtype)
    if op not in _native.REDUCE_OPS:
        raise ValueError(f"op must be one of {sorted(_native.REDUCE_OPS)}")
    out = _given(g, out, "out", x.shape, x.dtype, lambda: torch.empty_like(x))
    arg = _given(g, arg, "arg", x.shape, torch.int32,
                 lambda: torch.empty(x.shape, dtype=torch.int32, device=x.device))
    ws = _reduce_ws(g, F, dt, _check_ws(g, ws), x.device)
    rc = g._lib.reduce_agg_forward(g.handle, F, dt, _native.REDUCE_OPS[op], _ptr(x), _ptr(out),
                                   _ptr(arg), _ptr(ws), ws.numel(), _stream(stream, x.device))
    _native.check(rc, "reduce_agg_forward")
    return out, arg


def reduce_backward(g: Graph, arg: torch.Tensor, dout: torch.Tensor, dx=None, ws=None,
                    stream=None, ordered=False):
    """dx = the gradient of sum(out * dout) w.r.t. x, from the forward's arg.

    ordered: gather the terms over the cached CSC in a fixed order instead of
    adding them with atomics (bitwise reproducible, more bytes moved)."""
    F = _row_width(g, dout, "dout")
    _check_tensor(g, arg, "arg", dout.shape, torch.int32)
    dt = _dtype_code(dout.dtype)
    dx = _given(g, dx, "dx", dout.shape, dout.dtype, lambda: torch.empty_like(dout))
    ws = _reduce_ws(g, F, dt, _check_ws(g, ws), dout.device)
    fn = g._lib.reduce_agg_backward_ordered if ordered else g._lib.reduce_agg_backward
    rc = fn(g.handle, F, dt, _ptr(arg), _ptr(dout), _ptr(dx), _ptr(ws), ws.numel(),
            _stream(stream, dout.device))
    _native.check(rc, "reduce_agg_backward_ordered" if ordered else "reduce_agg_backward")
    return dx


class ReduceAggregate(torch.autograd.Function):
    """out = ReduceAggregate.apply(graph, x, op)."""

    @staticmethod
    def forward(ctx, g, x, op):
        out, arg = reduce_forward(g, x.contiguous(), op)
        ctx.g = g
        ctx.save_for_backward(arg)
        ctx.mark_non_differentiable(arg)
        return out

    @staticmethod
    def backward(ctx, dout):
        (arg,) = ctx.saved_tensors
        return None, reduce_backward(ctx.g, arg, dout.contiguous()), None


def check_device_error(g: Graph, stream=None) -> int:
    """Synchronise and read the graph's device status word (raises on error)."""
    info = ctypes.c_int32(0)
    rc = g._lib.gnn_check_device_error(g.handle, _stream(stream, g.device), ctypes.byref(info))
    _native.check(rc, "gnn_check_device_error")
    return info.value


class GATAggregate(torch.autograd.Function):
    """out = GATAggregate.apply(graph, h, a_src, a_dst, slope)."""

    @staticmethod
    def forward(ctx, g, h, a_src, a_dst, slope):
        h = h.contiguous()
        ws = g.workspace(h.shape[1], h.shape[2], h.dtype)
        out, lse = gat_forward(g, h, a_src, a_dst, slope, ws=ws)
        ctx.g = g
        ctx.slope = slope
        ctx.ws = ws  # its per-node scores serve the backward; nothing else writes it
        ctx.save_for_backward(h, a_src, a_dst, lse)
        return out

    @staticmethod
    def backward(ctx, dout):
        h, a_src, a_dst, lse = ctx.saved_tensors
        dh, da_s, da_d = gat_backward(ctx.g, h, a_src, a_dst, ctx.slope, lse, dout.contiguous(),
                                      ws=ctx.ws, reuse_scores=True)
        return None, dh, da_s.to(a_src.dtype), da_d.to(a_dst.dtype), None
