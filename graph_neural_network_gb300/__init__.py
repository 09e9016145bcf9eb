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
"""
from __future__ import annotations

import ctypes

import torch

from . import _native
from ._native import GnnError, Tiling

__all__ = ["Graph", "gat_forward", "gat_backward", "GATAggregate", "GnnError", "Tiling",
           "check_device_error", "default_tiling", "gcn_forward", "gcn_backward",
           "GCNAggregate"]


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


def _check_features(g: Graph, x: torch.Tensor, name: str):
    if x.dim() != 3 or x.shape[0] != g.n:
        raise ValueError(f"{name} must be [N, H, D] with N = {g.n}")
    if not x.is_cuda or not x.is_contiguous():
        raise ValueError(f"{name} must be a contiguous CUDA tensor")


def gat_forward(g: Graph, h: torch.Tensor, a_src: torch.Tensor, a_dst: torch.Tensor,
                slope: float = 0.2, out=None, lse=None, ws=None, stream=None):
    """out [N,H,D] (h's dtype) and lse [N,H] float32."""
    _check_features(g, h, "h")
    N, H, D = h.shape
    dt = _dtype_code(h.dtype)
    a_src = a_src.to(torch.float32).contiguous()
    a_dst = a_dst.to(torch.float32).contiguous()
    if out is None:
        out = torch.empty_like(h)
    if lse is None:
        lse = torch.empty((N, H), dtype=torch.float32, device=h.device)
    if ws is None:
        ws = g.workspace(H, D, h.dtype)
    rc = g._lib.gat_agg_forward(g.handle, H, D, dt, _ptr(h), _ptr(a_src), _ptr(a_dst),
                                float(slope), _ptr(out), _ptr(lse), _ptr(ws), ws.numel(),
                                _stream(stream, h.device))
    _native.check(rc, "gat_agg_forward")
    return out, lse


def gat_backward(g: Graph, h: torch.Tensor, a_src: torch.Tensor, a_dst: torch.Tensor,
                 slope: float, lse: torch.Tensor, dout: torch.Tensor, dh=None, da_src=None,
                 da_dst=None, ws=None, stream=None):
    """dh [N,H,D] (h's dtype), da_src and da_dst [H,D] float32."""
    _check_features(g, h, "h")
    _check_features(g, dout, "dout")
    if dout.dtype != h.dtype:
        raise TypeError("dout must have h's dtype")
    N, H, D = h.shape
    dt = _dtype_code(h.dtype)
    a_src = a_src.to(torch.float32).contiguous()
    a_dst = a_dst.to(torch.float32).contiguous()
    lse = lse.contiguous()
    if dh is None:
        dh = torch.empty_like(h)
    if da_src is None:
        da_src = torch.empty((H, D), dtype=torch.float32, device=h.device)
    if da_dst is None:
        da_dst = torch.empty((H, D), dtype=torch.float32, device=h.device)
    if ws is None:
        ws = g.workspace(H, D, h.dtype)
    rc = g._lib.gat_agg_backward(g.handle, H, D, dt, _ptr(h), _ptr(a_src), _ptr(a_dst),
                                 float(slope), _ptr(lse), _ptr(dout), _ptr(dh), _ptr(da_src),
                                 _ptr(da_dst), _ptr(ws), ws.numel(), _stream(stream, h.device))
    _native.check(rc, "gat_agg_backward")
    return dh, da_src, da_dst


def _row_width(g: Graph, x: torch.Tensor, name: str) -> int:
    if x.dim() < 2 or x.shape[0] != g.n or not x.is_cuda or not x.is_contiguous():
        raise ValueError(f"{name} must be a contiguous CUDA tensor [N, ...] with N = {g.n}")
    F = 1
    for d in x.shape[1:]:
        F *= d
    return F


def _gcn_call(fn, g, x, norm, out, ws, stream, what):
    F = _row_width(g, x, "features")
    dt = _dtype_code(x.dtype)
    if norm not in _native.NORMS:
        raise ValueError(f"norm must be one of {sorted(_native.NORMS)}")
    if out is None:
        out = torch.empty_like(x)
    if ws is None:
        n = g._lib.gcn_agg_workspace_bytes(g.handle, F, dt)
        if n == 0:
            raise GnnError(_native.ERR_UNSUPPORTED, f"(F={F}, {x.dtype})")
        ws = torch.empty(n, dtype=torch.uint8, device=x.device)
    rc = fn(g.handle, F, dt, _native.NORMS[norm], _ptr(x), _ptr(out), _ptr(ws), ws.numel(),
            _stream(stream, x.device))
    _native.check(rc, what)
    return out


def gcn_forward(g: Graph, x: torch.Tensor, norm: str = "sym", out=None, ws=None, stream=None):
    """out = A~ x (x [N, ...] float32 or bfloat16, features flattened per node)."""
    return _gcn_call(g._lib.gcn_agg_forward, g, x, norm, out, ws, stream, "gcn_agg_forward")


def gcn_backward(g: Graph, dout: torch.Tensor, norm: str = "sym", dx=None, ws=None, stream=None):
    """dx = A~^T dout."""
    return _gcn_call(g._lib.gcn_agg_backward, g, dout, norm, dx, ws, stream, "gcn_agg_backward")


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
        out, lse = gat_forward(g, h, a_src, a_dst, slope)
        ctx.g = g
        ctx.slope = slope
        ctx.save_for_backward(h, a_src, a_dst, lse)
        return out

    @staticmethod
    def backward(ctx, dout):
        h, a_src, a_dst, lse = ctx.saved_tensors
        dh, da_s, da_d = gat_backward(ctx.g, h, a_src, a_dst, ctx.slope, lse, dout.contiguous())
        return None, dh, da_s.to(a_src.dtype), da_d.to(a_dst.dtype), None
