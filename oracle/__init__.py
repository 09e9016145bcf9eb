"""fp64 CPU oracles of the neighbour aggregations (ctypes wrapper).

TEST INFRASTRUCTURE ONLY: imported by ``tests/``, by the smoke check in
``__graft_entry__`` and by the CPU-baseline leg of ``bench.py``; never by the
product package.  It shares no code with the CUDA library.  See
``gat_oracle.c`` (fused GAT attention), ``gatv2_oracle.c`` (fused GATv2
attention), ``transformer_oracle.c`` (graph-transformer attention),
``spmm_oracle.c`` (GCN / GraphConv propagation) and ``reduce_oracle.c`` (max /
min neighbourhood reduction) for what each computes and which passages it
follows.

Arrays: ``h`` and ``dout`` are float32 ``[N, H, D]``, uint16 bit patterns of
bfloat16 ``[N, H, D]``, or float64 (finite-difference checks); ``a_src`` /
``a_dst`` ``[H, D]`` (float32 or float64).
Every result is float64.
"""
from __future__ import annotations

import ctypes
import os
import subprocess
import threading

import numpy as np

_HERE = os.path.dirname(os.path.abspath(__file__))
_SRC = os.path.join(_HERE, "gat_oracle.c")
_SOURCES = ["gat_oracle.c", "spmm_oracle.c", "reduce_oracle.c", "gatv2_oracle.c",
            "transformer_oracle.c"]
_LIB = os.path.join(_HERE, "liboracle.so")
_lock = threading.Lock()
_lib = None


def build(force: bool = False) -> str:
    """Compile ``liboracle.so`` (gcc, OpenMP) next to this file when stale."""
    srcs = [os.path.join(_HERE, f) for f in _SOURCES]
    if (not force and os.path.exists(_LIB)
            and all(os.path.getmtime(_LIB) >= os.path.getmtime(f) for f in srcs)):
        return _LIB
    tmp = _LIB + f".tmp{os.getpid()}"
    subprocess.check_call(["gcc", "-O2", "-std=c99", "-fopenmp", "-fPIC", "-shared"] + srcs +
                          ["-o", tmp, "-lm"])
    os.replace(tmp, _LIB)
    return _LIB


def _bind(path: str):
    lib = ctypes.CDLL(path)
    P, i64, i32, f64 = ctypes.c_void_p, ctypes.c_int64, ctypes.c_int, ctypes.c_double
    common = [i64, P, P, i32, i32, i32, P, P, P, f64]
    lib.oracle_gat_forward.argtypes = common + [i64, P, P, P, P, P]
    lib.oracle_gat_forward.restype = i32
    lib.oracle_gat_node_stats.argtypes = common + [P, i64, P, P, P, P]
    lib.oracle_gat_node_stats.restype = i32
    lib.oracle_gat_backward.argtypes = common + [P, P, P, P, P, P, P, P]
    lib.oracle_gat_backward.restype = i32
    lib.oracle_gat_backward_rows.argtypes = common + [P, i64, P, P, P, P]
    lib.oracle_gat_backward_rows.restype = i32
    lib.oracle_gat_att_grads.argtypes = common + [P, P, P, P, P]
    lib.oracle_gat_att_grads.restype = i32
    spmm = [i64, P, P, i64, i32, P, i32]
    lib.oracle_spmm_forward.argtypes = spmm + [i64, P, P, P]
    lib.oracle_spmm_forward.restype = i32
    lib.oracle_spmm_backward.argtypes = spmm + [P, P]
    lib.oracle_spmm_backward.restype = i32
    lib.oracle_spmm_backward_rows.argtypes = spmm + [i64, P, P, P]
    lib.oracle_spmm_backward_rows.restype = i32
    lib.oracle_reduce_forward.argtypes = [i64, P, P, i64, i32, P, i32, i64, P, P, P]
    lib.oracle_reduce_forward.restype = i32
    lib.oracle_reduce_backward.argtypes = [i64, i64, i32, P, P, P, P]
    lib.oracle_reduce_backward.restype = i32
    lib.oracle_reduce_backward_rows.argtypes = [i64, P, P, i64, i32, P, i32, P, i64, P, P, P]
    lib.oracle_reduce_backward_rows.restype = i32
    v2 = [i64, P, P, i32, i32, i32, P, P, P, f64]
    lib.oracle_gatv2_forward.argtypes = v2 + [i64, P, P, P, P, P]
    lib.oracle_gatv2_forward.restype = i32
    lib.oracle_gatv2_delta.argtypes = v2 + [P, i64, P, P]
    lib.oracle_gatv2_delta.restype = i32
    lib.oracle_gatv2_backward.argtypes = v2 + [P, i64, P, P, P, P, P, P, P]
    lib.oracle_gatv2_backward.restype = i32
    gt = [i64, P, P, i32, i32, i32, P, P, P, f64]
    lib.oracle_gt_forward.argtypes = gt + [i64, P, P, P, P, P]
    lib.oracle_gt_forward.restype = i32
    lib.oracle_gt_backward.argtypes = gt + [P, i64, P, P, P, P, P, P, P]
    lib.oracle_gt_backward.restype = i32
    lib.oracle_num_threads.argtypes = []
    lib.oracle_num_threads.restype = i32
    lib.oracle_set_threads.argtypes = [i32]
    lib.oracle_set_threads.restype = None
    return lib


def _load():
    global _lib
    with _lock:
        if _lib is None:
            build()
            _lib = _bind(_LIB)
        return _lib


def compile_variant(source_text: str, out_path: str, name: str = "gat_oracle.c") -> str:
    """Compile the oracle library with the source file `name` replaced by a
    modified copy (used by tests that plant a mistake in the oracle to show
    that the pins catch it)."""
    srcs = []
    for f in _SOURCES:
        if f == name:
            src = out_path + "." + f
            with open(src, "w") as fh:
                fh.write(source_text)
            srcs.append(src)
        else:
            srcs.append(os.path.join(_HERE, f))
    subprocess.check_call(["gcc", "-O2", "-std=c99", "-fopenmp", "-fPIC", "-shared"] + srcs +
                          ["-o", out_path, "-lm"])
    return out_path


def source_text(name: str = "gat_oracle.c") -> str:
    with open(os.path.join(_HERE, name)) as f:
        return f.read()


class Oracle:
    """The oracle's entry points bound to one compiled library."""

    def __init__(self, path: str | None = None):
        self._path = path

    @property
    def lib(self):
        if self._path is None:
            return _load()
        if not hasattr(self, "_lib"):
            self._lib = _bind(self._path)
        return self._lib

    def num_threads(self) -> int:
        return int(self.lib.oracle_num_threads())

    def set_threads(self, n: int) -> None:
        """Threads of the oracle's later calls (no effect on the results)."""
        self.lib.oracle_set_threads(int(n))

    def forward(self, row_ptr, col, h, a_src, a_dst, slope, sel=None, with_mag=False, with_alpha_sum=False):
        row_ptr, col, h, a_src, a_dst, n, H, D, dt = _prep(row_ptr, col, h, a_src, a_dst)
        sel = _sel(sel)
        m = n if sel is None else len(sel)
        out = np.empty((m, H, D), np.float64)
        lse = np.empty((m, H), np.float64)
        mag = np.empty((m, H, D), np.float64) if with_mag else None
        asum = np.empty((m, H), np.float64) if with_alpha_sum else None
        rc = self.lib.oracle_gat_forward(n, _p(row_ptr), _p(col), H, D, dt, _p(h), _p(a_src), _p(a_dst),
                                        float(slope), 0 if sel is None else len(sel), _p(sel),
                                        _p(out), _p(lse), _p(mag), _p(asum))
        _check(rc, "forward")
        return dict(out=out, lse=lse, out_mag=mag, alpha_sum=asum)

    def node_stats(self, row_ptr, col, h, a_src, a_dst, slope, dout, sel=None):
        """lse, Delta (= sum_j alpha_ij dout_i . h_j) and ds_dst per (node, head)."""
        row_ptr, col, h, a_src, a_dst, n, H, D, dt = _prep(row_ptr, col, h, a_src, a_dst)
        dout = np.ascontiguousarray(dout)
        assert dout.shape == h.shape and dout.dtype == h.dtype
        sel = _sel(sel)
        m = n if sel is None else len(sel)
        lse, delta, ds = (np.empty((m, H), np.float64) for _ in range(3))
        rc = self.lib.oracle_gat_node_stats(n, _p(row_ptr), _p(col), H, D, dt, _p(h), _p(a_src),
                                           _p(a_dst), float(slope), _p(dout),
                                           0 if sel is None else len(sel), _p(sel),
                                           _p(lse), _p(delta), _p(ds))
        _check(rc, "node_stats")
        return dict(lse=lse, delta=delta, ds_dst=ds)

    def backward(self, row_ptr, col, h, a_src, a_dst, slope, dout, with_mag=False,
                 with_kink=False):
        """Whole-graph backward.  with_kink adds, per element, how far dh and da
        can move between the two LeakyReLU derivatives of edges whose z lies
        within float32 rounding of the kink (dh_kink, da_src_kink, da_dst_kink)."""
        row_ptr, col, h, a_src, a_dst, n, H, D, dt = _prep(row_ptr, col, h, a_src, a_dst)
        dout = np.ascontiguousarray(dout)
        assert dout.shape == h.shape and dout.dtype == h.dtype
        dh = np.empty((n, H, D), np.float64)
        da_src = np.empty((H, D), np.float64)
        da_dst = np.empty((H, D), np.float64)
        dh_mag = np.empty((n, H, D), np.float64) if with_mag else None
        da_mag = np.empty((2, H, D), np.float64) if with_mag else None
        dh_kink = np.empty((n, H, D), np.float64) if with_kink else None
        da_kink = np.empty((2, H, D), np.float64) if with_kink else None
        rc = self.lib.oracle_gat_backward(n, _p(row_ptr), _p(col), H, D, dt, _p(h), _p(a_src),
                                         _p(a_dst), float(slope), _p(dout), _p(dh), _p(da_src),
                                         _p(da_dst), _p(dh_mag), _p(da_mag), _p(dh_kink),
                                         _p(da_kink))
        _check(rc, "backward")
        return dict(dh=dh, da_src=da_src, da_dst=da_dst, dh_mag=dh_mag,
                    da_src_mag=None if da_mag is None else da_mag[0],
                    da_dst_mag=None if da_mag is None else da_mag[1], dh_kink=dh_kink,
                    da_src_kink=None if da_kink is None else da_kink[0],
                    da_dst_kink=None if da_kink is None else da_kink[1])

    def att_grads(self, row_ptr, col, h, a_src, a_dst, slope, dout, with_mag=False,
                  with_kink=False):
        """da_src, da_dst summed per destination row (parallel over rows)."""
        row_ptr, col, h, a_src, a_dst, n, H, D, dt = _prep(row_ptr, col, h, a_src, a_dst)
        dout = np.ascontiguousarray(dout)
        assert dout.shape == h.shape and dout.dtype == h.dtype
        da_src = np.empty((H, D), np.float64)
        da_dst = np.empty((H, D), np.float64)
        mag = np.empty((2, H, D), np.float64) if with_mag else None
        kink = np.empty((2, H, D), np.float64) if with_kink else None
        rc = self.lib.oracle_gat_att_grads(n, _p(row_ptr), _p(col), H, D, dt, _p(h), _p(a_src),
                                           _p(a_dst), float(slope), _p(dout), _p(da_src),
                                           _p(da_dst), _p(mag), _p(kink))
        _check(rc, "att_grads")
        return dict(da_src=da_src, da_dst=da_dst,
                    da_src_mag=None if mag is None else mag[0],
                    da_dst_mag=None if mag is None else mag[1],
                    da_src_kink=None if kink is None else kink[0],
                    da_dst_kink=None if kink is None else kink[1])

    def backward_rows(self, row_ptr, col, h, a_src, a_dst, slope, dout, sel, with_mag=False,
                      with_kink=False):
        """dh rows of the listed (distinct) nodes only, each from its neighbourhood."""
        row_ptr, col, h, a_src, a_dst, n, H, D, dt = _prep(row_ptr, col, h, a_src, a_dst)
        dout = np.ascontiguousarray(dout)
        assert dout.shape == h.shape and dout.dtype == h.dtype
        sel = _sel(sel)
        dh = np.empty((len(sel), H, D), np.float64)
        dh_mag = np.empty((len(sel), H, D), np.float64) if with_mag else None
        dh_kink = np.empty((len(sel), H, D), np.float64) if with_kink else None
        rc = self.lib.oracle_gat_backward_rows(n, _p(row_ptr), _p(col), H, D, dt, _p(h), _p(a_src),
                                              _p(a_dst), float(slope), _p(dout), len(sel), _p(sel),
                                              _p(dh), _p(dh_mag), _p(dh_kink))
        _check(rc, "backward_rows")
        return dict(dh=dh, dh_mag=dh_mag, dh_kink=dh_kink)


    # ---- SpMM family (spmm_oracle.c) ----------------------------------------

    NORMS = {"sum": 0, "mean": 1, "sym": 2}

    def spmm_forward(self, row_ptr, col, x, norm, sel=None, with_mag=False):
        """out = A~ x for x [N, F] (or [N, H, D], flattened per node)."""
        row_ptr, col, x, n, F, dt = _prep_rows(row_ptr, col, x)
        sel = _sel(sel)
        m = n if sel is None else len(sel)
        out = np.empty((m, F), np.float64)
        mag = np.empty((m, F), np.float64) if with_mag else None
        rc = self.lib.oracle_spmm_forward(n, _p(row_ptr), _p(col), F, dt, _p(x),
                                          self.NORMS[norm], 0 if sel is None else len(sel),
                                          _p(sel), _p(out), _p(mag))
        _check(rc, "spmm_forward")
        return dict(out=out, out_mag=mag)

    def spmm_backward(self, row_ptr, col, dout, norm, with_mag=False):
        """dx = A~^T dout over the whole graph."""
        row_ptr, col, dout, n, F, dt = _prep_rows(row_ptr, col, dout)
        dx = np.empty((n, F), np.float64)
        mag = np.empty((n, F), np.float64) if with_mag else None
        rc = self.lib.oracle_spmm_backward(n, _p(row_ptr), _p(col), F, dt, _p(dout),
                                           self.NORMS[norm], _p(dx), _p(mag))
        _check(rc, "spmm_backward")
        return dict(dx=dx, dx_mag=mag)

    def spmm_backward_rows(self, row_ptr, col, dout, norm, sel, with_mag=False):
        """dx rows of the listed (distinct) nodes only."""
        row_ptr, col, dout, n, F, dt = _prep_rows(row_ptr, col, dout)
        sel = _sel(sel)
        dx = np.empty((len(sel), F), np.float64)
        mag = np.empty((len(sel), F), np.float64) if with_mag else None
        rc = self.lib.oracle_spmm_backward_rows(n, _p(row_ptr), _p(col), F, dt, _p(dout),
                                                self.NORMS[norm], len(sel), _p(sel), _p(dx),
                                                _p(mag))
        _check(rc, "spmm_backward_rows")
        return dict(dx=dx, dx_mag=mag)

    # ---- reduction family (reduce_oracle.c) ---------------------------------

    OPS = {"max": 0, "min": 1}

    def reduce_forward(self, row_ptr, col, x, op, sel=None):
        """out [N, F] (float64) and arg [N, F] (int32, -1 for no in-neighbours)."""
        row_ptr, col, x, n, F, dt = _prep_rows(row_ptr, col, x)
        sel = _sel(sel)
        m = n if sel is None else len(sel)
        out = np.empty((m, F), np.float64)
        arg = np.empty((m, F), np.int32)
        rc = self.lib.oracle_reduce_forward(n, _p(row_ptr), _p(col), F, dt, _p(x), self.OPS[op],
                                            0 if sel is None else len(sel), _p(sel), _p(out),
                                            _p(arg))
        _check(rc, "reduce_forward")
        return dict(out=out, arg=arg)

    def reduce_backward(self, arg, dout, with_mag=False):
        """dx [N, F] from the forward's arg and dout [N, F]."""
        arg = np.ascontiguousarray(arg, np.int32)
        dout = np.ascontiguousarray(dout)
        n = arg.shape[0]
        F = arg.size // max(1, n)
        dt = {np.dtype(np.float32): 0, np.dtype(np.uint16): 1, np.dtype(np.float64): 2}[dout.dtype]
        assert dout.size == arg.size
        dx = np.empty((n, F), np.float64)
        mag = np.empty((n, F), np.float64) if with_mag else None
        rc = self.lib.oracle_reduce_backward(n, F, dt, _p(arg), _p(dout), _p(dx), _p(mag))
        _check(rc, "reduce_backward")
        return dict(dx=dx, dx_mag=mag)

    def reduce_backward_rows(self, row_ptr, col, x, op, dout, sel, with_mag=False):
        """dx rows of the listed (distinct) sources, recomputing the reductions."""
        row_ptr, col, x, n, F, dt = _prep_rows(row_ptr, col, x)
        dout = np.ascontiguousarray(dout).reshape(n, F)
        assert dout.dtype == x.dtype
        sel = _sel(sel)
        dx = np.empty((len(sel), F), np.float64)
        mag = np.empty((len(sel), F), np.float64) if with_mag else None
        rc = self.lib.oracle_reduce_backward_rows(n, _p(row_ptr), _p(col), F, dt, _p(x),
                                                  self.OPS[op], _p(dout), len(sel), _p(sel),
                                                  _p(dx), _p(mag))
        _check(rc, "reduce_backward_rows")
        return dict(dx=dx, dx_mag=mag)

    # ---- GATv2 (gatv2_oracle.c) ---------------------------------------------

    def gatv2_forward(self, row_ptr, col, xl, xr, att, slope, sel=None, with_mag=False,
                      with_alpha_sum=False):
        row_ptr, col, xl, att, _, n, H, D, dt = _prep(row_ptr, col, xl, att, att)
        xr = _same(xr, xl)
        sel = _sel(sel)
        m = n if sel is None else len(sel)
        out = np.empty((m, H, D), np.float64)
        lse = np.empty((m, H), np.float64)
        mag = np.empty((m, H, D), np.float64) if with_mag else None
        asum = np.empty((m, H), np.float64) if with_alpha_sum else None
        rc = self.lib.oracle_gatv2_forward(n, _p(row_ptr), _p(col), H, D, dt, _p(xl), _p(xr),
                                           _p(att), float(slope), 0 if sel is None else len(sel),
                                           _p(sel), _p(out), _p(lse), _p(mag), _p(asum))
        _check(rc, "gatv2_forward")
        return dict(out=out, lse=lse, out_mag=mag, alpha_sum=asum)

    def gatv2_delta(self, row_ptr, col, xl, xr, att, slope, dout, sel=None):
        row_ptr, col, xl, att, _, n, H, D, dt = _prep(row_ptr, col, xl, att, att)
        xr, dout = _same(xr, xl), _same(dout, xl)
        sel = _sel(sel)
        m = n if sel is None else len(sel)
        delta = np.empty((m, H), np.float64)
        rc = self.lib.oracle_gatv2_delta(n, _p(row_ptr), _p(col), H, D, dt, _p(xl), _p(xr),
                                         _p(att), float(slope), _p(dout),
                                         0 if sel is None else len(sel), _p(sel), _p(delta))
        _check(rc, "gatv2_delta")
        return delta

    def gatv2_backward(self, row_ptr, col, xl, xr, att, slope, dout, sel=None, with_mag=False):
        """dxl, dxr (rows of sel, or all), datt (whole graph)."""
        row_ptr, col, xl, att, _, n, H, D, dt = _prep(row_ptr, col, xl, att, att)
        xr, dout = _same(xr, xl), _same(dout, xl)
        sel = _sel(sel)
        m = n if sel is None else len(sel)
        dxl, dxr = np.empty((m, H, D)), np.empty((m, H, D))
        datt = np.empty((H, D))
        mags = [np.empty((m, H, D)), np.empty((m, H, D)), np.empty((H, D))] if with_mag \
            else [None, None, None]
        rc = self.lib.oracle_gatv2_backward(n, _p(row_ptr), _p(col), H, D, dt, _p(xl), _p(xr),
                                            _p(att), float(slope), _p(dout),
                                            0 if sel is None else len(sel), _p(sel), _p(dxl),
                                            _p(dxr), _p(datt), *[_p(x) for x in mags])
        _check(rc, "gatv2_backward")
        return dict(dxl=dxl, dxr=dxr, datt=datt, dxl_mag=mags[0], dxr_mag=mags[1],
                    datt_mag=mags[2])

    # ---- graph transformer (transformer_oracle.c) ---------------------------

    def gt_forward(self, row_ptr, col, q, key, val, scale, sel=None, with_mag=False,
                   with_alpha_sum=False):
        row_ptr, col, q, _, _, n, H, D, dt = _prep(row_ptr, col, q, np.zeros(q.shape[1:]),
                                                   np.zeros(q.shape[1:]))
        key, val = _same(key, q), _same(val, q)
        sel = _sel(sel)
        m = n if sel is None else len(sel)
        out = np.empty((m, H, D), np.float64)
        lse = np.empty((m, H), np.float64)
        mag = np.empty((m, H, D), np.float64) if with_mag else None
        asum = np.empty((m, H), np.float64) if with_alpha_sum else None
        rc = self.lib.oracle_gt_forward(n, _p(row_ptr), _p(col), H, D, dt, _p(q), _p(key),
                                        _p(val), float(scale), 0 if sel is None else len(sel),
                                        _p(sel), _p(out), _p(lse), _p(mag), _p(asum))
        _check(rc, "gt_forward")
        return dict(out=out, lse=lse, out_mag=mag, alpha_sum=asum)

    def gt_backward(self, row_ptr, col, q, key, val, scale, dout, sel=None, with_mag=False):
        """dq, dkey, dval (rows of sel, or all nodes)."""
        row_ptr, col, q, _, _, n, H, D, dt = _prep(row_ptr, col, q, np.zeros(q.shape[1:]),
                                                   np.zeros(q.shape[1:]))
        key, val, dout = _same(key, q), _same(val, q), _same(dout, q)
        sel = _sel(sel)
        m = n if sel is None else len(sel)
        outs = [np.empty((m, H, D)) for _ in range(3)]
        mags = [np.empty((m, H, D)) for _ in range(3)] if with_mag else [None] * 3
        rc = self.lib.oracle_gt_backward(n, _p(row_ptr), _p(col), H, D, dt, _p(q), _p(key),
                                         _p(val), float(scale), _p(dout),
                                         0 if sel is None else len(sel), _p(sel),
                                         *[_p(x) for x in outs], *[_p(x) for x in mags])
        _check(rc, "gt_backward")
        return dict(dq=outs[0], dkey=outs[1], dval=outs[2], dq_mag=mags[0], dkey_mag=mags[1],
                    dval_mag=mags[2])


def _same(x, like):
    x = np.ascontiguousarray(x)
    if x.shape != like.shape or x.dtype != like.dtype:
        raise ValueError("arrays must share shape and dtype")
    return x


def _prep_rows(row_ptr, col, x):
    row_ptr = np.ascontiguousarray(row_ptr, dtype=np.int32)
    col = np.ascontiguousarray(col, dtype=np.int32)
    x = np.ascontiguousarray(x)
    dt = {np.dtype(np.float32): 0, np.dtype(np.uint16): 1, np.dtype(np.float64): 2}.get(x.dtype)
    if dt is None:
        raise TypeError("features must be float32, float64 or bfloat16 bit patterns (uint16)")
    n = x.shape[0]
    F = int(np.prod(x.shape[1:])) if x.ndim > 1 else 1
    if len(row_ptr) != n + 1:
        raise ValueError("row_ptr must have N + 1 entries")
    return row_ptr, col, x.reshape(n, F), n, F, dt


def _p(a):
    return None if a is None else ctypes.c_void_p(a.ctypes.data)


def _prep(row_ptr, col, h, a_src, a_dst):
    row_ptr = np.ascontiguousarray(row_ptr, dtype=np.int32)
    col = np.ascontiguousarray(col, dtype=np.int32)
    if h.dtype == np.uint16:
        dtype = 1
    elif h.dtype == np.float32:
        dtype = 0
    elif h.dtype == np.float64:
        dtype = 2
    else:
        raise TypeError("h must be float32, float64 or bfloat16 bit patterns (uint16)")
    h = np.ascontiguousarray(h)
    if h.ndim != 3:
        raise ValueError("h must be [N, H, D]")
    n, H, D = h.shape
    if len(row_ptr) != n + 1:
        raise ValueError("row_ptr must have N + 1 entries")
    # float32 attention vectors widen exactly; float64 ones pass through
    a_src = np.ascontiguousarray(a_src, dtype=np.float64).reshape(H, D)
    a_dst = np.ascontiguousarray(a_dst, dtype=np.float64).reshape(H, D)
    return row_ptr, col, h, a_src, a_dst, n, H, D, dtype


def _check(rc, what):
    if rc != 0:
        raise ValueError(f"oracle {what} rejected its inputs (code {rc})")


def _sel(sel):
    return None if sel is None else np.ascontiguousarray(sel, dtype=np.int64)


_default = Oracle()
att_grads = _default.att_grads
num_threads = _default.num_threads
set_threads = _default.set_threads
forward = _default.forward
node_stats = _default.node_stats
backward = _default.backward
backward_rows = _default.backward_rows
spmm_forward = _default.spmm_forward
spmm_backward = _default.spmm_backward
spmm_backward_rows = _default.spmm_backward_rows
reduce_forward = _default.reduce_forward
reduce_backward = _default.reduce_backward
reduce_backward_rows = _default.reduce_backward_rows
gatv2_forward = _default.gatv2_forward
gatv2_delta = _default.gatv2_delta
gatv2_backward = _default.gatv2_backward
gt_forward = _default.gt_forward
gt_backward = _default.gt_backward
