"""Seeded synthetic inputs for the fused GAT aggregation: graphs and features.

This module is shared by the CUDA path's tests and bench and by the CPU oracle's
tests.  It draws inputs only; it contains none of the aggregation arithmetic.
The generators live in ``gen.cpp`` (threaded C++, counter-based random
numbers, so results do not depend on the thread count) and are loaded through
ctypes.

Graph convention (CSR, destination-major): ``row_ptr[N+1]``, ``col_idx[E]``,
both int32; row ``i`` lists the sources ``j`` of the edges ``j -> i``, sorted,
duplicates removed, one self-loop per node.
"""
from __future__ import annotations

import ctypes
import os
import subprocess
import threading

import numpy as np

_HERE = os.path.dirname(os.path.abspath(__file__))
_SRC = os.path.join(_HERE, "gen.cpp")
_LIB = os.path.join(_HERE, "libgnnwork.so")
_lock = threading.Lock()
_lib = None


def build(force: bool = False) -> str:
    """Compile ``libgnnwork.so`` next to this file (skipped when up to date)."""
    if (not force and os.path.exists(_LIB)
            and os.path.getmtime(_LIB) >= os.path.getmtime(_SRC)):
        return _LIB
    tmp = _LIB + f".tmp{os.getpid()}"
    subprocess.check_call(["g++", "-O2", "-std=c++17", "-fPIC", "-shared", "-pthread",
                           _SRC, "-o", tmp])
    os.replace(tmp, _LIB)
    return _LIB


def _load():
    global _lib
    with _lock:
        if _lib is not None:
            return _lib
        build()
        lib = ctypes.CDLL(_LIB)
        P = ctypes.c_void_p
        i64, u64, f64, i32 = ctypes.c_int64, ctypes.c_uint64, ctypes.c_double, ctypes.c_int
        lib.gen_normal_f32.argtypes = [u64, u64, i64, f64, P]
        lib.gen_f32_to_bf16.argtypes = [i64, P, P]
        lib.gen_graph_nodes.argtypes = [P]
        lib.gen_graph_nodes.restype = i64
        lib.gen_graph_edges.argtypes = [P]
        lib.gen_graph_edges.restype = i64
        lib.gen_graph_copy.argtypes = [P, P, P]
        lib.gen_graph_free.argtypes = [P]
        lib.gen_graph_from_csr.argtypes = [i64, P, P]
        lib.gen_graph_from_csr.restype = P
        lib.gen_graph_er.argtypes = [i64, f64, u64]
        lib.gen_graph_er.restype = P
        lib.gen_graph_uniform.argtypes = [i64, i64, u64]
        lib.gen_graph_uniform.restype = P
        lib.gen_graph_chung_lu.argtypes = [i64, f64, f64, f64, u64]
        lib.gen_graph_chung_lu.restype = P
        lib.gen_graph_rmat.argtypes = [i32, i64, f64, f64, f64, u64]
        lib.gen_graph_rmat.restype = P
        lib.gen_graph_permute_random.argtypes = [P, u64]
        lib.gen_graph_permute_random.restype = P
        lib.gen_rcm_order.argtypes = [P, P]
        lib.gen_graph_relabel.argtypes = [P, P]
        lib.gen_graph_relabel.restype = P
        _lib = lib
        return lib


def _ptr(a: np.ndarray):
    return ctypes.c_void_p(a.ctypes.data)


def _take(handle) -> tuple[np.ndarray, np.ndarray]:
    lib = _load()
    if not handle:
        raise ValueError("graph generator rejected its arguments")
    try:
        n = lib.gen_graph_nodes(handle)
        e = lib.gen_graph_edges(handle)
        row_ptr = np.empty(n + 1, dtype=np.int32)
        col = np.empty(e, dtype=np.int32)
        lib.gen_graph_copy(handle, _ptr(row_ptr), _ptr(col))
        return row_ptr, col
    finally:
        lib.gen_graph_free(handle)


def _wrap(row_ptr: np.ndarray, col: np.ndarray):
    row_ptr = np.ascontiguousarray(row_ptr, dtype=np.int32)
    col = np.ascontiguousarray(col, dtype=np.int32)
    return _load().gen_graph_from_csr(len(row_ptr) - 1, _ptr(row_ptr), _ptr(col))


# ---- graphs ------------------------------------------------------------------

def erdos_renyi(n: int, avg_deg: float, seed: int):
    return _take(_load().gen_graph_er(n, float(avg_deg), seed))


def uniform(n: int, k: int, seed: int):
    return _take(_load().gen_graph_uniform(n, k, seed))


def chung_lu(n: int, gamma: float, avg_deg: float, cap: float, seed: int):
    return _take(_load().gen_graph_chung_lu(n, float(gamma), float(avg_deg), float(cap), seed))


def rmat(scale: int, edge_factor: int, a: float, b: float, c: float, seed: int):
    return _take(_load().gen_graph_rmat(scale, edge_factor, a, b, c, seed))


def permute_random(row_ptr, col, seed: int):
    lib = _load()
    h = _wrap(row_ptr, col)
    try:
        return _take(lib.gen_graph_permute_random(h, seed))
    finally:
        lib.gen_graph_free(h)


def rcm_order(row_ptr, col) -> np.ndarray:
    """new_id[v] for reverse Cuthill-McKee on the symmetrised graph."""
    lib = _load()
    h = _wrap(row_ptr, col)
    try:
        new_id = np.empty(len(row_ptr) - 1, dtype=np.int32)
        lib.gen_rcm_order(h, _ptr(new_id))
        return new_id
    finally:
        lib.gen_graph_free(h)


def hubs_then_rcm_order(row_ptr, col, min_degree: int) -> np.ndarray:
    """new_id[v]: the nodes of in- plus out-degree above min_degree first, by
    descending degree (ties by id), then every other node in reverse
    Cuthill-McKee order.  The alternative reading of "degree-sorted + RCM"."""
    n = len(row_ptr) - 1
    deg = np.diff(np.asarray(row_ptr, np.int64)) + np.bincount(np.asarray(col), minlength=n)
    rcm = rcm_order(row_ptr, col)
    hubs = np.flatnonzero(deg > min_degree)
    hubs = hubs[np.lexsort((hubs, -deg[hubs]))]
    rest = np.flatnonzero(deg <= min_degree)
    rest = rest[np.argsort(rcm[rest], kind="stable")]
    order = np.concatenate([hubs, rest])  # order[k]: the node that gets id k
    new_id = np.empty(n, dtype=np.int32)
    new_id[order] = np.arange(n, dtype=np.int32)
    return new_id


def relabel(row_ptr, col, new_id):
    lib = _load()
    h = _wrap(row_ptr, col)
    new_id = np.ascontiguousarray(new_id, dtype=np.int32)
    try:
        return _take(lib.gen_graph_relabel(h, _ptr(new_id)))
    finally:
        lib.gen_graph_free(h)


# ---- features ----------------------------------------------------------------

def normal_f32(seed: int, stream: int, shape, std: float = 1.0) -> np.ndarray:
    out = np.empty(shape, dtype=np.float32)
    _load().gen_normal_f32(seed, stream, out.size, float(std), _ptr(out))
    return out


def f32_to_bf16_bits(x: np.ndarray) -> np.ndarray:
    """Round to bfloat16 (nearest, ties to even); returns the uint16 bit patterns."""
    x = np.ascontiguousarray(x, dtype=np.float32)
    out = np.empty(x.shape, dtype=np.uint16)
    _load().gen_f32_to_bf16(x.size, _ptr(x), _ptr(out))
    return out


def bf16_bits_to_f32(b: np.ndarray) -> np.ndarray:
    """Exact widening of bfloat16 bit patterns to float32."""
    return (np.ascontiguousarray(b, dtype=np.uint16).astype(np.uint32) << 16).view(np.float32)


from .configs import CONFIGS, Workload, make_graph, make_features  # noqa: E402,F401
