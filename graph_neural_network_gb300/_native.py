"""ctypes binding of ``libgnnagg.so`` (declared in ``include/gnnagg.h``).

Argument marshalling only: every step of the computation runs in the
library's CUDA kernels.  torch provides device memory and streams.  There is
no CPU fallback: when the library is missing or fails to load, every entry
point raises.
"""
from __future__ import annotations

import ctypes
import os
import threading

HERE = os.path.dirname(os.path.abspath(__file__))
LIB_PATH = os.path.join(HERE, "libgnnagg.so")

# status codes (gnn_status)
OK, ERR_INVALID_ARG, ERR_UNSUPPORTED, ERR_INVALID_GRAPH = 0, 1, 2, 3
ERR_WORKSPACE_TOO_SMALL, ERR_CUDA, ERR_DEVICE_ASSERT, ERR_TIMEOUT = 4, 5, 6, 7
F32, BF16 = 0, 1
NORMS = {"sum": 0, "mean": 1, "sym": 2}  # gnn_norm
REDUCE_OPS = {"max": 0, "min": 1}        # gnn_reduce_op

# (name, restype, argtypes) of every exported symbol, in header order
_P, _I64, _I32, _SZ, _F = (ctypes.c_void_p, ctypes.c_int64, ctypes.c_int32, ctypes.c_size_t,
                           ctypes.c_float)
SIGNATURES = [
    ("gnn_default_tiling", None, [_P]),
    ("gnn_graph_buffer_bytes", _SZ, [_I64, _I64, _P]),
    ("gnn_graph_scratch_bytes", _SZ, [_I64, _I64]),
    ("gnn_graph_prepare", _I32, [_I64, _I64, _P, _P, _P, _SZ, _P, _SZ, _P, _P, _P]),
    ("gnn_graph_destroy", _I32, [_P]),
    ("gnn_graph_stats", _I32, [_P, _P, _I32]),
    ("gnn_graph_arrays", _I32, [_P, _P, _I32]),
    ("gat_agg_workspace_bytes", _SZ, [_P, _I32, _I32, _I32]),
    ("gat_agg_forward", _I32, [_P, _I32, _I32, _I32, _P, _P, _P, _F, _P, _P, _P, _SZ, _P]),
    ("gat_agg_backward", _I32, [_P, _I32, _I32, _I32, _P, _P, _P, _F, _P, _P, _P, _P, _P, _P,
                                _SZ, _P]),
    ("gat_agg_forward_timed", _I32, [_P, _I32, _I32, _I32, _P, _P, _P, _F, _P, _P, _P, _SZ, _P,
                                     _P, _I32]),
    ("gat_agg_backward_timed", _I32, [_P, _I32, _I32, _I32, _P, _P, _P, _F, _P, _P, _P, _P, _P,
                                      _P, _SZ, _P, _P, _I32]),
    ("gat_agg_backward_reuse", _I32, [_P, _I32, _I32, _I32, _P, _P, _P, _F, _P, _P, _P, _P, _P,
                                      _P, _SZ, _P, _P, _I32]),
    ("gat_agg_forward_noalloc", _I32, [_P, _I32, _I32, _I32, _P, _P, _P, _F, _P, _P, _P]),
    ("gat_agg_forward_noalloc_capacity", _SZ, []),
    ("gcn_agg_workspace_bytes", _SZ, [_P, _I32, _I32]),
    ("gcn_agg_forward", _I32, [_P, _I32, _I32, _I32, _P, _P, _P, _SZ, _P]),
    ("gcn_agg_backward", _I32, [_P, _I32, _I32, _I32, _P, _P, _P, _SZ, _P]),
    ("gatv2_agg_workspace_bytes", _SZ, [_P, _I32, _I32, _I32]),
    ("gatv2_agg_forward", _I32, [_P, _I32, _I32, _I32, _P, _P, _P, _F, _P, _P, _P, _SZ, _P]),
    ("gatv2_agg_backward", _I32, [_P, _I32, _I32, _I32, _P, _P, _P, _F, _P, _P, _P, _P, _P,
                                  _P, _SZ, _P]),
    ("transformer_agg_workspace_bytes", _SZ, [_P, _I32, _I32, _I32]),
    ("transformer_agg_forward", _I32, [_P, _I32, _I32, _I32, _P, _P, _P, _F, _P, _P, _P, _SZ,
                                       _P]),
    ("transformer_agg_backward", _I32, [_P, _I32, _I32, _I32, _P, _P, _P, _F, _P, _P, _P, _P,
                                        _P, _P, _SZ, _P]),
    ("reduce_agg_workspace_bytes", _SZ, [_P, _I32, _I32]),
    ("reduce_agg_forward", _I32, [_P, _I32, _I32, _I32, _P, _P, _P, _P, _SZ, _P]),
    ("reduce_agg_backward", _I32, [_P, _I32, _I32, _P, _P, _P, _P, _SZ, _P]),
    ("reduce_agg_backward_ordered", _I32, [_P, _I32, _I32, _P, _P, _P, _P, _SZ, _P]),
    ("gnn_wait_selftest", _I32, [_P, _I32, _P]),
    ("gnn_check_device_error", _I32, [_P, _P, _P]),
    ("gnn_status_string", ctypes.c_char_p, [_I32]),
    ("gnn_abi_version", _I32, []),
]


class Tiling(ctypes.Structure):
    _fields_ = [("light_max_deg", ctypes.c_int32), ("cta_max_deg", ctypes.c_int32),
                ("hub_chunk", ctypes.c_int32)]


class GnnError(RuntimeError):
    def __init__(self, status: int, what: str):
        self.status = status
        super().__init__(f"{what}: {status_string(status)} (status {status})")


_lock = threading.Lock()
_lib = None


def load(path: str = LIB_PATH) -> ctypes.CDLL:
    """Load the library (once).  Raises when it is missing: build it with
    ``graph_neural_network_gb300.build.build()``."""
    global _lib
    with _lock:
        if _lib is not None:
            return _lib
        if not os.path.exists(path):
            raise RuntimeError(f"{path} is missing: the CUDA extension must be built "
                               "(graph_neural_network_gb300.build.build()); there is no "
                               "fallback implementation")
        lib = ctypes.CDLL(path)
        for name, res, args in SIGNATURES:
            fn = getattr(lib, name)
            fn.restype = res
            fn.argtypes = args
        _lib = lib
        return lib


def status_string(status: int) -> str:
    try:
        return load().gnn_status_string(status).decode()
    except Exception:
        return "unknown"


def check(status: int, what: str):
    if status != OK:
        raise GnnError(status, what)


def default_tiling() -> Tiling:
    t = Tiling()
    load().gnn_default_tiling(ctypes.byref(t))
    return t
