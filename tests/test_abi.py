"""The C-ABI library: it builds, loads, exports every symbol the header
declares, and rejects bad arguments before touching the GPU (CPU only)."""
import ctypes
import os
import re

import pytest

ROOT = os.path.dirname(os.path.dirname(os.path.abspath(__file__)))
HEADER = os.path.join(ROOT, "include", "gnnagg.h")


@pytest.fixture(scope="module")
def lib():
    from graph_neural_network_gb300 import build, _native
    build.build()
    return _native.load()


def declared_functions():
    text = open(HEADER).read()
    text = re.sub(r"/\*.*?\*/", "", text, flags=re.S)
    return sorted(set(re.findall(r"\b((?:gnn|gat|gatv2|gcn|reduce|transformer)_[a-z0-9_]+)\s*\(", text)))


def test_header_declares_the_boundary():
    names = declared_functions()
    for required in ("gnn_graph_prepare", "gat_agg_forward", "gat_agg_backward"):
        assert required in names


def test_library_exports_every_declared_symbol(lib):
    missing = [n for n in declared_functions() if not hasattr(lib, n)]
    assert not missing, missing


def test_binding_covers_the_header():
    from graph_neural_network_gb300 import _native
    bound = {name for name, _, _ in _native.SIGNATURES}
    assert bound == set(declared_functions())


def test_version_and_status_strings(lib):
    assert lib.gnn_abi_version() == 1
    for code in range(8):
        assert lib.gnn_status_string(code)
    assert b"unknown" in lib.gnn_status_string(99)


def test_sizes_are_host_only(lib):
    from graph_neural_network_gb300 import _native
    t = _native.default_tiling()
    assert (t.light_max_deg, t.cta_max_deg, t.hub_chunk) == (-1, 4096, 2048)   # automatic
    # an automatic light threshold is bounded by the buffer of its floor, 64
    for n, e in ((1000, 20000), (50_000, 3_000_000)):
        floor = _native.Tiling(64, 4096, 2048)
        assert lib.gnn_graph_buffer_bytes(n, e, None) == \
            lib.gnn_graph_buffer_bytes(n, e, ctypes.byref(floor))
        auto_low = _native.Tiling(-1, 16, 8)              # floor above cta_max_deg: 16
        low = _native.Tiling(16, 16, 8)
        assert lib.gnn_graph_buffer_bytes(n, e, ctypes.byref(auto_low)) == \
            lib.gnn_graph_buffer_bytes(n, e, ctypes.byref(low))
    assert lib.gnn_graph_buffer_bytes(10, 10, ctypes.byref(_native.Tiling(-2, 64, 8))) == 0
    b1 = lib.gnn_graph_buffer_bytes(1000, 20000, None)
    b2 = lib.gnn_graph_buffer_bytes(1000, 40000, None)
    assert 0 < b1 < b2
    assert lib.gnn_graph_buffer_bytes(-1, 5, None) == 0
    bad = _native.Tiling(10, 5, 8)                      # cta_max < light_max
    assert lib.gnn_graph_buffer_bytes(10, 10, ctypes.byref(bad)) == 0
    assert lib.gnn_graph_scratch_bytes(1000, 20000) > 16 * 20000


def test_bad_arguments_rejected_without_gpu(lib):
    from graph_neural_network_gb300 import _native
    out = ctypes.c_void_p()
    P = ctypes.c_void_p
    # missing output handle, null pointers, negative sizes
    assert lib.gnn_graph_prepare(4, 4, P(16), P(16), P(256), 1 << 20, P(256), 1 << 20, None,
                                 None, None) == _native.ERR_INVALID_ARG
    assert lib.gnn_graph_prepare(-4, 4, P(16), P(16), P(256), 1 << 20, P(256), 1 << 20, None,
                                 None, ctypes.byref(out)) == _native.ERR_INVALID_ARG
    assert lib.gnn_graph_prepare(4, 4, None, P(16), P(256), 1 << 20, P(256), 1 << 20, None,
                                 None, ctypes.byref(out)) == _native.ERR_INVALID_ARG
    # misaligned col_idx and buffer
    assert lib.gnn_graph_prepare(4, 4, P(16), P(20), P(256), 1 << 20, P(256), 1 << 20, None,
                                 None, ctypes.byref(out)) == _native.ERR_INVALID_ARG
    assert lib.gnn_graph_prepare(4, 4, P(16), P(16), P(264), 1 << 20, P(256), 1 << 20, None,
                                 None, ctypes.byref(out)) == _native.ERR_INVALID_ARG
    # buffers too small
    assert lib.gnn_graph_prepare(4, 4, P(16), P(16), P(256), 16, P(256), 1 << 20, None, None,
                                 ctypes.byref(out)) == _native.ERR_WORKSPACE_TOO_SMALL
    # compute calls without a graph
    assert lib.gat_agg_forward(None, 1, 16, 0, P(16), P(16), P(16), 0.2, P(16), P(16), P(256),
                               1 << 20, None) == _native.ERR_INVALID_ARG
    assert lib.gat_agg_backward(None, 1, 16, 0, P(16), P(16), P(16), 0.2, P(16), P(16), P(16),
                                P(16), P(16), P(256), 1 << 20, None) == _native.ERR_INVALID_ARG
    assert lib.gat_agg_workspace_bytes(None, 1, 16, 0) == 0
    assert lib.gnn_graph_stats(None, None, 16) == _native.ERR_INVALID_ARG
    assert lib.gnn_check_device_error(None, None, None) == _native.ERR_INVALID_ARG
    assert lib.gnn_wait_selftest(None, 100, None) == _native.ERR_INVALID_ARG


def test_product_package_does_not_use_the_oracle():
    pkg = os.path.join(ROOT, "graph_neural_network_gb300")
    for dirpath, _, files in os.walk(pkg):
        for f in files:
            if f.endswith((".py", ".cu", ".cuh", ".h", ".cpp")):
                text = open(os.path.join(dirpath, f)).read()
                assert "oracle" not in text.lower(), f"{f} mentions the oracle"
