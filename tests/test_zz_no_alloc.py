"""The forward entry point that allocates nothing (gat_agg_forward_noalloc).

It is for callers that must not allocate device memory; it keeps its hub
partials in a fixed array inside the library.  Checked through the C-ABI
against gat_agg_forward on the same inputs, on two calls in a row (the second
with new features, so a stale partial left by the first call would show), and
for its size limit.  This file is collected last on purpose: a failure here
comes after every other test has run.
"""
import ctypes

import pytest
import torch

from workload import testgraphs
from gpu_util import assert_close, device_graph, make_case, to_device, to_f64

pytestmark = pytest.mark.gpu


def _noalloc(lib, g, case, h, a_s, a_d, out, lse):
    P = ctypes.c_void_p
    code = 0 if case["dtype"] == "f32" else 1
    return lib.gat_agg_forward_noalloc(g.handle, case["H"], case["D"], code, P(h.data_ptr()),
                                       P(a_s.data_ptr()), P(a_d.data_ptr()), case["slope"],
                                       P(out.data_ptr()), P(lse.data_ptr()),
                                       P(torch.cuda.current_stream().cuda_stream))


@pytest.mark.parametrize("dtype", ["f32", "bf16"])
def test_noalloc_forward_matches_forward_twice(dtype):
    import graph_neural_network_gb300 as gnn
    from graph_neural_network_gb300 import _native
    lib = _native.load()
    rp, ci = testgraphs.with_in_degrees([0, 1, 9, 65, 300, 2049], n_nodes=1500, seed=61)
    graph = None
    for call, seed in enumerate((71, 72)):
        case = make_case(rp, ci, 4, 32 if dtype == "f32" else 64, dtype, seed)
        if graph is None:
            graph = device_graph(case, (8, 64, 16))     # hubs: the partials are used
            assert graph.stats()["csr"]["hub_chunks"] > 0
        h = to_device(case["h"], dtype)
        a_s = torch.from_numpy(case["a_src"]).cuda()
        a_d = torch.from_numpy(case["a_dst"]).cuda()
        ref_out, ref_lse = gnn.gat_forward(graph, h, a_s, a_d, case["slope"])
        out = torch.full_like(ref_out, float("nan"))
        lse = torch.full_like(ref_lse, float("nan"))
        rc = _noalloc(lib, graph, case, h, a_s, a_d, out, lse)
        assert rc == 0, _native.status_string(rc)
        torch.cuda.synchronize()
        gnn.check_device_error(graph)
        assert_close(to_f64(out), to_f64(ref_out), dtype, None, f"call {call} out")
        assert_close(to_f64(lse), to_f64(ref_lse), dtype, None, f"call {call} lse")


def test_noalloc_rejects_graphs_beyond_its_array():
    from graph_neural_network_gb300 import _native
    lib = _native.load()
    cap = lib.gat_agg_forward_noalloc_capacity()
    rp, ci = testgraphs.ring(12000)
    case = make_case(rp, ci, 8, 64, "f32", 81)
    g = device_graph(case, (0, 0, 1))                   # every node is a one-chunk hub
    assert g.stats()["csr"]["hub_chunks"] * 8 * 66 * 4 > cap
    h = to_device(case["h"], "f32")
    a = torch.zeros(8, 64, device="cuda")
    out = torch.empty_like(h)
    lse = torch.empty(g.n, 8, device="cuda")
    assert _noalloc(lib, g, case, h, a, a, out, lse) == _native.ERR_WORKSPACE_TOO_SMALL
