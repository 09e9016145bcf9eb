"""Edge cases of the GATv2, graph-transformer, GCN and max/min calls: no edges
at all, an empty graph, in-stars and out-stars (one hub each way), and a
side stream giving the same bits as the default stream."""
import numpy as np
import pytest
import torch

import oracle
import workload
from workload import testgraphs
from gpu_util import assert_close, device_graph, to_device, to_f64

pytestmark = pytest.mark.gpu


def feats(n, H, D, seed, k=4):
    return [workload.normal_f32(seed, 1 + s, (n, H, D), 1.0) for s in range(k)]


def run_all(g, rp, ci, H, D, stream=None):
    """Every op on f32 inputs; returns {name: device tensor} and the inputs."""
    import graph_neural_network_gb300 as gnn
    n = len(rp) - 1
    a, b, c, d = feats(n, H, D, 5)
    att = workload.normal_f32(5, 9, (H, D), 0.1)
    A, B, C, G = (to_device(x, "f32") for x in (a, b, c, d))
    T = torch.from_numpy(att).cuda()
    r = {}
    r["v2_out"], lse = gnn.gatv2_forward(g, A, B, T, 0.2, stream=stream)
    r["v2_dxl"], r["v2_dxr"], r["v2_datt"] = gnn.gatv2_backward(g, A, B, T, 0.2, lse, G,
                                                                stream=stream)
    r["gt_out"], lse2 = gnn.transformer_forward(g, A, B, C, stream=stream)
    r["gt_dq"], r["gt_dk"], r["gt_dv"] = gnn.transformer_backward(g, A, B, C, lse2, G,
                                                                  stream=stream)
    X, Y = A.view(n, H * D), G.view(n, H * D)
    r["gcn_out"] = gnn.gcn_forward(g, X, "mean", stream=stream)
    r["gcn_dx"] = gnn.gcn_backward(g, Y, "mean", stream=stream)
    r["max_out"], r["max_arg"] = gnn.reduce_forward(g, X, "max", stream=stream)
    r["max_dx"] = gnn.reduce_backward(g, r["max_arg"], Y, stream=stream)
    torch.cuda.synchronize()
    gnn.check_device_error(g)
    return r, (a, b, c, d, att)


def check_all(rp, ci, H=2, D=8, tiling=None):
    g = device_graph(dict(row_ptr=np.asarray(rp, np.int32), col=np.asarray(ci, np.int32)), tiling)
    r, (a, b, c, d, att) = run_all(g, rp, ci, H, D)
    n = len(rp) - 1
    fv = oracle.gatv2_forward(rp, ci, a, b, att, 0.2, with_mag=True)
    bv = oracle.gatv2_backward(rp, ci, a, b, att, 0.2, d, with_mag=True)
    assert_close(to_f64(r["v2_out"]), fv["out"], "f32", fv["out_mag"], "gatv2 out")
    for k in ("dxl", "dxr", "datt"):
        assert_close(to_f64(r["v2_" + k]), bv[k], "f32", bv[k + "_mag"], "gatv2 " + k)
    ft = oracle.gt_forward(rp, ci, a, b, c, D ** -0.5, with_mag=True)
    bt = oracle.gt_backward(rp, ci, a, b, c, D ** -0.5, d, with_mag=True)
    assert_close(to_f64(r["gt_out"]), ft["out"], "f32", ft["out_mag"], "transformer out")
    for k, key in (("dq", "dq"), ("dk", "dkey"), ("dv", "dval")):
        assert_close(to_f64(r["gt_" + k]), bt[key], "f32", bt[key + "_mag"], "transformer " + k)
    x, y = a.reshape(n, -1), d.reshape(n, -1)
    fs = oracle.spmm_forward(rp, ci, x, "mean", with_mag=True)
    bs = oracle.spmm_backward(rp, ci, y, "mean", with_mag=True)
    assert_close(to_f64(r["gcn_out"]), fs["out"], "f32", fs["out_mag"], "gcn out")
    assert_close(to_f64(r["gcn_dx"]), bs["dx"], "f32", bs["dx_mag"], "gcn dx")
    fm = oracle.reduce_forward(rp, ci, x, "max")
    bm = oracle.reduce_backward(fm["arg"], y, with_mag=True)
    assert np.array_equal(r["max_arg"].cpu().numpy(), fm["arg"])
    assert np.array_equal(to_f64(r["max_out"]), fm["out"])
    assert_close(to_f64(r["max_dx"]), bm["dx"], "f32", bm["dx_mag"], "max dx")
    return r


def test_no_edges():
    rp, ci = testgraphs.isolated(40)
    r = check_all(rp, ci)
    assert torch.all(r["max_arg"] == -1) and torch.all(r["gcn_out"] == 0)


def test_empty_graph():
    import graph_neural_network_gb300 as gnn
    rp = np.zeros(1, np.int32)
    ci = np.zeros(0, np.int32)
    g = device_graph(dict(row_ptr=rp, col=ci))
    z = torch.zeros((0, 2, 8), device="cuda")
    out, lse = gnn.gatv2_forward(g, z, z, torch.zeros((2, 8), device="cuda"))
    assert out.shape == (0, 2, 8) and lse.shape == (0, 2)
    assert gnn.gcn_forward(g, z.view(0, 16), "sym").shape == (0, 16)


@pytest.mark.parametrize("tiling", [(64, 4096, 2048), (0, 0, 1)], ids=str)
def test_stars(tiling):
    check_all(*testgraphs.star_in(3000), tiling=tiling)
    check_all(*testgraphs.star_out(3000), tiling=tiling)


def test_side_stream_matches_default_stream():
    rp, ci = testgraphs.with_in_degrees([0, 3, 70, 300, 5000], n_nodes=2000, seed=3)
    g = device_graph(dict(row_ptr=rp, col=ci), (8, 64, 16))
    a, _ = run_all(g, rp, ci, 2, 16)
    s = torch.cuda.Stream()
    with torch.cuda.stream(s):
        b, _ = run_all(g, rp, ci, 2, 16, stream=s)
    for k in a:
        if k == "max_dx":   # float atomics: the order of additions may differ
            continue
        assert torch.equal(a[k], b[k]), k
