"""Every compute call is capture-safe: a CUDA graph of one forward + backward
step of each aggregation family replays to the bits of the eager calls (the
max/min backward's float atomics aside; its ordered variant is bitwise)."""
import pytest
import torch

import workload
from workload import testgraphs
from gpu_util import device_graph, to_device

pytestmark = pytest.mark.gpu


def step(gnn, g, n, H, D, A, B, C, G, T, Ta, Tb):
    r = {}
    r["gat_out"], lse = gnn.gat_forward(g, A, Ta, Tb, 0.2)
    r["gat_dh"], r["gat_das"], r["gat_dad"] = gnn.gat_backward(g, A, Ta, Tb, 0.2, lse, G)
    r["v2_out"], lse2 = gnn.gatv2_forward(g, A, B, T, 0.2)
    r["v2_dxl"], r["v2_dxr"], r["v2_datt"] = gnn.gatv2_backward(g, A, B, T, 0.2, lse2, G)
    r["gt_out"], lse3 = gnn.transformer_forward(g, A, B, C)
    r["gt_dq"], r["gt_dk"], r["gt_dv"] = gnn.transformer_backward(g, A, B, C, lse3, G)
    X, Y = A.view(n, H * D), G.view(n, H * D)
    r["gcn_out"] = gnn.gcn_forward(g, X, "sym")
    r["gcn_dx"] = gnn.gcn_backward(g, Y, "sym")
    r["max_out"], r["max_arg"] = gnn.reduce_forward(g, X, "max")
    r["max_dx"] = gnn.reduce_backward(g, r["max_arg"], Y)
    r["max_dx_ordered"] = gnn.reduce_backward(g, r["max_arg"], Y, ordered=True)
    return r


def test_cuda_graph_replay_matches_eager():
    import graph_neural_network_gb300 as gnn
    rp, ci = testgraphs.with_in_degrees([0, 3, 70, 300, 5000], n_nodes=2000, seed=3)
    g = device_graph(dict(row_ptr=rp, col=ci), (8, 64, 16))
    n, H, D = len(rp) - 1, 2, 16
    A, B, C, G = (to_device(workload.normal_f32(7, s, (n, H, D), 1.0), "f32") for s in range(1, 5))
    T, Ta, Tb = (torch.from_numpy(workload.normal_f32(7, s, (H, D), 0.1)).cuda()
                 for s in range(5, 8))
    args = (gnn, g, n, H, D, A, B, C, G, T, Ta, Tb)
    eager = step(*args)
    torch.cuda.synchronize()
    side = torch.cuda.Stream()
    side.wait_stream(torch.cuda.current_stream())
    with torch.cuda.stream(side):  # a warm-up on a side stream before capture
        step(*args)
    torch.cuda.current_stream().wait_stream(side)
    torch.cuda.synchronize()
    cg = torch.cuda.CUDAGraph()
    with torch.cuda.graph(cg):
        static = step(*args)
    for _ in range(2):
        cg.replay()
    torch.cuda.synchronize()
    assert gnn.check_device_error(g) == 0
    for k in eager:
        if k == "max_dx":  # float atomics: the order of additions may differ
            torch.testing.assert_close(static[k], eager[k], rtol=1e-4, atol=1e-5)
            continue
        assert torch.equal(static[k], eager[k]), k
