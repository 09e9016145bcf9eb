"""Full-size workloads, in the launch configuration bench.py times (default
tiling, one workspace shared by the forward and the backward): the GAT
forward on every row, the GAT backward on every row of the two smaller graphs
and on sampled rows (with the largest CSC hubs) of the others, the
attention-vector gradients over the whole graph, and sampled rows of the
other aggregation families."""
import numpy as np
import pytest
import torch

import oracle
import workload
import gpu_util
from gpu_util import assert_close, run_gpu, to_f64

pytestmark = [pytest.mark.gpu, pytest.mark.slow]


def _rows(t, sel):
    return to_f64(t[torch.from_numpy(np.asarray(sel, np.int64)).to(t.device)])


def _backward_cost(rp, ci):
    """Edge visits the per-node oracle makes for dh_j: sum of the in-degrees
    of j's out-neighbours."""
    indeg = np.diff(rp).astype(np.float64)
    dst = np.repeat(np.arange(len(rp) - 1), np.diff(rp))
    return np.bincount(ci, weights=indeg[dst], minlength=len(rp) - 1)


CHUNK = 1 << 18   # nodes per oracle call when every row is compared


def _gat_bench_launch(case, w):
    """Forward and backward in the launch configuration bench.py times:
    default tiling, one workspace for both calls, so that the backward takes
    the per-node scores the forward left there."""
    import graph_neural_network_gb300 as gnn
    g = gpu_util.device_graph(case)
    h = gpu_util.to_device(case["h"], w.dtype)
    dout = gpu_util.to_device(case["dout"], w.dtype)
    a_s = torch.from_numpy(case["a_src"]).cuda()
    a_d = torch.from_numpy(case["a_dst"]).cuda()
    ws = g.workspace(w.H, w.D, h.dtype)
    out, lse = gnn.gat_forward(g, h, a_s, a_d, w.slope, ws=ws)
    dh, da_s, da_d = gnn.gat_backward(g, h, a_s, a_d, w.slope, lse, dout, ws=ws,
                                      reuse_scores=True)
    torch.cuda.synchronize()
    gnn.check_device_error(g)
    return dict(graph=g, out_t=out, lse_t=lse, dh_t=dh, da_src_t=da_s, da_dst_t=da_d)


@pytest.mark.parametrize("idx", [2, 3, 4, 5, 6])
def test_full_size_parity(idx):
    """Every row of out and lse against the oracle (strict bound; lse to the
    float32 tolerance); dh on every row for the two smaller graphs, else on
    2,000 random rows, the 24 largest out-degrees (CSC hubs of many chunks)
    and the ragged tail; da_src and da_dst over the whole graph.  The
    gradients accept either LeakyReLU derivative at edges within float32
    rounding of the kink (the oracle's kink term)."""
    w = workload.CONFIGS[idx]
    rp, ci = workload.make_graph(w)
    n = len(rp) - 1
    h, a_s, a_d, dout = workload.make_features(w, n)
    case = dict(row_ptr=rp, col=ci, h=h, dout=dout, a_src=a_s, a_dst=a_d, H=w.H, D=w.D,
                dtype=w.dtype, slope=w.slope)
    gpu = _gat_bench_launch(case, w)
    # forward: every row, in chunks of nodes
    for c0 in range(0, n, CHUNK):
        sel = np.arange(c0, min(n, c0 + CHUNK))
        f = oracle.forward(rp, ci, h, a_s, a_d, w.slope, sel=sel, with_mag=True)
        assert_close(_rows(gpu["out_t"], sel), f["out"], w.dtype, f["out_mag"], f"cfg{idx} out",
                     strict=True)
        assert_close(_rows(gpu["lse_t"], sel), f["lse"], "f32", None, f"cfg{idx} lse",
                     strict=True)
        del f
    rng = np.random.default_rng(1000 + idx)
    outdeg = np.bincount(ci, minlength=n)
    top = np.argsort(outdeg)[::-1][:24]
    if idx in (2, 3):
        b = oracle.backward(rp, ci, h, a_s, a_d, w.slope, dout, with_mag=True, with_kink=True)
        for c0 in range(0, n, CHUNK):
            sel = np.arange(c0, min(n, c0 + CHUNK))
            assert_close(_rows(gpu["dh_t"], sel), b["dh"][sel], w.dtype, b["dh_mag"][sel],
                         f"cfg{idx} dh", kink=b["dh_kink"][sel])
        da = {k: b[k] for k in ("da_src", "da_dst", "da_src_mag", "da_dst_mag", "da_src_kink",
                                "da_dst_kink")}
        del b
    else:
        sel_b = np.unique(np.concatenate([rng.choice(n, 2000, replace=False), top,
                                          np.arange(n - 9, n)]))
        b = oracle.backward_rows(rp, ci, h, a_s, a_d, w.slope, dout, sel_b, with_mag=True,
                                 with_kink=True)
        assert_close(_rows(gpu["dh_t"], sel_b), b["dh"], w.dtype, b["dh_mag"], f"cfg{idx} dh",
                     kink=b["dh_kink"])
        da = oracle.att_grads(rp, ci, h, a_s, a_d, w.slope, dout, with_mag=True, with_kink=True)
    assert_close(to_f64(gpu["da_src_t"]), da["da_src"], w.dtype, da["da_src_mag"],
                 f"cfg{idx} da_src", kink=da["da_src_kink"])
    assert_close(to_f64(gpu["da_dst_t"]), da["da_dst"], w.dtype, da["da_dst_mag"],
                 f"cfg{idx} da_dst", kink=da["da_dst_kink"])
    assert outdeg[top].max() > 4096 or idx == 2      # the CSC hub path was compared
    # SpMM-family propagation (symmetric normalisation) and the max reduction
    # on the same graph: sampled rows
    import graph_neural_network_gb300 as gnn
    g = gpu["graph"]
    del gpu
    F = w.H * w.D
    indeg = np.diff(rp)
    cost = _backward_cost(rp, ci)
    sel_f = np.unique(np.concatenate([rng.choice(n, 3000, replace=False),
                                      np.argsort(indeg)[-64:], np.arange(n - 17, n)]))
    cheap = np.nonzero(cost < 2e5)[0]
    sel_s = np.unique(np.concatenate([rng.choice(cheap, min(400, len(cheap)), replace=False),
                                      np.asarray([j for j in top if cost[j] < 3e7], np.int64)]))
    x = gpu_util.to_device(h.reshape(n, F), w.dtype)
    dy = gpu_util.to_device(dout.reshape(n, F), w.dtype)
    out = gnn.gcn_forward(g, x, "sym")
    dx = gnn.gcn_backward(g, dy, "sym")
    torch.cuda.synchronize()
    sf = oracle.spmm_forward(rp, ci, h.reshape(n, F), "sym", sel=sel_f, with_mag=True)
    assert_close(_rows(out, sel_f), sf["out"], w.dtype, sf["out_mag"], f"cfg{idx} gcn out")
    sb = oracle.spmm_backward_rows(rp, ci, dout.reshape(n, F), "sym", sel_s, with_mag=True)
    assert_close(_rows(dx, sel_s), sb["dx"], w.dtype, sb["dx_mag"], f"cfg{idx} gcn dx")
    # max reduction: sampled rows bit for bit, sampled gradient rows
    rout, rarg = gnn.reduce_forward(g, x, "max")
    rdx = gnn.reduce_backward(g, rarg, dy)
    torch.cuda.synchronize()
    rf = oracle.reduce_forward(rp, ci, h.reshape(n, F), "max", sel=sel_f)
    sel_t = torch.from_numpy(np.asarray(sel_f, np.int64)).to(rarg.device)
    assert np.array_equal(rarg[sel_t].cpu().numpy(), rf["arg"]), f"cfg{idx} max arg"
    assert np.array_equal(_rows(rout, sel_f), rf["out"]), f"cfg{idx} max out"
    cheap_r = sel_s[cost[sel_s] < 2e4][:150]     # the oracle recomputes every row they win
    rb = oracle.reduce_backward_rows(rp, ci, h.reshape(n, F), "max", dout.reshape(n, F), cheap_r,
                                     with_mag=True)
    assert_close(_rows(rdx, cheap_r), rb["dx"], w.dtype, rb["dx_mag"], f"cfg{idx} max dx")


@pytest.mark.parametrize("idx", [2, 3])
def test_full_size_sampled_parity_gatv2_and_transformer(idx):
    """GATv2 and graph-transformer attention on the full uniform and 1M-node
    Chung-Lu workloads, default tiling: sampled rows of every output against
    the oracle (GATv2's datt over the whole graph)."""
    import graph_neural_network_gb300 as gnn
    w = workload.CONFIGS[idx]
    rp, ci = workload.make_graph(w)
    n = len(rp) - 1
    h, a_s, _, dout = workload.make_features(w, n)
    extra = []
    for stream in (5, 6):
        x = workload.normal_f32(w.seed, stream, (n, w.H, w.D), 1.0)
        extra.append(workload.f32_to_bf16_bits(x) if w.dtype == "bf16" else x)
    xr, val = extra
    g = gpu_util.device_graph(dict(row_ptr=rp, col=ci))
    dev = [gpu_util.to_device(x, w.dtype) for x in (h, xr, val, dout)]
    A = torch.from_numpy(a_s).cuda()
    rng = np.random.default_rng(2000 + idx)
    indeg = np.diff(rp)
    sel_f = np.unique(np.concatenate([rng.choice(n, 2000, replace=False), np.argsort(indeg)[-32:],
                                      np.arange(n - 9, n)]))
    cost = _backward_cost(rp, ci)
    cheap = np.nonzero(cost < 1e5)[0]
    outdeg = np.bincount(ci, minlength=n)
    top = [j for j in np.argsort(outdeg)[::-1][:200] if cost[j] < 5e6][:8]
    sel_b = np.unique(np.concatenate([rng.choice(cheap, min(200, len(cheap)), replace=False),
                                      np.asarray(top, np.int64)]))
    # GATv2: xl = h, xr, att = a_src
    out, lse = gnn.gatv2_forward(g, dev[0], dev[1], A, w.slope)
    dxl, dxr, datt = gnn.gatv2_backward(g, dev[0], dev[1], A, w.slope, lse, dev[3])
    torch.cuda.synchronize()
    f = oracle.gatv2_forward(rp, ci, h, xr, a_s, w.slope, sel=sel_f, with_mag=True)
    assert_close(_rows(out, sel_f), f["out"], w.dtype, f["out_mag"], f"cfg{idx} gatv2 out")
    assert_close(_rows(lse, sel_f), f["lse"], "f32", None, f"cfg{idx} gatv2 lse")
    b = oracle.gatv2_backward(rp, ci, h, xr, a_s, w.slope, dout, sel=sel_b, with_mag=True)
    assert_close(_rows(dxl, sel_b), b["dxl"], w.dtype, b["dxl_mag"], f"cfg{idx} gatv2 dxl")
    assert_close(_rows(dxr, sel_b), b["dxr"], w.dtype, b["dxr_mag"], f"cfg{idx} gatv2 dxr")
    assert_close(to_f64(datt), b["datt"], w.dtype, b["datt_mag"], f"cfg{idx} gatv2 datt")
    # graph transformer: q = h, key = xr, val
    out, lse = gnn.transformer_forward(g, dev[0], dev[1], dev[2])
    dq, dk, dv = gnn.transformer_backward(g, dev[0], dev[1], dev[2], lse, dev[3])
    torch.cuda.synchronize()
    sc = w.D ** -0.5
    f = oracle.gt_forward(rp, ci, h, xr, val, sc, sel=sel_f, with_mag=True)
    assert_close(_rows(out, sel_f), f["out"], w.dtype, f["out_mag"], f"cfg{idx} gt out")
    assert_close(_rows(lse, sel_f), f["lse"], "f32", None, f"cfg{idx} gt lse")
    b = oracle.gt_backward(rp, ci, h, xr, val, sc, dout, sel=sel_b, with_mag=True)
    for name, got in (("dq", dq), ("dkey", dk), ("dval", dv)):
        assert_close(_rows(got, sel_b), b[name], w.dtype, b[name + "_mag"], f"cfg{idx} gt {name}")
    assert outdeg[top].max() > 2048 or idx == 2       # a CSC hub was sampled
