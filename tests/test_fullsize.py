"""Full-size workloads, in the launch configuration bench.py times (default
tiling): sampled outputs against the oracle computed node by node, and the
attention-vector gradients against the oracle's row-parallel sum."""
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


@pytest.mark.parametrize("idx", [2, 3, 4, 5, 6])
def test_full_size_sampled_parity(idx):
    w = workload.CONFIGS[idx]
    rp, ci = workload.make_graph(w)
    n = len(rp) - 1
    h, a_s, a_d, dout = workload.make_features(w, n)
    case = dict(row_ptr=rp, col=ci, h=h, dout=dout, a_src=a_s, a_dst=a_d, H=w.H, D=w.D,
                dtype=w.dtype, slope=w.slope)
    gpu = run_gpu(case, fetch=False)
    rng = np.random.default_rng(1000 + idx)
    indeg = np.diff(rp)
    outdeg = np.bincount(ci, minlength=n)
    # forward: random nodes, the largest in-degrees (hub split + merge), ragged tail
    sel_f = np.unique(np.concatenate([rng.choice(n, 3000, replace=False),
                                      np.argsort(indeg)[-64:], np.arange(n - 17, n)]))
    f = oracle.forward(rp, ci, h, a_s, a_d, w.slope, sel=sel_f, with_mag=True)
    assert_close(_rows(gpu["out_t"], sel_f), f["out"], w.dtype, f["out_mag"], f"cfg{idx} out")
    assert_close(_rows(gpu["lse_t"], sel_f), f["lse"], w.dtype, None, f"cfg{idx} lse")
    # backward rows: random nodes plus the largest out-degrees the oracle can afford
    cost = _backward_cost(rp, ci)
    cheap = np.nonzero(cost < 2e5)[0]
    top = [j for j in np.argsort(outdeg)[::-1][:400] if cost[j] < 3e7][:24]
    sel_b = np.unique(np.concatenate([rng.choice(cheap, min(400, len(cheap)), replace=False),
                                      np.asarray(top, np.int64)]))
    b = oracle.backward_rows(rp, ci, h, a_s, a_d, w.slope, dout, sel_b, with_mag=True)
    assert_close(_rows(gpu["dh_t"], sel_b), b["dh"], w.dtype, b["dh_mag"], f"cfg{idx} dh")
    ag = oracle.att_grads(rp, ci, h, a_s, a_d, w.slope, dout, with_mag=True)
    assert_close(to_f64(gpu["da_src_t"]), ag["da_src"], w.dtype, ag["da_src_mag"], "da_src")
    assert_close(to_f64(gpu["da_dst_t"]), ag["da_dst"], w.dtype, ag["da_dst_mag"], "da_dst")
    assert outdeg[top].max() > 4096 or idx == 2      # the CSC hub path was sampled
    # SpMM-family propagation (symmetric normalisation) on the same graph and rows
    import graph_neural_network_gb300 as gnn
    g = gpu["graph"]
    F = w.H * w.D
    x = gpu_util.to_device(h.reshape(n, F), w.dtype)
    dy = gpu_util.to_device(dout.reshape(n, F), w.dtype)
    out = gnn.gcn_forward(g, x, "sym")
    dx = gnn.gcn_backward(g, dy, "sym")
    torch.cuda.synchronize()
    sf = oracle.spmm_forward(rp, ci, h.reshape(n, F), "sym", sel=sel_f, with_mag=True)
    assert_close(_rows(out, sel_f), sf["out"], w.dtype, sf["out_mag"], f"cfg{idx} gcn out")
    sb = oracle.spmm_backward_rows(rp, ci, dout.reshape(n, F), "sym", sel_b, with_mag=True)
    assert_close(_rows(dx, sel_b), sb["dx"], w.dtype, sb["dx_mag"], f"cfg{idx} gcn dx")
    # max reduction: sampled rows bit for bit, sampled gradient rows
    rout, rarg = gnn.reduce_forward(g, x, "max")
    rdx = gnn.reduce_backward(g, rarg, dy)
    torch.cuda.synchronize()
    rf = oracle.reduce_forward(rp, ci, h.reshape(n, F), "max", sel=sel_f)
    sel_t = torch.from_numpy(np.asarray(sel_f, np.int64)).to(rarg.device)
    assert np.array_equal(rarg[sel_t].cpu().numpy(), rf["arg"]), f"cfg{idx} max arg"
    assert np.array_equal(_rows(rout, sel_f), rf["out"]), f"cfg{idx} max out"
    cheap_r = sel_b[cost[sel_b] < 2e4][:150]     # the oracle recomputes every row they win
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
    assert_close(_rows(lse, sel_f), f["lse"], w.dtype, None, f"cfg{idx} gatv2 lse")
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
    assert_close(_rows(lse, sel_f), f["lse"], w.dtype, None, f"cfg{idx} gt lse")
    b = oracle.gt_backward(rp, ci, h, xr, val, sc, dout, sel=sel_b, with_mag=True)
    for name, got in (("dq", dq), ("dkey", dk), ("dval", dv)):
        assert_close(_rows(got, sel_b), b[name], w.dtype, b[name + "_mag"], f"cfg{idx} gt {name}")
    assert outdeg[top].max() > 2048 or idx == 2       # a CSC hub was sampled
