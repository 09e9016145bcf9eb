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
