"""Checks that pin the fp64 GATv2 oracle to things other than itself.

Each check takes an oracle object (the real one, or a build with a planted
mistake) and raises AssertionError when the oracle disagrees with:
  * a dense masked-softmax formulation in torch fp64 (logits[i, j, k] =
    att[k] . LeakyReLU(xr[i, k] + xl[j, k]) + log multiplicity) and its
    autograd, on graphs with isolated nodes, a hub and multi-edges,
  * central finite differences of L = sum(out * G),
  * special cases: att = 0 gives the neighbour mean and lse = ln deg; one
    in-neighbour copies its row and makes every score gradient vanish;
    slope 1 makes the score additive, so it equals the GAT score with
    a_dst = a_src = att on h = xl = xr;
  * invariants: alpha sums to 1, Delta_i = dout_i . out_i, zero in-degree.
"""
from __future__ import annotations

import math

import numpy as np
import torch

import workload
from oracle_pins import close, csr_from_lists, irregular_graph


def rand(n, H, D, seed, dtype=np.float64):
    rng = np.random.default_rng(seed)
    xl = rng.standard_normal((n, H, D)).astype(dtype)
    xr = rng.standard_normal((n, H, D)).astype(dtype)
    att = (0.5 * rng.standard_normal((H, D))).astype(dtype)
    G = rng.standard_normal((n, H, D)).astype(dtype)
    return xl, xr, att, G


def dense_gatv2(row_ptr, col, xl, xr, att, slope, G):
    n = len(row_ptr) - 1
    cnt = np.zeros((n, n))
    for i in range(n):
        for j in col[row_ptr[i]:row_ptr[i + 1]]:
            cnt[i, j] += 1
    mask = torch.tensor(cnt > 0)
    logc = torch.tensor(np.log(np.where(cnt > 0, cnt, 1.0)))
    L = torch.tensor(np.asarray(xl, np.float64), requires_grad=True)
    R = torch.tensor(np.asarray(xr, np.float64), requires_grad=True)
    A = torch.tensor(np.asarray(att, np.float64), requires_grad=True)
    z = R[:, None] + L[None, :]                                   # [i, j, H, D]
    logits = (torch.nn.functional.leaky_relu(z, slope) * A).sum(-1) + logc[:, :, None]
    logits = torch.where(mask[:, :, None], logits, torch.full_like(logits, -math.inf))
    rows = torch.nonzero(mask.any(1)).flatten()
    P = torch.softmax(logits[rows], dim=1)
    out = torch.zeros_like(L).index_copy(0, rows, torch.einsum("ijk,jkd->ikd", P, L))
    lse = torch.full((n, xl.shape[1]), -math.inf, dtype=torch.float64)
    lse[rows] = torch.logsumexp(logits[rows], dim=1).detach()
    (out * torch.tensor(np.asarray(G, np.float64))).sum().backward()
    return dict(out=out.detach().numpy(), lse=lse.numpy(), dxl=L.grad.numpy(),
                dxr=R.grad.numpy(), datt=A.grad.numpy())


def pin_gatv2_dense(o):
    graphs = [irregular_graph(12, 5), workload.erdos_renyi(48, 5.0, 11)]
    for gi, (rp, ci) in enumerate(graphs):
        n = len(rp) - 1
        xl, xr, att, G = rand(n, 2, 3, 40 + gi)
        ref = dense_gatv2(rp, ci, xl, xr, att, 0.2, G)
        f = o.gatv2_forward(rp, ci, xl, xr, att, 0.2)
        close(f["out"], ref["out"], 1e-11, 1e-13, "dense out")
        close(f["lse"], ref["lse"], 1e-11, 1e-13, "dense lse")
        b = o.gatv2_backward(rp, ci, xl, xr, att, 0.2, G)
        close(b["dxl"], ref["dxl"], 1e-10, 1e-12, "autograd dxl")
        close(b["dxr"], ref["dxr"], 1e-10, 1e-12, "autograd dxr")
        close(b["datt"], ref["datt"], 1e-10, 1e-12, "autograd datt")
        sel = [0, 3, n - 1]
        bs = o.gatv2_backward(rp, ci, xl, xr, att, 0.2, G, sel=sel)
        close(bs["dxl"], ref["dxl"][sel], 1e-10, 1e-12, "sampled dxl")
        close(bs["dxr"], ref["dxr"][sel], 1e-10, 1e-12, "sampled dxr")
        fs = o.gatv2_forward(rp, ci, xl, xr, att, 0.2, sel=sel)
        close(fs["out"], ref["out"][sel], 1e-11, 1e-13, "sampled out")


def pin_gatv2_finite_differences(o):
    rp, ci = irregular_graph(9, 4)
    n = len(rp) - 1
    xl, xr, att, G = rand(n, 2, 2, 4)
    b = o.gatv2_backward(rp, ci, xl, xr, att, 0.2, G)

    def loss(l, r, a):
        return float((o.gatv2_forward(rp, ci, l, r, a, 0.2)["out"] * G).sum())

    eps = 1e-6
    for name, k, grad in (("xl", 0, b["dxl"]), ("xr", 1, b["dxr"]), ("att", 2, b["datt"])):
        base = [xl, xr, att]
        fd = np.zeros_like(base[k])
        for idx in np.ndindex(*base[k].shape):
            p = [x.copy() for x in base]
            m = [x.copy() for x in base]
            p[k][idx] += eps
            m[k][idx] -= eps
            fd[idx] = (loss(*p) - loss(*m)) / (2 * eps)
        err = float(np.abs(fd - grad).max())
        assert err <= 1e-6 * max(1.0, float(np.abs(grad).max())), (name, err)


def pin_gatv2_special_cases(o):
    # att = 0: every score 0 -> neighbour mean, lse = ln deg
    rp, ci = workload.erdos_renyi(150, 5.0, 21)
    n = len(rp) - 1
    xl, xr, _, _ = rand(n, 2, 4, 21, np.float32)
    z = np.zeros((2, 4), np.float32)
    f = o.gatv2_forward(rp, ci, xl, xr, z, 0.2)
    deg = np.diff(rp)
    mean = np.add.reduceat(xl[ci].astype(np.float64), rp[:-1], axis=0) / deg[:, None, None]
    close(f["out"], mean, 1e-13, 1e-14, "att=0 mean")
    close(f["lse"], np.log(deg)[:, None].repeat(2, 1), 1e-13, 1e-14, "att=0 ln deg")
    # one in-neighbour: out = xl_j exactly, score gradients vanish
    m = 7
    rp1, ci1 = csr_from_lists([[(i + 2) % m] for i in range(m)])
    xl1, xr1, att1, G1 = rand(m, 2, 4, 8, np.float32)
    f1 = o.gatv2_forward(rp1, ci1, xl1, xr1, att1, 0.2)
    assert np.array_equal(f1["out"], xl1[ci1].astype(np.float64))
    b1 = o.gatv2_backward(rp1, ci1, xl1, xr1, att1, 0.2, G1)
    expect = np.empty_like(b1["dxl"])
    expect[ci1] = G1.astype(np.float64)
    close(b1["dxl"], expect, 1e-14, 1e-15, "single-neighbour dxl")
    assert np.abs(b1["dxr"]).max() <= 1e-14 and np.abs(b1["datt"]).max() <= 1e-14
    # slope 1: e = att . xr_i + att . xl_j, the GAT score with a_dst = a_src = att
    rp2, ci2 = workload.erdos_renyi(80, 6.0, 5)
    n2 = len(rp2) - 1
    h, _, att2, G2 = rand(n2, 2, 4, 5)
    v2 = o.gatv2_forward(rp2, ci2, h, h, att2, 1.0)
    v1 = o.forward(rp2, ci2, h, att2, att2, 1.0)
    close(v2["out"], v1["out"], 1e-12, 1e-13, "slope 1 = GAT out")
    close(v2["lse"], v1["lse"], 1e-12, 1e-13, "slope 1 = GAT lse")


def pin_gatv2_kink_worked_example(o):
    """Node 0 <- {0, 1}, node 1 <- {}; H = D = 1; xr0 = -1, xl = [1, 3];
    att = 1, slope 0.2, dout0 = 1.  By hand: z00 = 0 (on the kink), z01 = 2,
    so e = (0, 2), alpha = (p, 1 - p) with p = 1 / (1 + e^2), out0 = 3 - 2p,
    lse0 = log(1 + e^2).  da = (1, 3), Delta = 3 - 2p, de = (-2p(1-p),
    2p(1-p)).  With the derivative at z = 0 taken as the slope,
    dxr0 = 0.2 de0 + 1 de1 = 0.8 * 2p(1-p); dxl0 = p + 0.2 de0,
    dxl1 = (1 - p) + de1; datt = de0 * 0 + de1 * 2."""
    rp, ci = csr_from_lists([[0, 1], []])
    xl = np.array([1, 3], np.float32).reshape(2, 1, 1)
    xr = np.array([-1, 0], np.float32).reshape(2, 1, 1)
    att = np.ones((1, 1), np.float32)
    G = np.array([1, 0], np.float32).reshape(2, 1, 1)
    p = 1.0 / (1.0 + math.exp(2.0))
    de1 = 2 * p * (1 - p)
    f = o.gatv2_forward(rp, ci, xl, xr, att, 0.2)
    close(f["out"].ravel(), [3 - 2 * p, 0.0], 1e-14, 1e-15, "kink out")
    close(f["lse"].ravel()[:1], [math.log(1 + math.exp(2.0))], 1e-14, 1e-15, "kink lse")
    b = o.gatv2_backward(rp, ci, xl, xr, att, 0.2, G)
    close(b["dxr"].ravel(), [0.8 * de1, 0.0], 1e-13, 1e-15, "kink dxr")
    close(b["dxl"].ravel(), [p - 0.2 * de1, (1 - p) + de1], 1e-13, 1e-15, "kink dxl")
    close(b["datt"].ravel(), [2 * de1], 1e-13, 1e-15, "kink datt")


def pin_gatv2_invariants(o):
    rp, ci = irregular_graph(12, 9)
    n = len(rp) - 1
    xl, xr, att, G = rand(n, 3, 4, 9, np.float32)
    deg = np.diff(rp)
    f = o.gatv2_forward(rp, ci, xl, xr, att, 0.2, with_alpha_sum=True)
    assert np.all(np.abs(f["alpha_sum"][deg > 0] - 1.0) <= 1e-12)
    assert np.all(f["out"][deg == 0] == 0.0) and np.all(np.isneginf(f["lse"][deg == 0]))
    delta = o.gatv2_delta(rp, ci, xl, xr, att, 0.2, G)
    close(delta, (G.astype(np.float64) * f["out"]).sum(-1), 1e-12, 1e-13, "Delta identity")
    b = o.gatv2_backward(rp, ci, xl, xr, att, 0.2, G)
    assert np.all(b["dxr"][deg == 0] == 0.0)
    # bf16 bit patterns widen exactly
    xlb, xrb, Gb = (workload.f32_to_bf16_bits(x) for x in (xl, xr, G))
    xlw, xrw, Gw = (workload.bf16_bits_to_f32(x) for x in (xlb, xrb, Gb))
    assert np.array_equal(o.gatv2_forward(rp, ci, xlb, xrb, att, 0.2)["out"],
                          o.gatv2_forward(rp, ci, xlw, xrw, att, 0.2)["out"])
    assert np.array_equal(o.gatv2_backward(rp, ci, xlb, xrb, att, 0.2, Gb)["dxl"],
                          o.gatv2_backward(rp, ci, xlw, xrw, att, 0.2, Gw)["dxl"])


ALL_PINS = [pin_gatv2_kink_worked_example, pin_gatv2_dense, pin_gatv2_finite_differences,
            pin_gatv2_special_cases, pin_gatv2_invariants]
