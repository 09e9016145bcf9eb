"""Checks that pin the fp64 graph-transformer attention oracle to things other
than itself.

Each check takes an oracle object (the real one, or a build with a planted
mistake) and raises AssertionError when the oracle disagrees with:
  * a dense masked-softmax formulation in torch fp64 (logits = scale q k^T
    + log multiplicity, masked to the edges) and its autograd,
  * torch's scaled_dot_product_attention on a complete graph (every node
    attends to every node: ordinary dense attention),
  * central finite differences of L = sum(out * G),
  * special cases: q = 0 gives the neighbour mean of the values and
    lse = ln deg; one in-neighbour copies its value row with vanishing
    query and key gradients; the scale only multiplies q;
  * invariants: alpha sums to 1, zero in-degree gives 0 and -inf.
"""
from __future__ import annotations

import math

import numpy as np
import torch

import workload
from oracle_pins import close, csr_from_lists, irregular_graph


def rand(n, H, D, seed, dtype=np.float64):
    rng = np.random.default_rng(seed)
    return tuple(rng.standard_normal((n, H, D)).astype(dtype) for _ in range(4))


def dense_gt(row_ptr, col, q, k, v, scale, G):
    n = len(row_ptr) - 1
    cnt = np.zeros((n, n))
    for i in range(n):
        for j in col[row_ptr[i]:row_ptr[i + 1]]:
            cnt[i, j] += 1
    mask = torch.tensor(cnt > 0)
    logc = torch.tensor(np.log(np.where(cnt > 0, cnt, 1.0)))
    Q, K, Vt = (torch.tensor(np.asarray(x, np.float64), requires_grad=True) for x in (q, k, v))
    logits = scale * torch.einsum("ikd,jkd->ijk", Q, K) + logc[:, :, None]
    logits = torch.where(mask[:, :, None], logits, torch.full_like(logits, -math.inf))
    rows = torch.nonzero(mask.any(1)).flatten()
    P = torch.softmax(logits[rows], dim=1)
    out = torch.zeros_like(Vt).index_copy(0, rows, torch.einsum("ijk,jkd->ikd", P, Vt))
    lse = torch.full((n, q.shape[1]), -math.inf, dtype=torch.float64)
    lse[rows] = torch.logsumexp(logits[rows], dim=1).detach()
    (out * torch.tensor(np.asarray(G, np.float64))).sum().backward()
    return dict(out=out.detach().numpy(), lse=lse.numpy(), dq=Q.grad.numpy(),
                dkey=K.grad.numpy(), dval=Vt.grad.numpy())


def pin_gt_dense(o):
    graphs = [irregular_graph(12, 5), workload.erdos_renyi(48, 5.0, 11)]
    for gi, (rp, ci) in enumerate(graphs):
        n = len(rp) - 1
        q, k, v, G = rand(n, 2, 3, 60 + gi)
        ref = dense_gt(rp, ci, q, k, v, 0.6, G)
        f = o.gt_forward(rp, ci, q, k, v, 0.6)
        close(f["out"], ref["out"], 1e-11, 1e-13, "dense out")
        close(f["lse"], ref["lse"], 1e-11, 1e-13, "dense lse")
        b = o.gt_backward(rp, ci, q, k, v, 0.6, G)
        for key in ("dq", "dkey", "dval"):
            close(b[key], ref[key], 1e-10, 1e-12, "autograd " + key)
        sel = [1, 4, n - 1]
        bs = o.gt_backward(rp, ci, q, k, v, 0.6, G, sel=sel)
        for key in ("dq", "dkey", "dval"):
            close(bs[key], ref[key][sel], 1e-10, 1e-12, "sampled " + key)


def pin_gt_complete_graph_is_dense_attention(o):
    n, H, D = 24, 2, 8
    rp, ci = csr_from_lists([list(range(n)) for _ in range(n)])
    q, k, v, _ = rand(n, H, D, 7)
    f = o.gt_forward(rp, ci, q, k, v, 1.0 / math.sqrt(D))
    t = [torch.tensor(x).permute(1, 0, 2) for x in (q, k, v)]       # [H, n, D]
    ref = torch.nn.functional.scaled_dot_product_attention(*t).permute(1, 0, 2).numpy()
    close(f["out"], ref, 1e-11, 1e-13, "complete graph = dense attention")


def pin_gt_finite_differences(o):
    rp, ci = irregular_graph(9, 4)
    n = len(rp) - 1
    q, k, v, G = rand(n, 2, 2, 4)
    b = o.gt_backward(rp, ci, q, k, v, 0.8, G)

    def loss(*x):
        return float((o.gt_forward(rp, ci, *x, 0.8)["out"] * G).sum())

    eps = 1e-6
    for name, a, grad in (("q", 0, b["dq"]), ("key", 1, b["dkey"]), ("val", 2, b["dval"])):
        base = [q, k, v]
        fd = np.zeros_like(base[a])
        for idx in np.ndindex(*base[a].shape):
            p = [x.copy() for x in base]
            m = [x.copy() for x in base]
            p[a][idx] += eps
            m[a][idx] -= eps
            fd[idx] = (loss(*p) - loss(*m)) / (2 * eps)
        err = float(np.abs(fd - grad).max())
        assert err <= 1e-6 * max(1.0, float(np.abs(grad).max())), (name, err)


def pin_gt_special_cases(o):
    rp, ci = workload.erdos_renyi(150, 5.0, 21)
    n = len(rp) - 1
    q, k, v, G = rand(n, 2, 4, 21, np.float32)
    f = o.gt_forward(rp, ci, np.zeros_like(q), k, v, 0.5)
    deg = np.diff(rp)
    mean = np.add.reduceat(v[ci].astype(np.float64), rp[:-1], axis=0) / deg[:, None, None]
    close(f["out"], mean, 1e-13, 1e-14, "q=0 mean")
    close(f["lse"], np.log(deg)[:, None].repeat(2, 1), 1e-13, 1e-14, "q=0 ln deg")
    # the scale multiplies q: (scale s, q) = (scale 1, s q)
    q64, k64, v64 = (x.astype(np.float64) for x in (q, k, v))
    f1 = o.gt_forward(rp, ci, q64 * 0.25, k64, v64, 1.0)
    f2 = o.gt_forward(rp, ci, q64, k64, v64, 0.25)
    close(f1["out"], f2["out"], 1e-12, 1e-13, "scale")
    # one in-neighbour
    m = 7
    rp1, ci1 = csr_from_lists([[(i + 3) % m] for i in range(m)])
    q1, k1, v1, G1 = rand(m, 2, 4, 8, np.float32)
    f3 = o.gt_forward(rp1, ci1, q1, k1, v1, 0.5)
    assert np.array_equal(f3["out"], v1[ci1].astype(np.float64))
    b3 = o.gt_backward(rp1, ci1, q1, k1, v1, 0.5, G1)
    expect = np.empty_like(b3["dval"])
    expect[ci1] = G1.astype(np.float64)
    close(b3["dval"], expect, 1e-14, 1e-15, "single-neighbour dval")
    assert np.abs(b3["dq"]).max() <= 1e-14 and np.abs(b3["dkey"]).max() <= 1e-14


def pin_gt_invariants(o):
    rp, ci = irregular_graph(12, 9)
    n = len(rp) - 1
    q, k, v, G = rand(n, 3, 4, 9, np.float32)
    deg = np.diff(rp)
    f = o.gt_forward(rp, ci, q, k, v, 0.5, with_alpha_sum=True)
    assert np.all(np.abs(f["alpha_sum"][deg > 0] - 1.0) <= 1e-12)
    assert np.all(f["out"][deg == 0] == 0.0) and np.all(np.isneginf(f["lse"][deg == 0]))
    b = o.gt_backward(rp, ci, q, k, v, 0.5, G)
    assert np.all(b["dq"][deg == 0] == 0.0)
    qb, kb, vb = (workload.f32_to_bf16_bits(x) for x in (q, k, v))
    qw, kw, vw = (workload.bf16_bits_to_f32(x) for x in (qb, kb, vb))
    assert np.array_equal(o.gt_forward(rp, ci, qb, kb, vb, 0.5)["out"],
                          o.gt_forward(rp, ci, qw, kw, vw, 0.5)["out"])


ALL_PINS = [pin_gt_dense, pin_gt_complete_graph_is_dense_attention, pin_gt_finite_differences,
            pin_gt_special_cases, pin_gt_invariants]
