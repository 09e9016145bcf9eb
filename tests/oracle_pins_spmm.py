"""Checks that pin the fp64 SpMM-family oracle (GCN / GraphConv propagation,
out = A~ x, dx = A~^T dout) to things other than itself.

Each check takes an oracle object (the real one, or a build with a planted
mistake) and raises AssertionError when the oracle disagrees with:
  * a hand-derived worked example (three nodes, every normalisation),
  * the dense matrix formulation built with numpy (A from the edge list, D
    from its row sums, D^-1/2 A D^-1/2 / D^-1 A / A, then a matrix product),
  * closed forms: mean propagation of a constant, the D^1/2 1 eigenvector of
    the symmetric propagation on an undirected graph, a regular graph where
    all three normalisations agree up to the degree,
  * the adjoint identity <A~ x, y> = <x, A~^T y> tying backward to forward.
"""
from __future__ import annotations

import math

import numpy as np

import workload
from oracle_pins import close, csr_from_lists, irregular_graph

NORMS = ("sum", "mean", "sym")


def dense_propagation(row_ptr, col, norm):
    """A~ as a dense [N, N] float64 matrix from the edge list."""
    n = len(row_ptr) - 1
    A = np.zeros((n, n))
    dst = np.repeat(np.arange(n), np.diff(row_ptr))
    np.add.at(A, (dst, np.asarray(col, np.int64)), 1.0)
    deg = A.sum(1)
    if norm == "sum":
        return A
    inv = np.where(deg > 0, 1.0 / np.where(deg > 0, deg, 1.0), 0.0)
    if norm == "mean":
        return inv[:, None] * A
    isq = np.sqrt(inv)
    return isq[:, None] * A * isq[None, :]


def pin_spmm_worked_example(o):
    """Rows: 0 <- {0, 1}, 1 <- {0}, 2 <- {}; x = [[0, 1], [2, 3], [4, 5]].
    In-degrees 2, 1, 0.  By hand:
      sum:  out0 = x0 + x1 = [2, 4], out1 = x0 = [0, 1], out2 = 0;
            dx0 = dout0 + dout1, dx1 = dout0, dx2 = 0 (dout = x here)
      mean: out0 = (x0 + x1) / 2 = [1, 2], out1 = [0, 1];
            dx0 = dout0 / 2 + dout1 = [2, 3.5], dx1 = dout0 / 2 = [0, 0.5]
      sym:  coef(0<-0) = 1/2, coef(0<-1) = 1/sqrt(2), coef(1<-0) = 1/sqrt(2);
            out0 = [sqrt(2), 1/2 + 3/sqrt(2)], out1 = [0, 1/sqrt(2)];
            A~ is symmetric here, so dx = out."""
    rp, ci = csr_from_lists([[0, 1], [0], []])
    x = np.array([[0, 1], [2, 3], [4, 5]], np.float32)
    r2 = math.sqrt(2.0)
    expect = {
        "sum": ([[2, 4], [0, 1], [0, 0]], [[2, 4], [0, 1], [0, 0]]),
        "mean": ([[1, 2], [0, 1], [0, 0]], [[2, 3.5], [0, 0.5], [0, 0]]),
        "sym": ([[r2, 0.5 + 3 / r2], [0, 1 / r2], [0, 0]],
                [[r2, 0.5 + 3 / r2], [0, 1 / r2], [0, 0]]),
    }
    for norm, (fwd, bwd) in expect.items():
        close(o.spmm_forward(rp, ci, x, norm)["out"], fwd, 1e-15, 1e-15, f"worked {norm} out")
        close(o.spmm_backward(rp, ci, x, norm)["dx"], bwd, 1e-15, 1e-15, f"worked {norm} dx")


def pin_spmm_dense(o):
    """Against the dense matrix product on graphs with isolated nodes, a hub,
    a multi-edge and sources without in-edges."""
    graphs = [irregular_graph(12, 5), workload.erdos_renyi(64, 6.0, 11)]
    rows = [[1, 1, 2], [], [0, 3], [2]]             # node 1: no in-edges, but a source
    graphs.append(csr_from_lists(rows))
    rng = np.random.default_rng(3)
    for rp, ci in graphs:
        n = len(rp) - 1
        x = rng.standard_normal((n, 5))
        g = rng.standard_normal((n, 5))
        for norm in NORMS:
            A = dense_propagation(rp, ci, norm)
            close(o.spmm_forward(rp, ci, x, norm)["out"], A @ x, 1e-13, 1e-14, f"dense {norm}")
            close(o.spmm_backward(rp, ci, g, norm)["dx"], A.T @ g, 1e-13, 1e-14,
                  f"dense {norm} transpose")


def pin_spmm_closed_forms(o):
    # mean propagation keeps a constant on every node with in-edges, 0 elsewhere
    rp, ci = irregular_graph(12, 9)
    n = len(rp) - 1
    c = np.full((n, 3), 2.5)
    deg = np.diff(rp)
    out = o.spmm_forward(rp, ci, c, "mean")["out"]
    close(out, np.where(deg[:, None] > 0, 2.5, 0.0) * np.ones((n, 3)), 1e-14, 0, "mean const")
    # undirected graph with self-loops: A~_sym D^1/2 1 = D^1/2 1
    rng = np.random.default_rng(4)
    m = 40
    pairs = {(int(a), int(b)) for a, b in rng.integers(0, m, (120, 2)) if a != b}
    adj = [[i] for i in range(m)]
    for a, b in pairs:
        if b not in adj[a]:
            adj[a].append(b)
            adj[b].append(a)
    rp2, ci2 = csr_from_lists([sorted(r) for r in adj])
    v = np.sqrt(np.diff(rp2).astype(np.float64))[:, None]
    close(o.spmm_forward(rp2, ci2, v, "sym")["out"], v, 1e-13, 0, "sym eigenvector")
    close(o.spmm_backward(rp2, ci2, v, "sym")["dx"], v, 1e-13, 0, "sym eigenvector (T)")
    # circulant graph, every in-degree k: sym = mean = sum / k
    k, m = 5, 30
    rp3, ci3 = csr_from_lists([sorted((i + s) % m for s in range(k)) for i in range(m)])
    x = rng.standard_normal((m, 4))
    s = o.spmm_forward(rp3, ci3, x, "sum")["out"]
    close(o.spmm_forward(rp3, ci3, x, "mean")["out"], s / k, 1e-14, 1e-15, "regular mean")
    close(o.spmm_forward(rp3, ci3, x, "sym")["out"], s / k, 1e-14, 1e-15, "regular sym")


def pin_spmm_adjoint(o):
    """<A~ x, y> = <x, A~^T y>, and the per-row backward agrees."""
    rp, ci = workload.chung_lu(300, 2.1, 6.0, 100.0, 17)
    n = len(rp) - 1
    rng = np.random.default_rng(17)
    x = rng.standard_normal((n, 3, 2))
    y = rng.standard_normal((n, 3, 2))
    for norm in NORMS:
        ax = o.spmm_forward(rp, ci, x, norm)["out"]
        aty = o.spmm_backward(rp, ci, y, norm)["dx"]
        lhs = float((ax * y.reshape(n, -1)).sum())
        rhs = float((x.reshape(n, -1) * aty).sum())
        assert abs(lhs - rhs) <= 1e-11 * max(1.0, abs(lhs)), (norm, lhs, rhs)
        sel = [0, 5, 17, n - 1]
        close(o.spmm_backward_rows(rp, ci, y, norm, sel)["dx"], aty[sel], 1e-14, 1e-15,
              f"rows {norm}")
        close(o.spmm_forward(rp, ci, x, norm, sel=sel)["out"], ax[sel], 1e-14, 0,
              f"sel {norm}")


def pin_spmm_bf16(o):
    """bfloat16 bit patterns widen exactly."""
    rp, ci = workload.erdos_renyi(80, 5.0, 51)
    n = len(rp) - 1
    x32 = workload.normal_f32(51, 1, (n, 16))
    xb = workload.f32_to_bf16_bits(x32)
    xw = workload.bf16_bits_to_f32(xb)
    for norm in NORMS:
        assert np.array_equal(o.spmm_forward(rp, ci, xb, norm)["out"],
                              o.spmm_forward(rp, ci, xw, norm)["out"])
        assert np.array_equal(o.spmm_backward(rp, ci, xb, norm)["dx"],
                              o.spmm_backward(rp, ci, xw, norm)["dx"])


ALL_PINS = [pin_spmm_worked_example, pin_spmm_dense, pin_spmm_closed_forms, pin_spmm_adjoint,
            pin_spmm_bf16]
