"""Checks that pin the fp64 reduction-family oracle (max / min over
in-neighbours with the winning source, and its gradient) to things other
than itself.

Each check takes an oracle object (the real one, or a build with a planted
mistake) and raises AssertionError when the oracle disagrees with:
  * a hand-derived worked example with ties, an empty row and both ops,
  * a dense brute force with numpy (masked max/min and first-occurrence
    argmax/argmin over the source axis),
  * the identity min(x) = -max(-x) (same winners),
  * central finite differences of L = sum(out * G) on fp64 inputs,
  * conservation: every destination with in-edges passes its whole dout on.
"""
from __future__ import annotations

import numpy as np

import workload
from oracle_pins import close, csr_from_lists, irregular_graph


def pin_reduce_worked_example(o):
    """Rows 0 <- {0, 1, 2}, 1 <- {0}, 2 <- {}; x = [[1, 5], [3, 5], [3, -1]].
    max: row 0 feature 0 ties 3 = 3 between sources 1 and 2 -> source 1;
         feature 1 ties 5 = 5 between 0 and 1 -> source 0; row 1 copies x0;
         row 2 is empty -> 0 with source -1.
    min: row 0 -> 1 (source 0) and -1 (source 2).
    Backward of max with dout = 1: dx0 = [1, 2] (row 1 f0; rows 0 and 1 f1),
    dx1 = [1, 0] (row 0 f0), dx2 = 0."""
    rp, ci = csr_from_lists([[0, 1, 2], [0], []])
    x = np.array([[1, 5], [3, 5], [3, -1]], np.float32)
    mx = o.reduce_forward(rp, ci, x, "max")
    assert np.array_equal(mx["out"], [[3, 5], [1, 5], [0, 0]])
    assert np.array_equal(mx["arg"], [[1, 0], [0, 0], [-1, -1]])
    mn = o.reduce_forward(rp, ci, x, "min")
    assert np.array_equal(mn["out"], [[1, -1], [1, 5], [0, 0]])
    assert np.array_equal(mn["arg"], [[0, 2], [0, 0], [-1, -1]])
    b = o.reduce_backward(mx["arg"], np.ones((3, 2), np.float32))
    assert np.array_equal(b["dx"], [[1, 2], [1, 0], [0, 0]])
    br = o.reduce_backward_rows(rp, ci, x, "max", np.ones((3, 2), np.float32), [2, 0])
    assert np.array_equal(br["dx"], [[0, 0], [1, 2]])


def dense_reduce(row_ptr, col, x, op):
    n = len(row_ptr) - 1
    mask = np.zeros((n, n), bool)
    dst = np.repeat(np.arange(n), np.diff(row_ptr))
    mask[dst, np.asarray(col, np.int64)] = True
    xv = np.asarray(x, np.float64)
    fill = -np.inf if op == "max" else np.inf
    cube = np.where(mask[:, :, None], xv[None, :, :], fill)      # [i, j, f]
    arg = np.argmax(cube, axis=1) if op == "max" else np.argmin(cube, axis=1)
    out = np.take_along_axis(cube, arg[:, None, :], axis=1)[:, 0, :]
    empty = ~mask.any(1)
    out[empty] = 0.0
    arg[empty] = -1
    return out, arg


def pin_reduce_dense(o):
    rng = np.random.default_rng(8)
    graphs = [irregular_graph(12, 5), workload.erdos_renyi(60, 5.0, 3)]
    for rp, ci in graphs:
        n = len(rp) - 1
        xs = [rng.standard_normal((n, 6)),
              rng.integers(-2, 3, (n, 6)).astype(np.float32)]     # many ties
        for x in xs:
            for op in ("max", "min"):
                out, arg = dense_reduce(rp, ci, x, op)
                r = o.reduce_forward(rp, ci, x, op)
                assert np.array_equal(r["out"], out), op
                assert np.array_equal(r["arg"], arg), op


def pin_reduce_min_is_negated_max(o):
    rp, ci = workload.chung_lu(400, 2.1, 6.0, 200.0, 5)
    n = len(rp) - 1
    x = np.random.default_rng(5).integers(-50, 50, (n, 8)).astype(np.float64)
    mx = o.reduce_forward(rp, ci, -x, "max")
    mn = o.reduce_forward(rp, ci, x, "min")
    assert np.array_equal(mn["out"], -mx["out"]) and np.array_equal(mn["arg"], mx["arg"])


def pin_reduce_finite_differences(o):
    """dL/dx by central differences of L = sum(out * G) (no ties: continuous
    random values), against the backward of the forward's winners."""
    rp, ci = irregular_graph(10, 3)
    n = len(rp) - 1
    rng = np.random.default_rng(3)
    x = rng.standard_normal((n, 3))
    G = rng.standard_normal((n, 3))
    for op in ("max", "min"):
        b = o.reduce_backward(o.reduce_forward(rp, ci, x, op)["arg"], G)["dx"]
        eps = 1e-7
        fd = np.zeros_like(x)
        for idx in np.ndindex(*x.shape):
            p, m = x.copy(), x.copy()
            p[idx] += eps
            m[idx] -= eps
            fd[idx] = ((o.reduce_forward(rp, ci, p, op)["out"] * G).sum()
                       - (o.reduce_forward(rp, ci, m, op)["out"] * G).sum()) / (2 * eps)
        close(b, fd, 1e-6, 1e-8, f"finite differences {op}")


def pin_reduce_conservation(o):
    rp, ci = workload.chung_lu(2000, 2.1, 8.0, 500.0, 9)
    n = len(rp) - 1
    rng = np.random.default_rng(9)
    x = rng.standard_normal((n, 5))
    dout = rng.standard_normal((n, 5))
    r = o.reduce_forward(rp, ci, x, "max")
    b = o.reduce_backward(r["arg"], dout)
    has = np.diff(rp) > 0
    close(b["dx"].sum(0), dout[has].sum(0), 1e-12, 1e-12, "conservation")
    sel = [0, 7, 99, n - 1]
    close(o.reduce_backward_rows(rp, ci, x, "max", dout, sel)["dx"], b["dx"][sel], 1e-14, 1e-15,
          "backward rows")
    s = o.reduce_forward(rp, ci, x, "max", sel=sel)
    assert np.array_equal(s["out"], r["out"][sel]) and np.array_equal(s["arg"], r["arg"][sel])


def pin_reduce_bf16(o):
    rp, ci = workload.erdos_renyi(80, 5.0, 51)
    n = len(rp) - 1
    xb = workload.f32_to_bf16_bits(workload.normal_f32(51, 1, (n, 16)))
    xw = workload.bf16_bits_to_f32(xb)
    for op in ("max", "min"):
        a, b = o.reduce_forward(rp, ci, xb, op), o.reduce_forward(rp, ci, xw, op)
        assert np.array_equal(a["out"], b["out"]) and np.array_equal(a["arg"], b["arg"])


ALL_PINS = [pin_reduce_worked_example, pin_reduce_dense, pin_reduce_min_is_negated_max,
            pin_reduce_finite_differences, pin_reduce_conservation, pin_reduce_bf16]
