"""Small hand-shaped graphs for edge cases (numpy, seeded).

These complement the benchmark generators: they allow zero in-degree nodes,
multi-edges, in-degrees placed exactly around tiling thresholds, and sources
with very large out-degree.  Like the rest of this package they only draw
inputs.  CSR convention as in ``workload``: row i lists the sources of i.
"""
from __future__ import annotations

import numpy as np


def csr_from_rows(rows):
    row_ptr = np.zeros(len(rows) + 1, np.int32)
    for i, r in enumerate(rows):
        row_ptr[i + 1] = row_ptr[i] + len(r)
    col = np.array([j for r in rows for j in r], dtype=np.int32)
    return row_ptr, col


def with_in_degrees(degrees, n_nodes=None, seed=0, src_skew=1.2, sort_rows=True):
    """Node i gets exactly degrees[i] in-edges (nodes past len(degrees) get a
    random small in-degree).  Sources follow a Zipf-like law over a random
    node order (exponent src_skew), so a few sources have very large
    out-degree; repeated sources are kept as multi-edges."""
    rng = np.random.default_rng(seed)
    degrees = list(degrees)
    n = n_nodes if n_nodes is not None else len(degrees)
    n = max(n, len(degrees), 1)
    degs = np.array(degrees + list(rng.integers(0, 6, size=n - len(degrees))), dtype=np.int64)
    rank = rng.permutation(n)
    w = 1.0 / np.power(np.arange(1, n + 1, dtype=np.float64), src_skew)
    w /= w.sum()
    total = int(degs.sum())
    src = rank[rng.choice(n, size=total, p=w)].astype(np.int32)
    row_ptr = np.zeros(n + 1, np.int32)
    row_ptr[1:] = np.cumsum(degs)
    if sort_rows:
        for i in range(n):
            src[row_ptr[i]:row_ptr[i + 1]].sort()
    return row_ptr, src


def ring(n):
    """Each node has exactly one in-neighbour: i <- (i + 1) mod n."""
    return csr_from_rows([[(i + 1) % n] for i in range(n)])


def isolated(n):
    """n nodes, no edges."""
    return np.zeros(n + 1, np.int32), np.zeros(0, np.int32)


def star_in(n):
    """Node 0 receives an edge from every node (itself included)."""
    rows = [list(range(n))] + [[i] for i in range(1, n)]
    return csr_from_rows(rows)


def star_out(n, extra=1):
    """Node 0 sends an edge to every node; every node also has `extra`
    in-edges from node 1 (a multi-edge when extra > 1)."""
    rows = [[0] + [1] * extra for _ in range(n)]
    return csr_from_rows(rows)


def paired_sources(n_a, n_b, n_c, seed=0, skew=1.6):
    """Three node groups: A = [0, n_a), B = [n_a, n_a + n_b) and the
    destinations C after them.  Each destination has exactly two in-edges,
    from one A node (Zipf law of exponent `skew` over A, so A's first node
    is a large out-degree hub) and from one B node (uniform); A and B nodes
    have none."""
    rng = np.random.default_rng(seed)
    a_of = np.minimum(rng.zipf(skew, n_c) - 1, n_a - 1).astype(np.int32)
    b_of = (n_a + rng.integers(0, n_b, n_c)).astype(np.int32)
    n = n_a + n_b + n_c
    row_ptr = np.zeros(n + 1, np.int32)
    row_ptr[n_a + n_b + 1:] = 2 * np.arange(1, n_c + 1, dtype=np.int32)
    col = np.empty(2 * n_c, np.int32)
    col[0::2] = a_of
    col[1::2] = b_of
    return row_ptr, col
