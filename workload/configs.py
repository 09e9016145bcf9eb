"""The five synthetic workloads of the benchmark, as data, plus their builders.

The pages measure on OGB, citation and GraphLand graphs, which are not
available here; these synthetic graphs stand in for them: a tiny
Erdos-Renyi graph (oracle-sized), a low-skew uniform graph, two Chung-Lu
power-law graphs and an R-MAT graph in two node orders.

Seeds: ``20261202 + config index``.  Feature streams: h = 1, a_src = 2,
a_dst = 3, dout = 4 (each an independent counter-based stream).
"""
from __future__ import annotations

from dataclasses import dataclass, field

import numpy as np

SEED_BASE = 20261202
STREAM_H, STREAM_ASRC, STREAM_ADST, STREAM_DOUT = 1, 2, 3, 4


@dataclass(frozen=True)
class Workload:
    index: int
    name: str
    kind: str                 # er | uniform | chung_lu | rmat
    params: dict = field(default_factory=dict)
    H: int = 1
    D: int = 16
    dtype: str = "f32"        # f32 | bf16
    slope: float = 0.2
    order: str = "natural"    # natural | random | rcm | hubs_rcm

    @property
    def seed(self) -> int:
        return SEED_BASE + self.index


CONFIGS = {
    1: Workload(1, "er_n512_deg8_h1d16_f32", "er", dict(n=512, avg=8.0), H=1, D=16, dtype="f32"),
    2: Workload(2, "uniform_n100k_deg16_h4d32_f32", "uniform", dict(n=100_000, k=16), H=4, D=32,
                dtype="f32"),
    3: Workload(3, "chunglu_n1m_g2.1_avg20_cap100k_h8d16_bf16", "chung_lu",
                dict(n=1_000_000, gamma=2.1, avg=20.0, cap=100_000.0), H=8, D=16, dtype="bf16"),
    4: Workload(4, "chunglu_n2.4m_g2.3_avg50_h1d128_bf16", "chung_lu",
                dict(n=2_400_000, gamma=2.3, avg=50.0, cap=2_399_999.0), H=1, D=128, dtype="bf16"),
    5: Workload(5, "rmat_s22_ef32_h4d64_bf16_randomids", "rmat",
                dict(scale=22, ef=32, a=0.57, b=0.19, c=0.19), H=4, D=64, dtype="bf16",
                order="random"),
    6: Workload(5, "rmat_s22_ef32_h4d64_bf16_rcm", "rmat",
                dict(scale=22, ef=32, a=0.57, b=0.19, c=0.19), H=4, D=64, dtype="bf16",
                order="rcm"),
    # the alternative reading of the reordered run: hubs first, then RCM
    7: Workload(5, "rmat_s22_ef32_h4d64_bf16_hubs_rcm", "rmat",
                dict(scale=22, ef=32, a=0.57, b=0.19, c=0.19), H=4, D=64, dtype="bf16",
                order="hubs_rcm"),
}

# nodes above this in- plus out-degree lead the hubs-first order (the
# default tiling's largest in-degree handled by one thread block)
HUB_DEGREE = 4096


def make_graph(w: Workload):
    """CSR (row_ptr, col_idx) of a workload, deterministic in its seed."""
    from . import (erdos_renyi, uniform, chung_lu, rmat, permute_random, rcm_order, relabel,
                   hubs_then_rcm_order)
    p = w.params
    if w.kind == "er":
        g = erdos_renyi(p["n"], p["avg"], w.seed)
    elif w.kind == "uniform":
        g = uniform(p["n"], p["k"], w.seed)
    elif w.kind == "chung_lu":
        g = chung_lu(p["n"], p["gamma"], p["avg"], p["cap"], w.seed)
    elif w.kind == "rmat":
        g = rmat(p["scale"], p["ef"], p["a"], p["b"], p["c"], w.seed)
    else:
        raise ValueError(w.kind)
    if w.order in ("random", "rcm", "hubs_rcm"):
        g = permute_random(g[0], g[1], w.seed)
    if w.order == "rcm":
        g = relabel(g[0], g[1], rcm_order(g[0], g[1]))
    if w.order == "hubs_rcm":
        g = relabel(g[0], g[1], hubs_then_rcm_order(g[0], g[1], HUB_DEGREE))
    return g


def make_features(w: Workload, n_nodes: int, with_dout: bool = True):
    """h [N,H,D], a_src [H,D], a_dst [H,D], dout [N,H,D].

    h and dout ~ N(0, 1), a ~ N(0, 0.1) (0.1 read as the standard deviation).
    For bf16 workloads h and dout are returned as uint16 bit patterns.
    """
    from . import normal_f32, f32_to_bf16_bits
    H, D = w.H, w.D
    h = normal_f32(w.seed, STREAM_H, (n_nodes, H, D), 1.0)
    a_src = normal_f32(w.seed, STREAM_ASRC, (H, D), 0.1)
    a_dst = normal_f32(w.seed, STREAM_ADST, (H, D), 0.1)
    dout = normal_f32(w.seed, STREAM_DOUT, (n_nodes, H, D), 1.0) if with_dout else None
    if w.dtype == "bf16":
        h = f32_to_bf16_bits(h)
        dout = f32_to_bf16_bits(dout) if dout is not None else None
    return h, a_src, a_dst, dout


def degree_stats(row_ptr: np.ndarray, col: np.ndarray) -> dict:
    n = len(row_ptr) - 1
    indeg = np.diff(row_ptr)
    outdeg = np.bincount(col, minlength=n)
    return dict(n=n, e=int(len(col)), max_in=int(indeg.max(initial=0)),
                max_out=int(outdeg.max(initial=0)))
