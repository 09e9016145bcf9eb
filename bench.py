#!/usr/bin/env python3
"""Benchmark of the fused GAT neighbour aggregation (forward + backward).

One step = one forward and one backward pass over one synthetic graph whose
inputs are resident in device memory (the graph is prepared once, outside the
timed region, as in training).  Default workload: the largest one, an R-MAT
graph of scale 22 (4,194,304 nodes, edge factor 32, about 132.5M edges after
duplicates are dropped and self-loops added) with random node ids, H = 4,
D = 64, bfloat16 features accumulated in float32.

    python bench.py [--gpus N] [--steps K] [--warmup W] [--config C]
    python bench.py --impl reference ...   # the fp64 CPU oracle, timed on the host

Prints one JSON line on rank 0.  `value` is forward+backward throughput in
GEdge*head/s (E * H / step time, E counting self-loops); a step passes one
workspace to both calls, so the backward reuses the forward's per-node
scores.  The forward-only figure, the forward and backward call fractions of
the HBM roofline, per-kernel times (from a separate instrumented pass), the
HBM roofline of the dominant kernel with its ncu DRAM traffic, an end-to-end
figure through the public API with host buffers and the host link's measured
rates, warm-L2 and CUDA-graph figures, the memory split, the oracle's CPU
throughput and the SM clocks seen during the timed region ride along.  On the
default workload a `power_law` list adds a compact line for each of the two
Chung-Lu graphs and the reordered R-MAT graph.
Under torchrun each rank runs an independent replica of the workload (the
operation has no exchange step on one graph); the max time over ranks is
used and `value` sums the replicas' units.
"""
from __future__ import annotations

import argparse
import ctypes
import hashlib
import json
import os
import statistics
import subprocess
import sys
import threading
import time

import numpy as np

ROOT = os.path.dirname(os.path.abspath(__file__))
sys.path.insert(0, ROOT)

METRIC = "GEdge·head/s fwd and fwd+bwd GAT aggregation; achieved HBM GB/s vs roofline"
UNIT = "GEdge*head/s"
DEFAULT_CONFIG = 5
# compact lines beside the default: both Chung-Lu graphs and R-MAT in RCM order
SUB_CONFIGS = (3, 4, 6)
FWD_EVENTS, BWD_EVENTS = 4, 8
FWD_KERNELS = ["fwd_scores", "fwd_main", "fwd_merge"]
BWD_KERNELS = ["bwd_scores", "bwd_dst_main", "bwd_dst_merge", "bwd_src_main", "bwd_src_merge",
               "da_partial", "da_final"]


def parse_args(argv=None):
    p = argparse.ArgumentParser()
    p.add_argument("--gpus", type=int, default=1)
    p.add_argument("--steps", type=int, default=100)
    p.add_argument("--warmup", type=int, default=10)
    p.add_argument("--config", type=int, default=DEFAULT_CONFIG)
    p.add_argument("--impl", choices=["gnnagg", "reference"], default="gnnagg")
    p.add_argument("--op", choices=["gat", "gatv2", "transformer", "gcn", "max"], default="gat",
                   help="gat: fused GAT attention aggregation (the headline); "
                        "gcn: SpMM-family propagation A~ x with the symmetric normalisation; "
                        "max: max neighbourhood reduction with its winners; "
                        "gatv2: GATv2 attention (xl = h, xr a second seeded feature array); "
                        "transformer: graph-transformer attention (q = h, key and val seeded)")
    p.add_argument("--no-cpu-baseline", action="store_true")
    p.add_argument("--no-e2e", action="store_true")
    p.add_argument("--cpu-budget-s", type=float, default=12.0,
                   help="CPU seconds for the oracle baseline sample")
    p.add_argument("--no-sub", action="store_true",
                   help="skip the compact lines of the other power-law workloads")
    p.add_argument("--sub", default=None,
                   help="comma-separated workload indices for the compact lines "
                        "(default: 3,4,6 with the default workload, none otherwise)")
    p.add_argument("--sub-steps", type=int, default=10,
                   help="timed steps of each compact line")
    return p.parse_args(argv)


# ---- bytes model (algorithmic, compulsory traffic) -----------------------------

def algorithmic_bytes(n, e, H, D, s):
    """Per-launch algorithmic bytes of the main kernels.

    idx: CSR or CSC pointers + indices; gathered rows: one H*D row of s-byte
    elements per edge; node rows: H*D per node.  Forward: indices, gathered
    h_j, out written, lse written.  Backward, destination side: CSR indices,
    gathered h_j, dout_i and h_i read.  Source side: CSC indices, gathered
    dout_i, h_j read, dh_j written.  The per-edge gather of the 16-byte
    destination statistics in the source-side pass is extra traffic, not
    counted here (reported separately as stats_bytes).  The per-node score
    pre-pass of the forward call reads h once and writes two float [N][H]
    arrays; the backward of a step reuses them."""
    idx = 4 * (n + 1) + 4 * e
    gath = s * e * H * D
    row = s * n * H * D
    return {
        "scores": row + 8 * n * H,
        "fwd_main": idx + gath + row + 4 * n * H,
        "bwd_dst_main": idx + gath + 2 * row,
        "bwd_src_main": idx + gath + 2 * row,
        "stats_bytes": 16 * e * H,
    }


def workload_config(w, rp, ci, world):
    """The `config` object of the JSON line, the same for both arms: the
    workload's name and sizes, its degree extremes and the L2 protocol."""
    n, e = len(rp) - 1, len(ci)
    s = 4 if w.dtype == "f32" else 2
    feat_mb = n * w.H * w.D * s / 1e6
    return {"workload": w.name, "n_nodes": n, "n_edges": e, "H": w.H, "D": w.D,
            "feature_dtype": w.dtype,
            "max_in_degree": int(np.diff(rp).max(initial=0)),
            "max_out_degree": int(np.bincount(ci, minlength=n).max(initial=0)) if e else 0,
            "l2": f"flushed before every timed GPU step (a write of twice the L2 size); "
                  f"feature matrix {feat_mb:.0f} MB",
            "parallelism": "replicas" if world > 1 else "single GPU"}


# ---- clocks during the timed region ------------------------------------------------

class ClockSampler:
    FIELDS = ("clocks.sm,clocks.max.sm,power.draw,clocks_event_reasons.active,"
              "clocks_event_reasons.hw_slowdown,clocks_event_reasons.hw_thermal_slowdown,"
              "clocks_event_reasons.sw_thermal_slowdown,clocks_event_reasons.sw_power_cap")

    def __init__(self, gpu_index):
        self.gpu = gpu_index
        self.proc = None
        self.lines = []

    def start(self):
        try:
            self.proc = subprocess.Popen(
                ["nvidia-smi", "-i", str(self.gpu), f"--query-gpu={self.FIELDS}",
                 "--format=csv,noheader,nounits", "-lms", "50"],
                stdout=subprocess.PIPE, stderr=subprocess.DEVNULL, text=True)
            self.reader = threading.Thread(target=self._read, daemon=True)
            self.reader.start()
        except OSError:
            self.proc = None

    def _read(self):
        for line in self.proc.stdout:
            self.lines.append(line.strip())

    def stop(self):
        if self.proc is None:
            return None
        self.proc.terminate()
        try:
            self.proc.wait(timeout=5)
        except subprocess.TimeoutExpired:
            self.proc.kill()
        self.reader.join(timeout=2)
        sm, mx, reasons = [], [], set()
        names = ["hw_slowdown", "hw_thermal_slowdown", "sw_thermal_slowdown", "sw_power_cap"]
        for ln in self.lines:
            parts = [x.strip() for x in ln.split(",")]
            if len(parts) < 8:
                continue
            try:
                sm.append(float(parts[0]))
                mx.append(float(parts[1]))
            except ValueError:
                continue
            for nm, val in zip(names, parts[4:8]):
                if val.lower().startswith("active"):
                    reasons.add(nm)
        if not sm:
            return {"sm_mhz": None, "sm_max_mhz": None, "reasons": [], "samples": 0}
        return {"sm_mhz": statistics.median(sm), "sm_max_mhz": max(mx),
                "reasons": sorted(reasons), "samples": len(sm)}


# ---- workload ---------------------------------------------------------------------

def load_workload(idx):
    import workload
    w = workload.CONFIGS[idx]
    rp, ci = workload.make_graph(w)
    h, a_s, a_d, dout = workload.make_features(w, len(rp) - 1)
    return w, rp, ci, h, a_s, a_d, dout


# what the oracle's threads run: the forward and the destination side of the
# backward are split over nodes; the source-side scatter of the backward runs
# on one thread in edge order (deterministic by construction)
ORACLE_THREADS = ("forward and backward destination side on all threads (OpenMP over "
                  "nodes); backward source-side scatter on one thread")


def cpu_sample(rp, ci, frac_edges):
    """The subgraph of the first m destination rows (all N nodes kept), with
    about frac_edges of the edges: a prefix of the CSR."""
    e_target = max(1, int(len(ci) * frac_edges))
    m = int(np.searchsorted(rp, e_target, side="left"))
    m = max(1, min(m, len(rp) - 1))
    rp2 = rp.copy()
    rp2[m + 1:] = rp[m]
    return rp2, ci[:rp[m]].copy(), m


def time_oracle(rp, ci, h, a_s, a_d, dout, slope):
    import oracle
    t0 = time.perf_counter()
    oracle.forward(rp, ci, h, a_s, a_d, slope)
    oracle.backward(rp, ci, h, a_s, a_d, slope, dout)
    return time.perf_counter() - t0


def oracle_sample_rate(w, rp, ci, h, a_s, a_d, dout, budget_s, max_reps=10):
    """Oracle throughput on a bounded sample: a probe on 2% of the edges sizes
    a prefix subgraph that takes about budget_s seconds; when the whole graph
    takes less, it is timed several times (at most max_reps) within the
    budget and the rate is over all of them."""
    probe_rp, probe_ci, _ = cpu_sample(rp, ci, 0.02)
    t_probe = time_oracle(probe_rp, probe_ci, h, a_s, a_d, dout, w.slope)
    frac = min(1.0, 0.02 * budget_s / max(t_probe, 1e-3))
    srp, sci, m = cpu_sample(rp, ci, frac)
    t = time_oracle(srp, sci, h, a_s, a_d, dout, w.slope)
    reps = 1
    while reps < max_reps and t * (reps + 1) / reps <= budget_s:
        t += time_oracle(srp, sci, h, a_s, a_d, dout, w.slope)
        reps += 1
    sample = (f"destinations 0..{m - 1} of {len(rp) - 1} with their {len(sci)} in-edges "
              f"({100.0 * len(sci) / len(ci):.1f}% of E), all N nodes; fp64 forward + "
              f"backward, {reps} run(s), {t:.2f} s; {ORACLE_THREADS}")
    return len(sci) * w.H * reps / t / 1e9, sample


def oracle_baseline(w, rp, ci, h, a_s, a_d, dout, budget_s, one_core=False):
    """The oracle on all host cores; with one_core also on one core (a
    smaller sample, half the budget)."""
    import oracle
    value, sample = oracle_sample_rate(w, rp, ci, h, a_s, a_d, dout, budget_s)
    res = {"value": value, "unit": UNIT, "cores": oracle.num_threads(), "kind": "oracle",
           "sample": sample}
    if one_core:
        n_all = oracle.num_threads()
        oracle.set_threads(1)
        try:
            v1, s1 = oracle_sample_rate(w, rp, ci, h, a_s, a_d, dout, budget_s / 2)
        finally:
            oracle.set_threads(n_all)
        res["one_core"] = {"value": v1, "unit": UNIT, "cores": 1, "sample": s1}
    return res


# ---- reference arm: the oracle on the host ------------------------------------------

def run_reference(args, rank, world):
    if rank != 0:
        return 0
    import oracle
    w, rp, ci, h, a_s, a_d, dout = load_workload(args.config)
    # size each step so that warmup + steps fit in about three minutes
    per_step = 180.0 / max(1, args.steps + args.warmup)
    probe_rp, probe_ci, _ = cpu_sample(rp, ci, 0.02)
    t_probe = time_oracle(probe_rp, probe_ci, h, a_s, a_d, dout, w.slope)
    frac = min(1.0, 0.02 * per_step / max(t_probe, 1e-3))
    srp, sci, m = cpu_sample(rp, ci, frac)
    for _ in range(args.warmup):
        time_oracle(srp, sci, h, a_s, a_d, dout, w.slope)
    t = 0.0
    for _ in range(args.steps):
        t += time_oracle(srp, sci, h, a_s, a_d, dout, w.slope)
    units = len(sci) * w.H
    value = units * args.steps / t / 1e9
    sample = (f"destinations 0..{m - 1} of {len(rp) - 1} with their {len(sci)} in-edges "
              f"({100.0 * len(sci) / len(ci):.1f}% of E) per step, all N nodes; {ORACLE_THREADS}")
    line = {"metric": METRIC, "value": value, "unit": UNIT, "n_gpus": args.gpus,
            "steps": args.steps, "warmup": args.warmup, "ms_per_step": 1e3 * t / args.steps,
            "higher_is_better": True, "scaling": "weak", "vs_baseline": None, "dtype": "f64",
            "data": "synthetic", "impl": "reference",
            "config": workload_config(w, rp, ci, world),
            "cpu_baseline": {"value": value, "unit": UNIT, "kind": "oracle",
                             "cores": oracle.num_threads(), "sample": sample},
            "e2e": {"value": value, "unit": UNIT, "h2d_bytes_per_step": 0,
                    "d2h_bytes_per_step": 0}}
    print(json.dumps(line), flush=True)
    return 0


# ---- the CUDA path ------------------------------------------------------------------

def source_hash(paths):
    h = hashlib.sha256()
    for p in paths:
        with open(p, "rb") as f:
            h.update(f.read())
    return h.hexdigest()[:16]


def measured_traffic(workload_name, kernel):
    """Per-launch DRAM bytes of `kernel` from the committed ncu summary, if its
    kernel source is unchanged since the capture; else None."""
    entry = measured_entry(workload_name, kernel)
    return entry["bytes_per_launch"] if entry else None


def measured_entry(workload_name, kernel):
    """The committed ncu record of `kernel` (bytes_per_launch, l2_hit_pct),
    if its kernel source is unchanged since the capture; else None."""
    path = os.path.join(ROOT, "profiles", "traffic.json")
    if not os.path.exists(path):
        return None
    try:
        with open(path) as f:
            rec = json.load(f)
        entry = rec.get(workload_name, {}).get(kernel)
        if not entry:
            return None
        srcs = [os.path.join(ROOT, p) for p in entry["sources"]]
        if source_hash(srcs) != entry["source_hash"]:
            return None
        return entry
    except (OSError, ValueError, KeyError):
        return None


def peaks():
    path = os.path.join(ROOT, "MEASURED_PEAKS.json")
    try:
        with open(path) as f:
            p = json.load(f)
        return float(p["hbm_gbs"]), "measured"
    except (OSError, ValueError, KeyError):
        return 6800.0, "fallback"


class L2Flush:
    """Run between timed steps, outside the timed region: writes a buffer
    twice the size of L2, so that a step starts with none of its own data in
    L2.  Harness memory: allocated before the peak-memory baseline."""

    def __init__(self, dev):
        import torch
        l2 = torch.cuda.get_device_properties(dev).L2_cache_size
        self.w = torch.empty(max(2 * l2, 256 << 20), dtype=torch.uint8, device=dev)

    def __call__(self):
        self.w.zero_()

    def describe(self):
        return f"flushed before every step ({self.w.numel() >> 20} MiB write)"


def max_over_ranks(values, world, device):
    """Each value's maximum over the ranks (a job is as slow as its slowest
    replica); the identity on one rank."""
    values = [float(v) for v in values]
    if world <= 1:
        return values
    import torch
    import torch.distributed as dist
    t = torch.tensor(values, dtype=torch.float64, device=device)
    dist.all_reduce(t, op=dist.ReduceOp.MAX)
    return [float(x) for x in t]


def job_rate(units_per_rank, world, ms):
    """Whole-job throughput in G units/s: every rank processed units_per_rank
    in at most ms milliseconds."""
    return world * units_per_rank / (ms * 1e-3) / 1e9


class GatSession:
    """One workload on the device: inputs resident, graph prepared once, outputs
    and one workspace shared by the forward and the backward call of a step."""

    def __init__(self, idx, dev):
        import torch
        import graph_neural_network_gb300 as gnn
        from graph_neural_network_gb300 import _native
        self.torch, self.gnn, self.native = torch, gnn, _native
        self.dev = dev
        w, rp, ci, h_np, a_s_np, a_d_np, dout_np = load_workload(idx)
        self.w, self.rp, self.ci = w, rp, ci
        self.host = (h_np, a_s_np, a_d_np, dout_np)
        self.n, self.e, self.H, self.D = len(rp) - 1, len(ci), w.H, w.D
        self.s = 4 if w.dtype == "f32" else 2
        self.tdt = torch.float32 if w.dtype == "f32" else torch.bfloat16

        def dev_feat(x):
            x = np.ascontiguousarray(x)
            t = torch.from_numpy(x.view(np.int16) if w.dtype == "bf16" else x).to(dev)
            return t.view(torch.bfloat16) if w.dtype == "bf16" else t

        self.rp_d = torch.from_numpy(rp).to(dev)
        self.ci_d = torch.from_numpy(ci).to(dev)
        self.h = dev_feat(h_np)
        self.dout = dev_feat(dout_np)
        self.a_s = torch.from_numpy(a_s_np).to(dev)
        self.a_d = torch.from_numpy(a_d_np).to(dev)

    def prepare(self):
        torch, gnn = self.torch, self.gnn
        n, H, D, dev = self.n, self.H, self.D, self.dev
        torch.cuda.synchronize()
        t0 = time.perf_counter()
        self.g = gnn.Graph(self.rp_d, self.ci_d)
        self.prepare_ms = 1e3 * (time.perf_counter() - t0)
        self.st = self.g.stats()
        self.out = torch.empty_like(self.h)
        self.lse = torch.empty((n, H), dtype=torch.float32, device=dev)
        self.dh = torch.empty_like(self.h)
        self.da_s = torch.empty((H, D), dtype=torch.float32, device=dev)
        self.da_d = torch.empty((H, D), dtype=torch.float32, device=dev)
        self.ws = self.g.workspace(H, D, self.tdt)
        self.lib = self.native.load()
        self.dt_code = self.native.F32 if self.w.dtype == "f32" else self.native.BF16
        self.stream = torch.cuda.current_stream(dev)
        self.sp = ctypes.c_void_p(self.stream.cuda_stream)

    @staticmethod
    def ptr(t):
        return ctypes.c_void_p(t.data_ptr())

    def fwd(self, fe=None, sp=None):
        p = self.ptr
        rc = self.lib.gat_agg_forward_timed(
            self.g.handle, self.H, self.D, self.dt_code, p(self.h), p(self.a_s), p(self.a_d),
            self.w.slope, p(self.out), p(self.lse), p(self.ws), self.ws.numel(),
            sp if sp is not None else self.sp, fe, FWD_EVENTS if fe is not None else 0)
        self.native.check(rc, "forward")

    # a step passes one workspace to both calls, so the backward takes the
    # per-node scores the forward left there
    def bwd(self, be=None, sp=None):
        p = self.ptr
        rc = self.lib.gat_agg_backward_reuse(
            self.g.handle, self.H, self.D, self.dt_code, p(self.h), p(self.a_s), p(self.a_d),
            self.w.slope, p(self.lse), p(self.dout), p(self.dh), p(self.da_s), p(self.da_d),
            p(self.ws), self.ws.numel(), sp if sp is not None else self.sp, be,
            BWD_EVENTS if be is not None else 0)
        self.native.check(rc, "backward")

    def step(self, fe=None, be=None, sp=None):
        self.fwd(fe, sp)
        self.bwd(be, sp)

    def check(self):
        self.torch.cuda.synchronize()
        self.gnn.check_device_error(self.g)

    def timed_steps(self, K, flush):
        """K flushed steps with three events each (start, between the calls,
        end): mean forward and backward ms and the per-step totals."""
        torch = self.torch
        tev = [[torch.cuda.Event(enable_timing=True) for _ in range(3)] for _ in range(K)]
        for k in range(K):
            flush()  # outside the timed events
            tev[k][0].record(self.stream)
            self.fwd()
            tev[k][1].record(self.stream)
            self.bwd()
            tev[k][2].record(self.stream)
        torch.cuda.synchronize()
        tf = [a.elapsed_time(b) for a, b, _ in tev]
        tb = [b.elapsed_time(c) for _, b, c in tev]
        return sum(tf) / K, sum(tb) / K, [x + y for x, y in zip(tf, tb)]

    def kernel_times(self, K, flush):
        """Mean per-kernel ms over K flushed steps run through the timed API,
        whose caller events sit between the kernels."""
        torch = self.torch

        def make_events(k):
            evs = [torch.cuda.Event(enable_timing=True) for _ in range(k)]
            for ev in evs:
                ev.record(self.stream)  # creates the underlying event
            arr = (ctypes.c_void_p * k)(*[ev.cuda_event for ev in evs])
            return evs, arr

        fev = [make_events(FWD_EVENTS) for _ in range(K)]
        bev = [make_events(BWD_EVENTS) for _ in range(K)]
        for k in range(K):
            flush()
            self.step(fev[k][1], bev[k][1])
        self.check()
        kern = {name: 0.0 for name in FWD_KERNELS + BWD_KERNELS}
        for k in range(K):
            fe, be = fev[k][0], bev[k][0]
            for i, name in enumerate(FWD_KERNELS):
                kern[name] += fe[i].elapsed_time(fe[i + 1])
            for i, name in enumerate(BWD_KERNELS):
                kern[name] += be[i].elapsed_time(be[i + 1])
        return {k: v / K for k, v in kern.items()}

    def pass_fracs(self, t_fwd, t_bwd, peak):
        """Forward and backward call roofline fractions: the algorithmic bytes
        of the call's kernels (forward: score pre-pass + main kernel; backward:
        both main passes) over the call's event time."""
        ab = algorithmic_bytes(self.n, self.e, self.H, self.D, self.s)
        b_fwd = ab["scores"] + ab["fwd_main"]
        b_bwd = ab["bwd_dst_main"] + ab["bwd_src_main"]
        return (b_fwd / (t_fwd * 1e-3) / 1e9 / peak, b_bwd / (t_bwd * 1e-3) / 1e9 / peak,
                b_fwd, b_bwd)

    def kernel_fracs(self, kern, peak):
        ab = algorithmic_bytes(self.n, self.e, self.H, self.D, self.s)
        fr = {k: ab[k] / (kern[k] * 1e-3) / 1e9 / peak
              for k in ("fwd_main", "bwd_dst_main", "bwd_src_main") if kern[k] > 0}
        if kern["fwd_scores"] > 0:  # the backward reuses these scores: no bwd_scores kernel
            fr["fwd_scores"] = ab["scores"] / (kern["fwd_scores"] * 1e-3) / 1e9 / peak
        return fr

    def dram(self, kern, peak):
        """Real DRAM rate of each main kernel from its committed ncu record
        (bytes per launch over its event time), where the record matches the
        kernel sources."""
        res = {}
        for k in ("fwd_main", "bwd_dst_main", "bwd_src_main"):
            rec = measured_entry(self.w.name, k)
            if rec and kern[k] > 0:
                gbs = rec["bytes_per_launch"] / (kern[k] * 1e-3) / 1e9
                res[k] = {"traffic": rec["bytes_per_launch"], "dram_gbs": gbs,
                          "dram_frac": gbs / peak, "l2_hit_pct": rec.get("l2_hit_pct")}
        return res

    def launches_per_step(self):
        st = self.st
        # forward: scores, main, hub merge; backward (scores reused): two main
        # kernels and their hub merges, two attention-gradient kernels
        return (2 + (st["csr"]["hubs"] > 0)) + (1 + (st["csr"]["hubs"] > 0)) + \
            (1 + (st["csc"]["hubs"] > 0)) + 2

    def release(self):
        for name in ("g", "out", "lse", "dh", "da_s", "da_d", "ws", "h", "dout", "a_s", "a_d",
                     "rp_d", "ci_d"):
            if hasattr(self, name):
                delattr(self, name)
        self.torch.cuda.synchronize()
        self.torch.cuda.empty_cache()


def power_law_line(idx, dev, flush, steps, warmup, peak):
    """A compact figure of one more workload: K flushed steps, the per-kernel
    times, and the forward / backward call roofline fractions."""
    S = GatSession(idx, dev)
    S.prepare()
    for _ in range(max(3, warmup)):
        flush()
        S.step()
    S.check()
    t_fwd, t_bwd, per_step = S.timed_steps(steps, flush)
    S.check()
    kern = S.kernel_times(min(steps, 10), flush)
    ffr, bfr, b_fwd, b_bwd = S.pass_fracs(t_fwd, t_bwd, peak)
    units = S.e * S.H
    res = {"workload": S.w.name, "n_nodes": S.n, "n_edges": S.e, "H": S.H, "D": S.D,
           "feature_dtype": S.w.dtype, "steps": steps,
           "value": units / ((t_fwd + t_bwd) * 1e-3) / 1e9, "fwd_value": units / (t_fwd * 1e-3) / 1e9,
           "ms_per_step": t_fwd + t_bwd, "ms_per_step_median": float(np.median(per_step)),
           "fwd_ms": t_fwd, "bwd_ms": t_bwd, "fwd_frac": ffr, "bwd_frac": bfr,
           "algorithmic_bytes_fwd": b_fwd, "algorithmic_bytes_bwd": b_bwd,
           "kernels_ms": {k: kern[k] for k in ("fwd_scores", "fwd_main", "bwd_dst_main",
                                                 "bwd_src_main")},
           "kernel_hbm_frac": S.kernel_fracs(kern, peak), "prepare_ms": S.prepare_ms}
    dram = S.dram(kern, peak)
    if dram:
        res["dram"] = dram
    S.release()
    return res


def run_gnnagg(args, rank, world):
    import torch
    import torch.distributed as dist
    import graph_neural_network_gb300 as gnn
    from graph_neural_network_gb300 import _native

    dev = torch.device("cuda", int(os.environ.get("LOCAL_RANK", "0")))
    torch.cuda.set_device(dev)
    S = GatSession(args.config, dev)
    w, n, e, H, D = S.w, S.n, S.e, S.H, S.D
    flush = L2Flush(dev)  # harness memory, not counted in peak_mem_gb
    torch.cuda.synchronize()
    torch.cuda.reset_peak_memory_stats(dev)
    mem0 = torch.cuda.memory_allocated(dev)
    S.prepare()
    g, stream = S.g, S.stream

    for _ in range(max(3, args.warmup)):
        flush()
        S.step()
    S.check()
    peak_mem = torch.cuda.max_memory_allocated(dev) - mem0

    # the timed steps carry three events each (start, between the calls, end);
    # the per-kernel events of the timed API go on a separate pass below, so
    # that their own recording gaps stay out of the step time
    K = args.steps
    visible = os.environ.get("CUDA_VISIBLE_DEVICES")
    sampler = ClockSampler(visible.split(",")[dev.index].strip() if visible else dev.index)
    if world > 1:
        dist.barrier()
    torch.cuda.synchronize()
    sampler.start()
    time.sleep(0.2)
    wall0 = time.perf_counter()
    t_fwd, t_bwd, per_step = S.timed_steps(K, flush)
    wall = time.perf_counter() - wall0
    if world > 1:
        dist.barrier()
    clocks = sampler.stop()
    S.check()

    # per-kernel times: the same flushed steps again, with the timed API's
    # events between kernels
    Ki = min(K, 50)
    kern = S.kernel_times(Ki, flush)

    # secondary figure: the same steps back to back with no flush (warm L2)
    Kw = min(K, 50)
    wev = [(torch.cuda.Event(enable_timing=True), torch.cuda.Event(enable_timing=True))
           for _ in range(Kw)]
    for a, b in wev:
        a.record(stream)
        S.step()
        b.record(stream)
    S.check()
    (warm_ms,) = max_over_ranks([sum(a.elapsed_time(b) for a, b in wev) / Kw], world, dev)

    # secondary figure: the same flushed step replayed from a CUDA graph of
    # the two calls (no host launch path between kernels)
    gs = torch.cuda.Stream(dev)
    spg = ctypes.c_void_p(gs.cuda_stream)
    gs.wait_stream(stream)
    with torch.cuda.stream(gs):
        S.step(sp=spg)  # a warm-up on the capture stream
    stream.wait_stream(gs)
    torch.cuda.synchronize()
    cg = torch.cuda.CUDAGraph()
    with torch.cuda.graph(cg, stream=gs):
        S.step(sp=spg)
    Kg = min(K, 50)
    gev = [(torch.cuda.Event(enable_timing=True), torch.cuda.Event(enable_timing=True))
           for _ in range(Kg)]
    for a, b in gev:
        flush()
        a.record(stream)
        cg.replay()
        b.record(stream)
    S.check()
    (graph_ms,) = max_over_ranks([sum(a.elapsed_time(b) for a, b in gev) / Kg], world, dev)
    del cg
    ms_step, t_fwd, t_bwd = max_over_ranks([t_fwd + t_bwd, t_fwd, t_bwd], world, dev)
    units = e * H
    value = job_rate(units, world, ms_step)
    fwd_value = job_rate(units, world, t_fwd)

    # roofline of the dominant kernel
    ab = algorithmic_bytes(n, e, H, D, S.s)
    main = {k: kern[k] for k in ("fwd_main", "bwd_dst_main", "bwd_src_main")}
    dom = max(main, key=main.get)
    peak, peak_kind = peaks()
    achieved = ab[dom] / (kern[dom] * 1e-3) / 1e9
    dram = S.dram(kern, peak)
    rec = dram.get(dom)
    roofline = {"bound": "hbm", "kernel": dom, "achieved": achieved, "peak": peak,
                "unit": "GB/s", "frac": achieved / peak,
                "traffic": rec["traffic"] if rec else None,
                "algorithmic_bytes": ab[dom], "peak_source": peak_kind}
    if rec:
        # real DRAM rate of the same kernel: ncu bytes per launch over its event time
        roofline["dram_gbs"] = rec["dram_gbs"]
        roofline["dram_frac"] = rec["dram_frac"]
        if rec.get("l2_hit_pct") is not None:
            roofline["l2_hit_pct"] = rec["l2_hit_pct"]
    step_bytes = ab["fwd_main"] + ab["bwd_dst_main"] + ab["bwd_src_main"] + ab["scores"]
    ffr, bfr, _, _ = S.pass_fracs(t_fwd, t_bwd, peak)
    io_bytes = sum(t.numel() * t.element_size()
                   for t in (S.rp_d, S.ci_d, S.h, S.dout, S.a_s, S.a_d, S.out, S.lse, S.dh,
                             S.da_s, S.da_d))

    line = {"metric": METRIC, "value": value, "unit": UNIT, "n_gpus": world, "steps": K,
            "warmup": args.warmup, "ms_per_step": ms_step, "higher_is_better": True,
            # arithmetic type: every kernel accumulates in float32 (bf16 rows are
            # widened as they are loaded); the storage type is config.feature_dtype
            "scaling": "weak", "vs_baseline": None, "dtype": "f32", "data": "synthetic",
            "config": workload_config(w, S.rp, S.ci, world),
            "fwd_value": fwd_value, "fwd_ms": t_fwd, "bwd_ms": t_bwd,
            # call-level fractions of the HBM roofline (algorithmic bytes of the
            # call's kernels over the call's event time, of the measured peak)
            "fwd_frac": ffr, "bwd_frac": bfr,
            "ms_per_step_median": float(np.median(per_step)),
            "warm": {"ms_per_step": warm_ms, "value": job_rate(units, world, warm_ms),
                     "steps": Kw, "l2": "not flushed between steps"},
            "cuda_graph": {"ms_per_step": graph_ms, "value": job_rate(units, world, graph_ms),
                           "steps": Kg, "l2": "flushed before every step",
                           "what": "the forward and backward calls captured once, replayed"},
            "kernels_ms": kern, "kernel_hbm_frac": S.kernel_fracs(kern, peak),
            "roofline": roofline,
            "dram": dram,
            "step_roofline": {"achieved": step_bytes / (ms_step * 1e-3) / 1e9, "peak": peak,
                              "unit": "GB/s", "frac": step_bytes / (ms_step * 1e-3) / 1e9 / peak},
            "gpu_launches": S.launches_per_step() * K,
            "prepare_ms": S.prepare_ms, "peak_mem_gb": peak_mem / 1e9,
            "memory_gb": {"graph_buffer": g.buffer.numel() / 1e9, "workspace": S.ws.numel() / 1e9,
                          "inputs_outputs": io_bytes / 1e9,
                          "peak_above_inputs": peak_mem / 1e9,
                          "not_counted": "the L2-flush buffer and the 16 MiB array of the "
                                         "allocation-free forward (not loaded by this run)"},
            "l2_flush": flush.describe(),
            "clocks": clocks, "wall_s": wall}

    if not args.no_e2e:
        line["e2e"] = e2e(args, g, w, S.h, S.dout, S.a_s, S.a_d, S.out, S.lse, S.dh, S.da_s,
                          S.da_d, S.ws, world, dev, units)
    h_np, a_s_np, a_d_np, dout_np = S.host
    rp, ci = S.rp, S.ci
    S.release()
    del S, g
    if rank == 0 and world == 1 and not args.no_cpu_baseline:
        line["cpu_baseline"] = oracle_baseline(w, rp, ci, h_np, a_s_np, a_d_np, dout_np,
                                               args.cpu_budget_s, one_core=args.config <= 2)
    del h_np, a_s_np, a_d_np, dout_np
    subs = sub_configs(args)
    if subs:
        # the other power-law workloads (and the reordered R-MAT run), compact
        line["power_law"] = [power_law_line(i, dev, flush, args.sub_steps, 3, peak)
                             for i in subs]
    if rank == 0:
        print(json.dumps(line), flush=True)
    return 0


def sub_configs(args):
    if args.no_sub:
        return []
    if args.sub is not None:
        return [int(x) for x in args.sub.split(",") if x.strip()]
    return list(SUB_CONFIGS) if args.config == DEFAULT_CONFIG else []


def e2e(args, g, w, h, dout, a_s, a_d, out, lse, dh, da_s, da_d, ws, world, dev, units):
    """Same metric through the public API with host buffers: every step copies
    the step's inputs from pinned host memory and reads every result back.
    Steps are pipelined the way a training loop with a prefetching loader
    runs: inputs go up on two copy streams, results come back on two others
    and the kernels run on the compute stream, with two sets of device
    buffers so that step k + 1's upload and step k - 1's download overlap
    step k."""
    import torch
    import torch.distributed as dist
    import graph_neural_network_gb300 as gnn
    pin = lambda t: torch.empty(t.shape, dtype=t.dtype, pin_memory=True)
    h_host, d_host = pin(h), pin(dout)
    h_host.copy_(h)
    d_host.copy_(dout)
    as_host, ad_host = pin(a_s), pin(a_d)
    as_host.copy_(a_s)
    ad_host.copy_(a_d)
    o_host, l_host, dh_host = pin(out), pin(lse), pin(dh)
    das_host, dad_host = pin(da_s), pin(da_d)
    h2d = sum(t.numel() * t.element_size() for t in (h_host, d_host, as_host, ad_host))
    d2h = sum(t.numel() * t.element_size() for t in (o_host, l_host, dh_host, das_host, dad_host))
    comp = torch.cuda.current_stream(dev)
    # two upload and two download streams, so that both copies of a direction
    # can use separate copy engines
    s_h, s_d = torch.cuda.Stream(dev), torch.cuda.Stream(dev)
    s_o, s_g = torch.cuda.Stream(dev), torch.cuda.Stream(dev)
    names = ("h", "dout", "a_s", "a_d", "out", "lse", "dh", "da_s", "da_d")
    first = (h, dout, a_s, a_d, out, lse, dh, da_s, da_d)
    bufs = [dict(zip(names, first)), {n: torch.empty_like(t) for n, t in zip(names, first)}]
    ev = lambda: [torch.cuda.Event() for _ in range(2)]
    h_ready, d_ready, fwd_done, comp_done, o_done, g_done = ev(), ev(), ev(), ev(), ev(), ev()
    for e in comp_done + o_done + g_done:
        e.record(comp)

    def one(k):
        i = k % 2
        b = bufs[i]
        for st, ready, copies in ((s_h, h_ready, (("h", h_host), ("a_s", as_host),
                                                   ("a_d", ad_host))),
                                  (s_d, d_ready, (("dout", d_host),))):
            st.wait_event(comp_done[i])        # step k - 2 no longer reads these inputs
            with torch.cuda.stream(st):
                for name, src in copies:
                    b[name].copy_(src, non_blocking=True)
                ready[i].record(st)
        comp.wait_event(h_ready[i])
        comp.wait_event(o_done[i])             # step k - 2's results have left these buffers
        comp.wait_event(g_done[i])
        gnn.gat_forward(g, b["h"], b["a_s"], b["a_d"], w.slope, out=b["out"], lse=b["lse"],
                        ws=ws, stream=comp)
        fwd_done[i].record(comp)
        comp.wait_event(d_ready[i])            # dout arrived while the forward ran
        gnn.gat_backward(g, b["h"], b["a_s"], b["a_d"], w.slope, b["lse"], b["dout"],
                         dh=b["dh"], da_src=b["da_s"], da_dst=b["da_d"], ws=ws, stream=comp,
                         reuse_scores=True)
        comp_done[i].record(comp)
        for st, after, done, copies in ((s_o, fwd_done, o_done, ((o_host, "out"),
                                                                   (l_host, "lse"))),
                                        (s_g, comp_done, g_done, ((dh_host, "dh"),
                                                                   (das_host, "da_s"),
                                                                   (dad_host, "da_d")))):
            st.wait_event(after[i])            # out and lse leave while the backward runs
            with torch.cuda.stream(st):
                for dst, name in copies:
                    dst.copy_(b[name], non_blocking=True)
                done[i].record(st)

    for k in range(4):
        one(k)
    K = max(1, min(args.steps, 200))
    if world > 1:
        dist.barrier()
    torch.cuda.synchronize()
    e0 = torch.cuda.Event(enable_timing=True)
    e1 = torch.cuda.Event(enable_timing=True)
    e0.record(s_h)
    s_d.wait_event(e0)
    for k in range(K):
        one(k)
    s_g.wait_event(o_done[(K - 1) % 2])
    e1.record(s_g)
    torch.cuda.synchronize()
    (ms,) = max_over_ranks([e0.elapsed_time(e1) / K], world, dev)
    link = link_rates(bufs[0], ((h_host, "h"), (d_host, "dout")),
                      ((o_host, "out"), (dh_host, "dh")), s_h, s_o)
    # the step's copies cannot finish faster than the link moves them
    link["copy_bound_ms"] = (h2d + d2h) / (link["both_gbs"] * 1e6)
    return {"value": job_rate(units, world, ms), "unit": UNIT, "ms_per_step": ms,
            "steps": K, "h2d_bytes_per_step": h2d, "d2h_bytes_per_step": d2h,
            "host_link": link,
            "pipeline": "two upload, one compute and two download streams, two device buffer "
                        "sets; dout uploads during the forward, out and lse download during "
                        "the backward"}


def link_rates(b, ups, downs, s_up, s_down, reps=5):
    """Host link bandwidth in GB/s measured with the e2e buffers (pinned host
    memory, copy engines): uploads alone, downloads alone, and both directions
    at once on their own streams, each timed with events after a warm-up."""
    import torch

    def rate(do_up, do_down):
        nbytes = 0
        t0, t1 = torch.cuda.Event(enable_timing=True), torch.cuda.Event(enable_timing=True)
        for r in range(reps + 1):
            if r == 1:
                torch.cuda.synchronize()
                t0.record(s_up)
                s_down.wait_event(t0)
            if do_up:
                with torch.cuda.stream(s_up):
                    for src, name in ups:
                        b[name].copy_(src, non_blocking=True)
                        nbytes += src.numel() * src.element_size() if r else 0
            if do_down:
                with torch.cuda.stream(s_down):
                    for dst, name in downs:
                        dst.copy_(b[name], non_blocking=True)
                        nbytes += dst.numel() * dst.element_size() if r else 0
        done = torch.cuda.Event()
        done.record(s_down)
        s_up.wait_event(done)
        t1.record(s_up)
        torch.cuda.synchronize()
        return nbytes / (t0.elapsed_time(t1) * 1e6)

    return {"h2d_gbs": rate(True, False), "d2h_gbs": rate(False, True),
            "both_gbs": rate(True, True)}


def run_layer(args, rank, world):
    """The other aggregation families on the same workload (features [N, H*D]).
    gcn: a step is out = A~ x (CSR) plus dx = A~^T dout (cached CSC), norm
    "sym".  max: a step is (out, arg) = max over in-neighbours plus dx from
    arg and dout."""
    import torch
    import graph_neural_network_gb300 as gnn

    dev = torch.device("cuda", int(os.environ.get("LOCAL_RANK", "0")))
    torch.cuda.set_device(dev)
    w, rp, ci, h_np, _, _, dout_np = load_workload(args.config)
    n, e, F = len(rp) - 1, len(ci), w.H * w.D
    s = 4 if w.dtype == "f32" else 2

    def dev_feat(x):
        x = np.ascontiguousarray(x).reshape(n, F)
        t = torch.from_numpy(x.view(np.int16) if w.dtype == "bf16" else x).to(dev)
        return t.view(torch.bfloat16) if w.dtype == "bf16" else t

    g = gnn.Graph(torch.from_numpy(rp).to(dev), torch.from_numpy(ci).to(dev))
    x, dout = dev_feat(h_np), dev_feat(dout_np)
    out, dx = torch.empty_like(x), torch.empty_like(x)
    arg = torch.empty((n, F), dtype=torch.int32, device=dev)
    dtc = 0 if w.dtype == "f32" else 1
    units = e
    if args.op == "gatv2":
        import workload
        H, D = w.H, w.D
        xr_np = workload.normal_f32(w.seed, 5, (n, H, D), 1.0)
        if w.dtype == "bf16":
            xr_np = workload.f32_to_bf16_bits(xr_np)
        xl3, xr3, dout3 = x.view(n, H, D), dev_feat(xr_np).view(n, H, D), dout.view(n, H, D)
        att = torch.from_numpy(workload.normal_f32(w.seed, 2, (H, D), 0.1)).to(dev)
        lse = torch.empty((n, H), dtype=torch.float32, device=dev)
        dxr = torch.empty_like(xr3)
        datt = torch.empty((H, D), dtype=torch.float32, device=dev)
        ws = torch.empty(g._lib.gatv2_agg_workspace_bytes(g.handle, H, D, dtc),
                         dtype=torch.uint8, device=dev)
        out3, dx3 = out.view(n, H, D), dx.view(n, H, D)

        def fwd():
            gnn.gatv2_forward(g, xl3, xr3, att, w.slope, out=out3, lse=lse, ws=ws)

        def bwd():
            gnn.gatv2_backward(g, xl3, xr3, att, w.slope, lse, dout3, dxl=dx3, dxr=dxr,
                               datt=datt, ws=ws)
        idx = 4 * (n + 1) + 4 * e
        row = s * n * F
        b_fwd = idx + s * e * F + 2 * row + 4 * n * H            # xl_j gathered, xr_i, out, lse
        # pass 1: xl_j gathered, xr_i and dout_i read, dxr written; pass 2: xr_i and
        # dout_i gathered, xl_j read, dxl written
        b_bwd = 2 * idx + 3 * s * e * F + 5 * row
        units = e * H
        metric = ("GEdge*head/s fwd and fwd+bwd GATv2 attention aggregation; "
                  "achieved HBM GB/s vs roofline")
    elif args.op == "transformer":
        import workload
        H, D = w.H, w.D

        def seeded(stream_id):
            a = workload.normal_f32(w.seed, stream_id, (n, H, D), 1.0)
            return dev_feat(workload.f32_to_bf16_bits(a) if w.dtype == "bf16" else a).view(n, H, D)
        q3, k3, v3, dout3 = x.view(n, H, D), seeded(5), seeded(6), dout.view(n, H, D)
        lse = torch.empty((n, H), dtype=torch.float32, device=dev)
        dq3, dk3, dv3 = dx.view(n, H, D), torch.empty_like(k3), torch.empty_like(v3)
        out3 = out.view(n, H, D)
        ws = torch.empty(g._lib.transformer_agg_workspace_bytes(g.handle, H, D, dtc),
                         dtype=torch.uint8, device=dev)

        def fwd():
            gnn.transformer_forward(g, q3, k3, v3, out=out3, lse=lse, ws=ws)

        def bwd():
            gnn.transformer_backward(g, q3, k3, v3, lse, dout3, dq=dq3, dkey=dk3, dval=dv3,
                                     ws=ws)
        idx = 4 * (n + 1) + 4 * e
        row = s * n * F
        b_fwd = idx + 2 * s * e * F + 2 * row + 4 * n * H      # key_j, val_j gathered; q, out
        # pass 1: key_j, val_j gathered, q_i and dout_i read, dq written; pass 2: q_i
        # and dout_i gathered, key_j and val_j read, dkey and dval written
        b_bwd = 2 * idx + 4 * s * e * F + 7 * row
        units = e * H
        metric = ("GEdge*head/s fwd and fwd+bwd graph-transformer attention aggregation; "
                  "achieved HBM GB/s vs roofline")
    elif args.op == "gcn":
        ws = torch.empty(g._lib.gcn_agg_workspace_bytes(g.handle, F, dtc), dtype=torch.uint8,
                         device=dev)

        def fwd():
            gnn.gcn_forward(g, x, "sym", out=out, ws=ws)

        def bwd():
            gnn.gcn_backward(g, dout, "sym", dx=dx, ws=ws)
        idx = 4 * (n + 1) + 4 * e
        b_fwd = b_bwd = idx + s * e * F + s * n * F    # indices, gathered rows, written rows
        metric = "GEdge/s fwd and fwd+bwd GCN propagation (sym); achieved HBM GB/s vs roofline"
    else:
        ws = torch.empty(g._lib.reduce_agg_workspace_bytes(g.handle, F, dtc), dtype=torch.uint8,
                         device=dev)

        def fwd():
            gnn.reduce_forward(g, x, "max", out=out, arg=arg, ws=ws)

        def bwd():
            gnn.reduce_backward(g, arg, dout, dx=dx, ws=ws)
        b_fwd = 4 * (n + 1) + 4 * e + s * e * F + (s + 4) * n * F   # + out and arg written
        b_bwd = (4 + 2 * s) * n * F                                  # arg, dout read; dx written
        metric = "GEdge/s fwd and fwd+bwd max neighbourhood reduction; achieved HBM GB/s vs roofline"
    flush = L2Flush(dev)
    stream = torch.cuda.current_stream(dev)
    for _ in range(max(3, args.warmup)):
        flush()
        fwd()
        bwd()
    torch.cuda.synchronize()
    gnn.check_device_error(g)
    K = args.steps
    ev = [[torch.cuda.Event(enable_timing=True) for _ in range(3)] for _ in range(K)]
    sampler = ClockSampler(dev.index)
    sampler.start()
    time.sleep(0.2)
    for k in range(K):
        flush()
        ev[k][0].record(stream)
        fwd()
        ev[k][1].record(stream)
        bwd()
        ev[k][2].record(stream)
    torch.cuda.synchronize()
    clocks = sampler.stop()
    gnn.check_device_error(g)
    t_f = sum(a.elapsed_time(b) for a, b, _ in ev) / K
    t_b = sum(b.elapsed_time(c) for _, b, c in ev) / K
    median = float(np.median([a.elapsed_time(c) for a, _, c in ev]))
    # secondary figure: the same steps back to back with no flush (warm L2)
    Kw = min(K, 50)
    wev = [(torch.cuda.Event(enable_timing=True), torch.cuda.Event(enable_timing=True))
           for _ in range(Kw)]
    for a, b in wev:
        a.record(stream)
        fwd()
        bwd()
        b.record(stream)
    torch.cuda.synchronize()
    gnn.check_device_error(g)
    t_f, t_b, warm_ms = max_over_ranks(
        [t_f, t_b, sum(a.elapsed_time(b) for a, b in wev) / Kw], world, dev)
    peak, peak_kind = peaks()
    line = {"metric": metric, "op": args.op,
            "value": job_rate(units, world, t_f + t_b),
            "unit": "GEdge*head/s" if args.op in ("gatv2", "transformer") else "GEdge/s",
            "fwd_value": job_rate(units, world, t_f), "n_gpus": world,
            "steps": K, "warmup": args.warmup, "ms_per_step": t_f + t_b, "fwd_ms": t_f,
            "bwd_ms": t_b, "ms_per_step_median": median,
            "warm": {"ms_per_step": warm_ms, "value": job_rate(units, world, warm_ms),
                     "steps": Kw, "l2": "not flushed between steps"},
            "higher_is_better": True, "dtype": "f32", "data": "synthetic",
            "config": {"workload": w.name, "n_nodes": n, "n_edges": e, "F": F,
                       "feature_dtype": w.dtype,
                       "l2": flush.describe()},
            "roofline": {"bound": "hbm", "kernel": f"{args.op} forward / backward calls",
                         "achieved_fwd": b_fwd / (t_f * 1e-3) / 1e9,
                         "achieved_bwd": b_bwd / (t_b * 1e-3) / 1e9, "peak": peak,
                         "unit": "GB/s", "frac_fwd": b_fwd / (t_f * 1e-3) / 1e9 / peak,
                         "frac_bwd": b_bwd / (t_b * 1e-3) / 1e9 / peak,
                         "algorithmic_bytes_fwd": b_fwd, "algorithmic_bytes_bwd": b_bwd,
                         "peak_source": peak_kind},
            "clocks": clocks}
    if args.op == "max":
        # the atomic-free backward on the same steps: a masked gather over the
        # cached CSC (indices, the winners and dout rows of every out-edge's
        # destination, dx written)
        def bwd_ordered():
            gnn.reduce_backward(g, arg, dout, dx=dx, ws=ws, ordered=True)
        bwd_ordered()
        torch.cuda.synchronize()
        oev = [(torch.cuda.Event(enable_timing=True), torch.cuda.Event(enable_timing=True))
               for _ in range(K)]
        for a, b in oev:
            flush()
            a.record(stream)
            bwd_ordered()
            b.record(stream)
        torch.cuda.synchronize()
        gnn.check_device_error(g)
        (t_o,) = max_over_ranks([sum(a.elapsed_time(b) for a, b in oev) / K], world, dev)
        b_o = 4 * (n + 1) + 4 * e + (4 + s) * e * F + s * n * F
        line["bwd_ordered"] = {"ms": t_o, "vs_atomic": t_o / t_b, "algorithmic_bytes": b_o,
                               "frac": b_o / (t_o * 1e-3) / 1e9 / peak,
                               "what": "reduce_agg_backward_ordered: no atomics, bitwise "
                                       "reproducible"}
    if rank == 0:
        print(json.dumps(line), flush=True)
    return 0


def main(argv=None):
    args = parse_args(argv)
    world = int(os.environ.get("WORLD_SIZE", "1"))
    rank = int(os.environ.get("RANK", "0"))
    if args.impl == "reference":
        return run_reference(args, rank, world)
    if world > 1:
        import torch
        import torch.distributed as dist
        torch.cuda.set_device(int(os.environ.get("LOCAL_RANK", "0")))
        dist.init_process_group("nccl")
    try:
        if args.op != "gat":
            return run_layer(args, rank, world)
        return run_gnnagg(args, rank, world)
    finally:
        if world > 1:
            import torch.distributed as dist
            dist.destroy_process_group()


if __name__ == "__main__":
    sys.exit(main())
