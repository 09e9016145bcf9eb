"""Shared helpers of the GPU parity tests: move seeded inputs to the device,
run the CUDA path through the C-ABI binding, run the fp64 oracle on the same
inputs, and compare element by element.

Tolerance (per element, |gpu - oracle| <= bound):
    bound = atol + rtol * |oracle| + GAMMA * mag
  fp32 features: rtol 1e-4, atol 1e-5;  bf16 features: rtol 2e-2, atol 1e-5.
  mag is the oracle's sum of |terms| of that element and GAMMA = 32 * 2^-24:
  a float32 sum cannot be relatively accurate where its terms cancel, and the
  GPU's error is bounded by a small multiple of unit roundoff times mag.
  out and lse are held to the plain atol + rtol bound (strict); lse, a
  float32 statistic of exactly widened inputs, to the float32 tolerance for
  either feature type.  The GAT gradients also get the oracle's kink term:
  where an edge's z lies within float32 rounding of the LeakyReLU kink both
  derivatives are valid results, and the oracle reports how far each
  gradient element can move between them.  Every comparison counts the
  elements that needed the mag or the kink term (REPORT; written as JSON at
  the end of the session when the environment variable GNN_PARITY_REPORT
  names a file).
"""
from __future__ import annotations

import numpy as np
import torch

import oracle
import workload

U32 = 2.0 ** -24
GAMMA = 32 * U32
TOL = {"f32": (1e-4, 1e-5), "bf16": (2e-2, 1e-5)}


def to_device(x, dtype):
    x = np.ascontiguousarray(x)
    if dtype == "bf16":
        return torch.from_numpy(x.view(np.int16)).cuda().view(torch.bfloat16)
    return torch.from_numpy(x).cuda()


def to_f64(t):
    if t.dtype == torch.bfloat16:
        bits = t.contiguous().view(torch.int16).cpu().numpy().view(np.uint16)
        return workload.bf16_bits_to_f32(bits).astype(np.float64)
    return t.detach().cpu().numpy().astype(np.float64)


def make_case(row_ptr, col, H, D, dtype, seed, slope=0.2):
    n = len(row_ptr) - 1
    h = workload.normal_f32(seed, 1, (n, H, D), 1.0)
    dout = workload.normal_f32(seed, 4, (n, H, D), 1.0)
    a_s = workload.normal_f32(seed, 2, (H, D), 0.1)
    a_d = workload.normal_f32(seed, 3, (H, D), 0.1)
    if dtype == "bf16":
        h = workload.f32_to_bf16_bits(h)
        dout = workload.f32_to_bf16_bits(dout)
    return dict(row_ptr=np.asarray(row_ptr, np.int32), col=np.asarray(col, np.int32), h=h,
                dout=dout, a_src=a_s, a_dst=a_d, H=H, D=D, dtype=dtype, slope=slope)


def device_graph(case, tiling=None, stream=None):
    import graph_neural_network_gb300 as gnn
    rp = torch.from_numpy(case["row_ptr"]).cuda()
    ci = torch.from_numpy(case["col"]).cuda() if len(case["col"]) else \
        torch.zeros(0, dtype=torch.int32, device="cuda")
    t = None
    if tiling is not None:
        t = gnn.Tiling(*tiling)
    return gnn.Graph(rp, ci, t, stream=stream)


def run_gpu(case, tiling=None, backward=True, stream=None, graph=None, fetch=True):
    import graph_neural_network_gb300 as gnn
    g = graph if graph is not None else device_graph(case, tiling, stream)
    h = to_device(case["h"], case["dtype"])
    a_s = torch.from_numpy(case["a_src"]).cuda()
    a_d = torch.from_numpy(case["a_dst"]).cuda()
    out, lse = gnn.gat_forward(g, h, a_s, a_d, case["slope"], stream=stream)
    res = dict(graph=g, out_t=out, lse_t=lse)
    if backward:
        dout = to_device(case["dout"], case["dtype"])
        dh, da_s, da_d = gnn.gat_backward(g, h, a_s, a_d, case["slope"], lse, dout, stream=stream)
        res.update(dh_t=dh, da_src_t=da_s, da_dst_t=da_d)
    torch.cuda.synchronize()
    gnn.check_device_error(g)
    if not fetch:
        return res
    res["out"] = to_f64(out)
    res["lse"] = to_f64(lse)
    if backward:
        res["dh"] = to_f64(dh)
        res["da_src"] = to_f64(da_s)
        res["da_dst"] = to_f64(da_d)
    return res


def run_oracle(case, backward=True):
    f = oracle.forward(case["row_ptr"], case["col"], case["h"], case["a_src"], case["a_dst"],
                       case["slope"], with_mag=True)
    res = dict(out=f["out"], lse=f["lse"], out_mag=f["out_mag"])
    if backward:
        b = oracle.backward(case["row_ptr"], case["col"], case["h"], case["a_src"],
                            case["a_dst"], case["slope"], case["dout"], with_mag=True,
                            with_kink=True)
        res.update(dh=b["dh"], dh_mag=b["dh_mag"], da_src=b["da_src"], da_dst=b["da_dst"],
                   da_src_mag=b["da_src_mag"], da_dst_mag=b["da_dst_mag"],
                   dh_kink=b["dh_kink"], da_src_kink=b["da_src_kink"],
                   da_dst_kink=b["da_dst_kink"])
    return res


# Every comparison's accounting: elements compared, elements that pass only
# through the float32 summation term (GAMMA * mag), and the worst ratio of the
# error to the plain atol + rtol * |oracle| bound.
REPORT = []


def assert_close(gpu, ref, dtype, mag=None, what="", strict=False, kink=None):
    """Element-wise |gpu - oracle| <= atol + rtol |oracle| (+ GAMMA * mag)
    (+ kink).  kink: the oracle's per-element ambiguity from edges whose z lies
    within float32 rounding of the LeakyReLU kink, where either derivative is
    a valid result.  strict: no element may need the GAMMA * mag term.
    Returns the comparison's accounting (also appended to REPORT)."""
    gpu = np.asarray(gpu, np.float64)
    ref = np.asarray(ref, np.float64)
    assert gpu.shape == ref.shape, (what, gpu.shape, ref.shape)
    rtol, atol = TOL[dtype]
    base = atol + rtol * np.abs(np.where(np.isfinite(ref), ref, 0.0))
    plain = base + GAMMA * mag if mag is not None else base
    bound = plain + kink if kink is not None else plain
    same_inf = np.isinf(gpu) & np.isinf(ref) & (np.sign(gpu) == np.sign(ref))
    with np.errstate(invalid="ignore"):
        err = np.where(same_inf, 0.0, np.abs(gpu - ref))
    bad = ~(err <= bound)
    # what an element beyond the plain bound needed: the kink term alone (an
    # edge on the kink took the other derivative), else the summation term
    beyond = ~bad & (err > base)
    kink_only = beyond & (err <= base + kink) if kink is not None else np.zeros_like(beyond)
    mag_only = beyond & ~kink_only
    ratio = np.where(np.isnan(err), np.inf, err / base)
    stats = {"what": what, "n": int(err.size), "mag_only": int(mag_only.sum()),
             "kink_only": int(kink_only.sum()),
             "kink_elements": int((kink > 0).sum()) if kink is not None else 0,
             "worst_strict_ratio": float(ratio.max()) if ratio.size else 0.0}
    REPORT.append(stats)
    if bad.any():
        idx = np.argwhere(bad)[:5]
        worst = np.unravel_index(np.nanargmax(np.where(np.isnan(err), np.inf, err / bound)),
                                 err.shape)
        raise AssertionError(
            f"{what}: {int(bad.sum())} of {bad.size} elements outside tolerance; first at "
            f"{idx.tolist()}; worst {worst}: gpu {gpu[worst]!r} oracle {ref[worst]!r} "
            f"bound {bound[worst]!r}")
    if strict and stats["mag_only"]:
        raise AssertionError(f"{what}: {stats['mag_only']} of {err.size} elements pass only "
                             f"through the float32 summation term")
    return stats


def compare(gpu, ref, dtype, backward=True, what=""):
    assert_close(gpu["out"], ref["out"], dtype, ref.get("out_mag"), what + " out", strict=True)
    # lse is a float32 statistic of exactly widened inputs: float32 tolerance
    assert_close(gpu["lse"], ref["lse"], "f32", None, what + " lse", strict=True)
    if backward:
        for k in ("dh", "da_src", "da_dst"):
            assert_close(gpu[k], ref[k], dtype, ref.get(k + "_mag"), f"{what} {k}",
                         kink=ref.get(k + "_kink"))
