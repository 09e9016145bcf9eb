"""Checks that pin the fp64 oracle to things other than itself.

Each check takes an oracle object (the real one, or a build with a planted
mistake) and raises AssertionError when the oracle disagrees with:
  * a hand-derived worked example (tests/golden/worked_example.json),
  * a dense masked-softmax formulation in torch fp64 and its autograd,
  * central finite differences of L = sum(out * G) on fp64 inputs,
  * closed forms and invariants (alpha sums to 1, zero in-degree, single
    neighbour, equal scores = neighbour mean, slope 1 = shift invariance,
    Delta_i = dout_i . out_i, permutation equivariance).
"""
from __future__ import annotations

import json
import math
import os

import numpy as np
import torch

import workload

GOLDEN = os.path.join(os.path.dirname(os.path.abspath(__file__)), "golden")


# ---- small graphs -------------------------------------------------------------

def csr_from_lists(rows):
    row_ptr = np.zeros(len(rows) + 1, np.int32)
    for i, r in enumerate(rows):
        row_ptr[i + 1] = row_ptr[i] + len(r)
    col = np.array([j for r in rows for j in r], np.int32)
    return row_ptr, col


def irregular_graph(n=12, seed=5):
    """Hand-shaped graph: isolated nodes, a double edge, a hub, self-loops."""
    rng = np.random.default_rng(seed)
    rows = []
    for i in range(n):
        if i in (3, 7):
            rows.append([])                       # zero in-degree
        elif i == 0:
            rows.append(list(range(n)))           # hub: every node
        else:
            k = int(rng.integers(1, 5))
            r = sorted(set(rng.integers(0, n, size=k).tolist()))
            if i == 5:
                r = r + [r[-1]]                   # multi-edge
            rows.append(r)
    return csr_from_lists(rows)


def random_inputs(n, H, D, seed, dtype=np.float64, a_std=0.5):
    rng = np.random.default_rng(seed)
    h = rng.standard_normal((n, H, D)).astype(dtype)
    a_src = (a_std * rng.standard_normal((H, D))).astype(dtype)
    a_dst = (a_std * rng.standard_normal((H, D))).astype(dtype)
    dout = rng.standard_normal((n, H, D)).astype(dtype)
    return h, a_src, a_dst, dout


# ---- independent dense formulation ---------------------------------------------

def dense_torch(row_ptr, col, h, a_src, a_dst, slope, dout=None):
    """Dense masked softmax in torch fp64: logits[i, j] = LeakyReLU(s_dst[i] +
    s_src[j]) + log(multiplicity of j -> i); softmax over j per row; out = P @ h.
    With dout, also returns the autograd gradients of sum(out * dout)."""
    n = len(row_ptr) - 1
    cnt = np.zeros((n, n))
    for i in range(n):
        for j in col[row_ptr[i]:row_ptr[i + 1]]:
            cnt[i, j] += 1
    mask = torch.tensor(cnt > 0)
    logc = torch.tensor(np.log(np.where(cnt > 0, cnt, 1.0)))
    ht = torch.tensor(np.asarray(h, np.float64), requires_grad=True)
    at_s = torch.tensor(np.asarray(a_src, np.float64), requires_grad=True)
    at_d = torch.tensor(np.asarray(a_dst, np.float64), requires_grad=True)
    s_src = (ht * at_s[None]).sum(-1)                      # [n, H]
    s_dst = (ht * at_d[None]).sum(-1)
    logits = torch.nn.functional.leaky_relu(s_dst[:, None, :] + s_src[None, :, :], slope)
    logits = logits + logc[:, :, None]
    neg = torch.full_like(logits, -math.inf)
    logits = torch.where(mask[:, :, None], logits, neg)
    rows = torch.nonzero(mask.any(1)).flatten()
    P = torch.softmax(logits[rows], dim=1)                 # [r, n, H]
    out = torch.zeros_like(ht)
    out = out.index_copy(0, rows, torch.einsum("ijk,jkd->ikd", P, ht))
    lse = torch.full((n, h.shape[1]), -math.inf, dtype=torch.float64)
    lse[rows] = torch.logsumexp(logits[rows], dim=1).detach()
    res = dict(out=out.detach().numpy(), lse=lse.numpy())
    if dout is not None:
        loss = (out * torch.tensor(np.asarray(dout, np.float64))).sum()
        loss.backward()
        res.update(dh=ht.grad.numpy(), da_src=at_s.grad.numpy(), da_dst=at_d.grad.numpy())
    return res


def close(a, b, rtol, atol, what):
    a = np.asarray(a, np.float64)
    b = np.asarray(b, np.float64)
    assert a.shape == b.shape, (what, a.shape, b.shape)
    both_inf = np.isinf(a) & np.isinf(b) & (np.sign(a) == np.sign(b))
    with np.errstate(invalid="ignore"):
        err = np.where(both_inf, 0.0, np.abs(a - b))
    bad = ~(err <= atol + rtol * np.abs(b))
    assert not bad.any(), f"{what}: {int(bad.sum())} mismatches, max err {np.nanmax(err)}"


# ---- the pins -------------------------------------------------------------------

def pin_worked_example(o):
    with open(os.path.join(GOLDEN, "worked_example.json")) as f:
        fx = json.load(f)
    H, D = fx["H"], fx["D"]
    rp = np.array(fx["row_ptr"], np.int32)
    ci = np.array(fx["col_idx"], np.int32)
    h = np.array(fx["h"], np.float32).reshape(-1, H, D)
    dout = np.array(fx["dout"], np.float32).reshape(-1, H, D)
    a_src = np.array(fx["a_src"], np.float32).reshape(H, D)
    a_dst = np.array(fx["a_dst"], np.float32).reshape(H, D)
    ex = fx["expected"]
    f = o.forward(rp, ci, h, a_src, a_dst, fx["slope"])
    close(f["out"].reshape(-1, D), ex["out"], 1e-12, 1e-14, "worked out")
    lse_ex = [(-math.inf if v == "-inf" else v) for v in ex["lse"]]
    close(f["lse"].ravel(), lse_ex, 1e-12, 1e-14, "worked lse")
    st = o.node_stats(rp, ci, h, a_src, a_dst, fx["slope"], dout)
    close(st["delta"].ravel(), ex["delta"], 1e-12, 1e-14, "worked delta")
    close(st["ds_dst"].ravel(), ex["ds_dst"], 1e-12, 1e-14, "worked ds_dst")
    b = o.backward(rp, ci, h, a_src, a_dst, fx["slope"], dout)
    close(b["dh"].reshape(-1, D), ex["dh"], 1e-12, 1e-14, "worked dh")
    close(b["da_src"].ravel(), ex["da_src"], 1e-12, 1e-14, "worked da_src")
    close(b["da_dst"].ravel(), ex["da_dst"], 1e-12, 1e-14, "worked da_dst")


def pin_dense_forward_backward(o, seeds=(1, 2)):
    cases = [irregular_graph(12, 5)]
    cases.append(workload.erdos_renyi(64, 6.0, 11))
    for g_i, (rp, ci) in enumerate(cases):
        n = len(rp) - 1
        for s in seeds:
            h, a_s, a_d, dout = random_inputs(n, 2, 3, 100 * g_i + s)
            ref = dense_torch(rp, ci, h, a_s, a_d, 0.2, dout)
            f = o.forward(rp, ci, h, a_s, a_d, 0.2)
            close(f["out"], ref["out"], 1e-11, 1e-13, "dense out")
            close(f["lse"], ref["lse"], 1e-11, 1e-13, "dense lse")
            b = o.backward(rp, ci, h, a_s, a_d, 0.2, dout)
            close(b["dh"], ref["dh"], 1e-10, 1e-12, "autograd dh")
            close(b["da_src"], ref["da_src"], 1e-10, 1e-12, "autograd da_src")
            close(b["da_dst"], ref["da_dst"], 1e-10, 1e-12, "autograd da_dst")


def pin_dense_float32_config1(o):
    """The tiny Erdos-Renyi workload itself (N = 512, H = 1, D = 16, fp32)."""
    w = workload.CONFIGS[1]
    rp, ci = workload.make_graph(w)
    h, a_s, a_d, dout = workload.make_features(w, len(rp) - 1)
    ref = dense_torch(rp, ci, h.astype(np.float64), a_s.astype(np.float64),
                      a_d.astype(np.float64), w.slope, dout.astype(np.float64))
    f = o.forward(rp, ci, h, a_s, a_d, w.slope)
    close(f["out"], ref["out"], 1e-11, 1e-13, "cfg1 out")
    close(f["lse"], ref["lse"], 1e-11, 1e-13, "cfg1 lse")
    b = o.backward(rp, ci, h, a_s, a_d, w.slope, dout)
    close(b["dh"], ref["dh"], 1e-10, 1e-12, "cfg1 dh")
    close(b["da_src"], ref["da_src"], 1e-10, 1e-12, "cfg1 da_src")
    close(b["da_dst"], ref["da_dst"], 1e-10, 1e-12, "cfg1 da_dst")


def pin_finite_differences(o, seed=3):
    """Central differences (step 1e-6, fp64) of L = sum(out * G)."""
    rp, ci = irregular_graph(10, seed)
    n, H, D = len(rp) - 1, 2, 3
    h, a_s, a_d, G = random_inputs(n, H, D, seed)
    # keep every edge away from the LeakyReLU kink
    f0 = o.forward(rp, ci, h, a_s, a_d, 0.2)
    b = o.backward(rp, ci, h, a_s, a_d, 0.2, G)

    def loss(h_, a_s_, a_d_):
        return float((o.forward(rp, ci, h_, a_s_, a_d_, 0.2)["out"] * G).sum())

    eps = 1e-6
    for name, arr, grad in (("h", h, b["dh"]), ("a_src", a_s, b["da_src"]), ("a_dst", a_d, b["da_dst"])):
        fd = np.zeros_like(arr)
        it = np.nditer(arr, flags=["multi_index"])
        for _ in it:
            idx = it.multi_index
            plus, minus = arr.copy(), arr.copy()
            plus[idx] += eps
            minus[idx] -= eps
            args_p = [h, a_s, a_d]
            args_m = [h, a_s, a_d]
            k = ("h", "a_src", "a_dst").index(name)
            args_p[k], args_m[k] = plus, minus
            fd[idx] = (loss(*args_p) - loss(*args_m)) / (2 * eps)
        scale = max(1.0, float(np.abs(grad).max()))
        err = float(np.abs(fd - grad).max())
        assert err <= 1e-6 * scale, f"finite differences for {name}: max err {err}"
    assert np.isfinite(f0["out"]).all()


def pin_invariants(o):
    rp, ci = irregular_graph(12, 9)
    n, H, D = len(rp) - 1, 3, 4
    h, a_s, a_d, dout = random_inputs(n, H, D, 9, np.float32)
    deg = np.diff(rp)
    f = o.forward(rp, ci, h, a_s, a_d, 0.2, with_alpha_sum=True)
    # alpha sums to one on every node with in-degree > 0
    assert np.all(np.abs(f["alpha_sum"][deg > 0] - 1.0) <= 1e-12)
    # zero in-degree: out = 0 exactly, lse = -inf, no NaN anywhere
    assert np.all(f["out"][deg == 0] == 0.0)
    assert np.all(np.isneginf(f["lse"][deg == 0]))
    assert not np.isnan(f["out"]).any() and not np.isnan(f["lse"]).any()
    # Delta_i = dout_i . out_i (the identity the GPU backward does not rely on,
    # but which ties the oracle's backward statistics to its forward)
    st = o.node_stats(rp, ci, h, a_s, a_d, 0.2, dout)
    lhs = st["delta"]
    rhs = (dout.astype(np.float64) * f["out"]).sum(-1)
    close(lhs, rhs, 1e-12, 1e-13, "Delta identity")
    b = o.backward(rp, ci, h, a_s, a_d, 0.2, dout)
    assert np.isfinite(b["dh"]).all() and np.isfinite(b["da_src"]).all()


def pin_single_neighbour(o):
    """One in-neighbour: out = h_j exactly, lse = its score, and the score
    gradients vanish (alpha = 1 for any score)."""
    n = 6
    rows = [[(i + 1) % n] for i in range(n)]
    rp, ci = csr_from_lists(rows)
    h, a_s, a_d, dout = random_inputs(n, 2, 8, 4, np.float32)
    f = o.forward(rp, ci, h, a_s, a_d, 0.2)
    assert np.array_equal(f["out"], h[ci].astype(np.float64))
    b = o.backward(rp, ci, h, a_s, a_d, 0.2, dout)
    # dh_j = dout_i for the unique i with j -> i; no score terms
    expect = np.empty_like(b["dh"])
    expect[ci] = dout.astype(np.float64)
    close(b["dh"], expect, 1e-13, 1e-14, "single-neighbour dh")
    assert np.abs(b["da_src"]).max() <= 1e-13 and np.abs(b["da_dst"]).max() <= 1e-13
    # lse is the single score, computed here from the inputs
    sd = (h.astype(np.float64) * a_d.astype(np.float64)).sum(-1)
    ss = (h.astype(np.float64) * a_s.astype(np.float64)).sum(-1)
    z = sd + ss[ci]
    close(f["lse"], np.where(z > 0, z, 0.2 * z), 1e-13, 1e-14, "single-neighbour lse")


def pin_equal_scores(o):
    """a = 0: every score is 0, so out = the neighbour mean, lse = ln(deg)."""
    rp, ci = workload.erdos_renyi(200, 5.0, 21)
    n = len(rp) - 1
    h = workload.normal_f32(21, 1, (n, 2, 8))
    z = np.zeros((2, 8), np.float32)
    f = o.forward(rp, ci, h, z, z, 0.2)
    deg = np.diff(rp)
    mean = np.add.reduceat(h[ci].astype(np.float64), rp[:-1], axis=0) / deg[:, None, None]
    close(f["out"], mean, 1e-13, 1e-14, "neighbour mean")
    close(f["lse"], np.log(deg)[:, None].repeat(2, 1), 1e-13, 1e-14, "ln deg")


def pin_hub_mean(o):
    """A hub with 100,000 equal-score in-neighbours returns their fp64 mean."""
    n = 100_001
    rp = np.zeros(n + 1, np.int32)
    rp[1:] = n                                   # node 0 <- every node
    ci = np.arange(n, dtype=np.int32)
    h = workload.normal_f32(7, 1, (n, 1, 8))
    z = np.zeros((1, 8), np.float32)
    f = o.forward(rp, ci, h, z, z, 0.2, sel=[0])
    close(f["out"][0], h.astype(np.float64).mean(0), 1e-12, 1e-14, "hub mean")
    close(f["lse"][0], [math.log(n)], 1e-14, 0, "hub lse")


def pin_slope_one(o):
    """slope = 1: e = s_dst + s_src, and softmax is shift-invariant, so out does
    not depend on a_dst, ds_dst = 0 and da_dst = 0."""
    rp, ci = workload.erdos_renyi(100, 6.0, 31)
    n = len(rp) - 1
    h, a_s, a_d, dout = random_inputs(n, 2, 4, 31, np.float32)
    f1 = o.forward(rp, ci, h, a_s, a_d, 1.0)
    f0 = o.forward(rp, ci, h, a_s, np.zeros_like(a_d), 1.0)
    close(f1["out"], f0["out"], 1e-12, 1e-13, "slope 1 out")
    st = o.node_stats(rp, ci, h, a_s, a_d, 1.0, dout)
    assert np.abs(st["ds_dst"]).max() <= 1e-12
    b = o.backward(rp, ci, h, a_s, a_d, 1.0, dout)
    assert np.abs(b["da_dst"]).max() <= 1e-11


def pin_permutation(o):
    """Relabelling the nodes permutes every per-node result and leaves da."""
    rp, ci = workload.erdos_renyi(150, 7.0, 41)
    n = len(rp) - 1
    h, a_s, a_d, dout = random_inputs(n, 2, 4, 41, np.float32)
    perm = np.random.default_rng(41).permutation(n).astype(np.int32)
    rp2, ci2 = workload.relabel(rp, ci, perm)
    h2 = np.empty_like(h); h2[perm] = h
    d2 = np.empty_like(dout); d2[perm] = dout
    f = o.forward(rp, ci, h, a_s, a_d, 0.2)
    f2 = o.forward(rp2, ci2, h2, a_s, a_d, 0.2)
    close(f2["out"][perm], f["out"], 1e-12, 1e-13, "perm out")
    close(f2["lse"][perm], f["lse"], 1e-12, 1e-13, "perm lse")
    b = o.backward(rp, ci, h, a_s, a_d, 0.2, dout)
    b2 = o.backward(rp2, ci2, h2, a_s, a_d, 0.2, d2)
    close(b2["dh"][perm], b["dh"], 1e-11, 1e-12, "perm dh")
    close(b2["da_src"], b["da_src"], 1e-11, 1e-12, "perm da_src")


def pin_sampled_modes(o):
    """The per-node entry points agree with the whole-graph ones."""
    rp, ci = irregular_graph(12, 13)
    n = len(rp) - 1
    h, a_s, a_d, dout = random_inputs(n, 2, 4, 13, np.float32)
    sel = [0, 3, 5, 11]
    f = o.forward(rp, ci, h, a_s, a_d, 0.2)
    fs = o.forward(rp, ci, h, a_s, a_d, 0.2, sel=sel)
    close(fs["out"], f["out"][sel], 1e-14, 0, "sampled out")
    b = o.backward(rp, ci, h, a_s, a_d, 0.2, dout, with_mag=True)
    bs = o.backward_rows(rp, ci, h, a_s, a_d, 0.2, dout, sel, with_mag=True)
    close(bs["dh"], b["dh"][sel], 1e-12, 1e-13, "sampled dh")
    close(bs["dh_mag"], b["dh_mag"][sel], 1e-12, 1e-13, "sampled dh_mag")
    # the per-node rows against the dense autograd directly, on two graphs
    # (the hub of the irregular graph reaches every node)
    for rp_x, ci_x, sel_x, seed in ((rp, ci, sel, 13),
                                    (*workload.erdos_renyi(48, 5.0, 17), [1, 2, 30, 47], 17)):
        nx = len(rp_x) - 1
        hx, asx, adx, dx = random_inputs(nx, 2, 4, seed, np.float32)
        ref = dense_torch(rp_x, ci_x, hx.astype(np.float64), asx.astype(np.float64),
                          adx.astype(np.float64), 0.2, dx.astype(np.float64))
        rows = o.backward_rows(rp_x, ci_x, hx, asx, adx, 0.2, dx, sel_x)
        close(rows["dh"], ref["dh"][sel_x], 1e-10, 1e-12, "sampled dh vs autograd")
    ag = o.att_grads(rp, ci, h, a_s, a_d, 0.2, dout, with_mag=True)
    for k in ("da_src", "da_dst", "da_src_mag", "da_dst_mag"):
        close(ag[k], b[k], 1e-12, 1e-13, "row-grouped " + k)


def pin_bf16_inputs(o):
    """bfloat16 bit patterns widen exactly: same result as their float32 values."""
    rp, ci = workload.erdos_renyi(80, 5.0, 51)
    n = len(rp) - 1
    h32, a_s, a_d, d32 = random_inputs(n, 2, 8, 51, np.float32)
    hb = workload.f32_to_bf16_bits(h32)
    db = workload.f32_to_bf16_bits(d32)
    hw = workload.bf16_bits_to_f32(hb)
    dw = workload.bf16_bits_to_f32(db)
    fb = o.forward(rp, ci, hb, a_s, a_d, 0.2)
    fw = o.forward(rp, ci, hw, a_s, a_d, 0.2)
    assert np.array_equal(fb["out"], fw["out"])
    bb = o.backward(rp, ci, hb, a_s, a_d, 0.2, db)
    bw = o.backward(rp, ci, hw, a_s, a_d, 0.2, dw)
    assert np.array_equal(bb["dh"], bw["dh"])


def pin_kink_ambiguity(o):
    """The edge 1 -> 0 of the worked example sits exactly on the LeakyReLU kink
    (z = 0).  By hand: its weight is 1/S0 with S0 = e + 1 + e^0.25, its
    da = dout_0 . h_1 = 0 and Delta_0 = (e + 0.25 e^0.25)/S0, so the two
    derivatives (slope 0.2 or 1) move dz of that edge by
    amb = 0.8 Delta_0 / S0; ds_src(1) and ds_dst(0) by amb, dh_1 by
    amb |a_src|, dh_0 by amb |a_dst|, da_src by amb |h_1| and da_dst by
    amb |h_0|; nothing else.  Inputs with no z near 0 give no ambiguity, and
    the per-node and row-grouped entry points agree with the whole graph."""
    with open(os.path.join(GOLDEN, "worked_example.json")) as f:
        fx = json.load(f)
    H, D = fx["H"], fx["D"]
    rp = np.array(fx["row_ptr"], np.int32)
    ci = np.array(fx["col_idx"], np.int32)
    h = np.array(fx["h"], np.float32).reshape(-1, H, D)
    dout = np.array(fx["dout"], np.float32).reshape(-1, H, D)
    a_src = np.array(fx["a_src"], np.float32).reshape(H, D)
    a_dst = np.array(fx["a_dst"], np.float32).reshape(H, D)
    s0 = math.e + 1.0 + math.exp(0.25)
    amb = 0.8 * (math.e + 0.25 * math.exp(0.25)) / s0 / s0
    want = np.zeros((5, D))
    want[1] = amb * np.abs(a_src[0].astype(np.float64))
    want[0] = amb * np.abs(a_dst[0].astype(np.float64))
    b = o.backward(rp, ci, h, a_src, a_dst, fx["slope"], dout, with_kink=True)
    close(b["dh_kink"].reshape(-1, D), want, 1e-12, 1e-15, "kink dh")
    close(b["da_src_kink"].ravel(), amb * np.abs(h[1, 0].astype(np.float64)), 1e-12, 1e-15,
          "kink da_src")
    close(b["da_dst_kink"].ravel(), amb * np.abs(h[0, 0].astype(np.float64)), 1e-12, 1e-15,
          "kink da_dst")
    rows = o.backward_rows(rp, ci, h, a_src, a_dst, fx["slope"], dout, [0, 1, 3], with_kink=True)
    close(rows["dh_kink"].reshape(-1, D), want[[0, 1, 3]], 1e-12, 1e-15, "kink rows")
    ag = o.att_grads(rp, ci, h, a_src, a_dst, fx["slope"], dout, with_kink=True)
    close(ag["da_src_kink"], b["da_src_kink"], 1e-12, 1e-15, "kink row-grouped da_src")
    close(ag["da_dst_kink"], b["da_dst_kink"], 1e-12, 1e-15, "kink row-grouped da_dst")
    # random fp64 inputs: no z within rounding of 0
    rp2, ci2 = irregular_graph(12, 5)
    h2, as2, ad2, d2 = random_inputs(len(rp2) - 1, 2, 3, 77)
    b2 = o.backward(rp2, ci2, h2, as2, ad2, 0.2, d2, with_kink=True)
    assert not b2["dh_kink"].any() and not b2["da_src_kink"].any()


ALL_PINS = [pin_worked_example, pin_dense_forward_backward, pin_dense_float32_config1,
            pin_finite_differences, pin_invariants, pin_single_neighbour, pin_equal_scores,
            pin_hub_mean, pin_slope_one, pin_permutation, pin_sampled_modes, pin_bf16_inputs,
            pin_kink_ambiguity]
