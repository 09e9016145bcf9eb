"""Max / min neighbourhood reduction: the CUDA path against the fp64 oracle
on the same seeded inputs.  out and arg are compared bit for bit (out is
always an input value, arg an index); dx element by element within the
float32 summation bound."""
import numpy as np
import pytest
import torch

import oracle
import workload
from workload import testgraphs
from gpu_util import assert_close, device_graph, to_device, to_f64

pytestmark = pytest.mark.gpu

TILINGS = [(64, 4096, 2048), (1024, 4096, 2048), (8, 64, 16), (0, 0, 1)]
THRESHOLD_DEGREES = [0, 1, 2, 3, 7, 8, 9, 15, 16, 17, 63, 64, 65, 127, 128, 129, 257, 1000, 2049,
                     4096, 4097]


def features(n, F, dtype, seed, ties=False):
    if ties:   # small integers: many equal values, decided by the source id
        x = np.random.default_rng(seed).integers(-3, 4, (n, F)).astype(np.float32)
    else:
        x = workload.normal_f32(seed, 1, (n, F), 1.0)
    return workload.f32_to_bf16_bits(x) if dtype == "bf16" else x


def check(rp, ci, F, dtype, op, tiling=None, seed=3, ties=False, what=""):
    import graph_neural_network_gb300 as gnn
    n = len(rp) - 1
    x = features(n, F, dtype, seed, ties)
    dy = features(n, F, dtype, seed + 1)
    g = device_graph(dict(row_ptr=np.asarray(rp, np.int32), col=np.asarray(ci, np.int32)), tiling)
    out, arg = gnn.reduce_forward(g, to_device(x, dtype), op)
    dx = gnn.reduce_backward(g, arg, to_device(dy, dtype))
    torch.cuda.synchronize()
    gnn.check_device_error(g)
    f = oracle.reduce_forward(rp, ci, x, op)
    b = oracle.reduce_backward(f["arg"], dy, with_mag=True)
    got_arg = arg.cpu().numpy()
    assert np.array_equal(got_arg, f["arg"]), f"{what} {op} arg: {(got_arg != f['arg']).sum()} differ"
    assert np.array_equal(to_f64(out), f["out"]), f"{what} {op} out"
    assert_close(to_f64(dx), b["dx"], dtype, b["dx_mag"], f"{what} {op} dx")
    return out, arg


@pytest.mark.parametrize("op", ["max", "min"])
@pytest.mark.parametrize("tiling", TILINGS, ids=lambda t: "t%d_%d_%d" % t)
@pytest.mark.parametrize("dtype", ["f32", "bf16"])
def test_reduce_bucket_thresholds(dtype, tiling, op):
    rp, ci = testgraphs.with_in_degrees(THRESHOLD_DEGREES, n_nodes=2500, seed=7)
    check(rp, ci, 32 if dtype == "f32" else 64, dtype, op, tiling, what=f"thr {tiling}")
    check(rp, ci, 16, dtype, op, tiling, ties=True, what=f"ties {tiling}")


@pytest.mark.parametrize("op", ["max", "min"])
@pytest.mark.parametrize("tiling", TILINGS, ids=lambda t: "t%d_%d_%d" % t)
@pytest.mark.parametrize("dtype", ["f32", "bf16"])
def test_reduce_rows_in_any_order(dtype, tiling, op):
    """Rows that list their sources in no particular order take the full
    (value, source) comparison; rows in ascending order take the strict one.
    With many equal values the winner is the smallest source id either way."""
    for sort_rows in (False, True):
        rp, ci = testgraphs.with_in_degrees(THRESHOLD_DEGREES, n_nodes=2500, seed=17,
                                            sort_rows=sort_rows)
        if not sort_rows:
            rows = np.split(ci, rp[1:-1])
            assert any(np.any(np.diff(r) < 0) for r in rows)
        for F in ((16, 64) if dtype == "f32" else (16, 128)):
            check(rp, ci, F, dtype, op, tiling, ties=True, what=f"sorted={sort_rows} F={F}")


@pytest.mark.parametrize("F,dtype", [(4, "f32"), (12, "f32"), (128, "f32"), (512, "f32"),
                                     (8, "bf16"), (24, "bf16"), (256, "bf16"), (1024, "bf16")])
def test_reduce_row_widths(F, dtype):
    rp, ci = testgraphs.with_in_degrees([0, 5, 70, 300], n_nodes=700, seed=F)
    for op in ("max", "min"):
        check(rp, ci, F, dtype, op, (8, 64, 16), seed=F, what=f"F={F}")


@pytest.mark.parametrize("dtype", ["f32", "bf16"])
def test_reduce_power_law_default_tiling(dtype):
    rp, ci = workload.chung_lu(50_000, 2.1, 20.0, 10_000.0, 13)
    check(rp, ci, 128, dtype, "max", what="chung-lu")
    check(rp, ci, 64, dtype, "min", ties=True, what="chung-lu ties")


def test_reduce_reproducible_and_autograd():
    import graph_neural_network_gb300 as gnn
    rp, ci = workload.chung_lu(20_000, 2.1, 20.0, 5_000.0, 29)
    o1, a1 = check(rp, ci, 64, "f32", "max", ties=True, what="run 1")
    o2, a2 = check(rp, ci, 64, "f32", "max", ties=True, what="run 2")
    assert torch.equal(o1, o2) and torch.equal(a1, a2)
    n = len(rp) - 1
    g = device_graph(dict(row_ptr=rp, col=ci))
    x, dy = features(n, 64, "f32", 31), features(n, 64, "f32", 32)
    xt = to_device(x, "f32").requires_grad_(True)
    y = gnn.ReduceAggregate.apply(g, xt, "min")
    y.backward(to_device(dy, "f32"))
    f = oracle.reduce_forward(rp, ci, x, "min")
    b = oracle.reduce_backward(f["arg"], dy, with_mag=True)
    assert np.array_equal(to_f64(y.detach()), f["out"])
    # the gradient's float32 additions may run in another order: compare values
    assert_close(to_f64(xt.grad), b["dx"], "f32", b["dx_mag"], "autograd dx")


@pytest.mark.parametrize("tiling", TILINGS, ids=lambda t: "t%d_%d_%d" % t)
@pytest.mark.parametrize("dtype", ["f32", "bf16"])
def test_reduce_ordered_backward(dtype, tiling):
    """The atomic-free backward (a masked gather over the cached CSC, hubs in
    chunk order) against the oracle, on graphs whose CSC has light, mid and
    chunked hub sources, with ties; bitwise the same over three runs."""
    import graph_neural_network_gb300 as gnn
    rp, ci = testgraphs.with_in_degrees(THRESHOLD_DEGREES, n_nodes=2500, seed=67)
    n = len(rp) - 1
    F = 32 if dtype == "f32" else 64
    for ties in (False, True):
        x = features(n, F, dtype, 71, ties)
        dy = features(n, F, dtype, 72)
        g = device_graph(dict(row_ptr=rp, col=ci), tiling)
        _, arg = gnn.reduce_forward(g, to_device(x, dtype), "max")
        dyt = to_device(dy, dtype)
        runs = [gnn.reduce_backward(g, arg, dyt, ordered=True) for _ in range(3)]
        torch.cuda.synchronize()
        gnn.check_device_error(g)
        f = oracle.reduce_forward(rp, ci, x, "max")
        b = oracle.reduce_backward(f["arg"], dy, with_mag=True)
        assert np.array_equal(arg.cpu().numpy(), f["arg"])
        assert_close(to_f64(runs[0]), b["dx"], dtype, b["dx_mag"], f"ordered dx {tiling} {ties}")
        for r in runs[1:]:
            assert torch.equal(r, runs[0])
    assert g.stats()["csc"]["hubs"] > 0 or tiling[1] == 4096


def test_reduce_ordered_backward_power_law():
    import graph_neural_network_gb300 as gnn
    rp, ci = workload.chung_lu(50_000, 2.1, 20.0, 10_000.0, 73)
    n = len(rp) - 1
    x, dy = features(n, 128, "bf16", 74), features(n, 128, "bf16", 75)
    g = device_graph(dict(row_ptr=rp, col=ci))
    _, arg = gnn.reduce_forward(g, to_device(x, "bf16"), "min")
    dx = gnn.reduce_backward(g, arg, to_device(dy, "bf16"), ordered=True)
    torch.cuda.synchronize()
    f = oracle.reduce_forward(rp, ci, x, "min")
    b = oracle.reduce_backward(f["arg"], dy, with_mag=True)
    assert_close(to_f64(dx), b["dx"], "bf16", b["dx_mag"], "ordered dx chung-lu")
