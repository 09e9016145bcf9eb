"""SpMM-family propagation (GCN / GraphConv): the CUDA path against the fp64
oracle on the same seeded inputs, element by element, forward (A~ x over the
CSR) and backward (A~^T dout over the cached CSC), every normalisation,
bucket path, row width and dtype."""
import numpy as np
import pytest
import torch

import oracle
import workload
from workload import testgraphs
from gpu_util import assert_close, device_graph, to_device, to_f64

pytestmark = pytest.mark.gpu

NORMS = ["sum", "mean", "sym"]
TILINGS = [(64, 4096, 2048), (1024, 4096, 2048), (8, 64, 16), (0, 0, 1)]
THRESHOLD_DEGREES = [0, 1, 2, 3, 7, 8, 9, 15, 16, 17, 63, 64, 65, 127, 128, 129, 257, 1000, 2049,
                     4096, 4097]


def features(n, F, dtype, seed):
    x = workload.normal_f32(seed, 1, (n, F), 1.0)
    return workload.f32_to_bf16_bits(x) if dtype == "bf16" else x


def check(rp, ci, F, dtype, norm, tiling=None, seed=3, what=""):
    import graph_neural_network_gb300 as gnn
    n = len(rp) - 1
    x = features(n, F, dtype, seed)
    g_out = features(n, F, dtype, seed + 1)
    g = device_graph(dict(row_ptr=np.asarray(rp, np.int32), col=np.asarray(ci, np.int32)), tiling)
    out = gnn.gcn_forward(g, to_device(x, dtype), norm)
    dx = gnn.gcn_backward(g, to_device(g_out, dtype), norm)
    torch.cuda.synchronize()
    gnn.check_device_error(g)
    f = oracle.spmm_forward(rp, ci, x, norm, with_mag=True)
    b = oracle.spmm_backward(rp, ci, g_out, norm, with_mag=True)
    assert_close(to_f64(out), f["out"], dtype, f["out_mag"], f"{what} {norm} out")
    assert_close(to_f64(dx), b["dx"], dtype, b["dx_mag"], f"{what} {norm} dx")
    return out, dx


@pytest.mark.parametrize("norm", NORMS)
@pytest.mark.parametrize("tiling", TILINGS, ids=lambda t: "t%d_%d_%d" % t)
@pytest.mark.parametrize("dtype", ["f32", "bf16"])
def test_spmm_bucket_thresholds(dtype, tiling, norm):
    """In-degrees at every threshold +-1, zero in-degree, multi-edges, hubs of
    one, two and many chunks; Zipf sources give CSC hubs."""
    rp, ci = testgraphs.with_in_degrees(THRESHOLD_DEGREES, n_nodes=2500, seed=7)
    check(rp, ci, 64 if dtype == "bf16" else 32, dtype, norm, tiling, what=f"thr {tiling}")


@pytest.mark.parametrize("F,dtype", [(4, "f32"), (12, "f32"), (64, "f32"), (128, "f32"),
                                     (256, "f32"), (512, "f32"), (8, "bf16"), (24, "bf16"),
                                     (128, "bf16"), (256, "bf16"), (1024, "bf16")])
def test_spmm_row_widths(F, dtype):
    rp, ci = testgraphs.with_in_degrees([0, 5, 70, 300], n_nodes=700, seed=F)
    for norm in NORMS:
        check(rp, ci, F, dtype, norm, (8, 64, 16), seed=F, what=f"F={F}")


@pytest.mark.parametrize("dtype", ["f32", "bf16"])
def test_spmm_power_law_default_tiling(dtype):
    rp, ci = workload.chung_lu(50_000, 2.1, 20.0, 10_000.0, 13)
    check(rp, ci, 128, dtype, "sym", what="chung-lu")


def _offset_copy(x, dtype):
    """x on the device at an address 16 bytes past a 32-byte boundary."""
    t = to_device(x, dtype)
    pad = 16 // t.element_size()
    buf = torch.empty(t.numel() + pad, dtype=t.dtype, device="cuda")
    view = buf[pad:].view(t.shape)
    view.copy_(t)
    assert view.data_ptr() % 32 == 16
    return view


@pytest.mark.parametrize("dtype", ["f32", "bf16"])
def test_spmm_rows_off_32_byte_boundaries(dtype):
    """Rows of an even number of 16-byte vectors run with 32-byte lane vectors
    when they start on 32-byte boundaries, else with 16-byte ones; both
    against the oracle, light nodes one per sub-group, mid nodes and hubs."""
    import graph_neural_network_gb300 as gnn
    rp, ci = testgraphs.with_in_degrees(THRESHOLD_DEGREES, n_nodes=2500, seed=61)
    n = len(rp) - 1
    F = 64 if dtype == "f32" else 128
    x = features(n, F, dtype, 61)
    g_out = features(n, F, dtype, 62)
    g = device_graph(dict(row_ptr=np.asarray(rp, np.int32), col=np.asarray(ci, np.int32)),
                     (8, 64, 16))
    f = oracle.spmm_forward(rp, ci, x, "sym", with_mag=True)
    b = oracle.spmm_backward(rp, ci, g_out, "sym", with_mag=True)
    for xd, gd in ((to_device(x, dtype), to_device(g_out, dtype)),
                   (_offset_copy(x, dtype), _offset_copy(g_out, dtype))):
        out = gnn.gcn_forward(g, xd, "sym")
        dx = gnn.gcn_backward(g, gd, "sym")
        torch.cuda.synchronize()
        what = f"offset {xd.data_ptr() % 32}"
        assert_close(to_f64(out), f["out"], dtype, f["out_mag"], f"{what} sym out")
        assert_close(to_f64(dx), b["dx"], dtype, b["dx_mag"], f"{what} sym dx")


def test_spmm_reproducible_and_autograd():
    import graph_neural_network_gb300 as gnn
    rp, ci = workload.chung_lu(20_000, 2.1, 20.0, 5_000.0, 29)
    n = len(rp) - 1
    x = features(n, 64, "f32", 29)
    o1, d1 = check(rp, ci, 64, "f32", "sym", seed=29, what="run 1")
    o2, d2 = check(rp, ci, 64, "f32", "sym", seed=29, what="run 2")
    assert torch.equal(o1, o2) and torch.equal(d1, d2)
    g = device_graph(dict(row_ptr=rp, col=ci))
    xt = to_device(x, "f32").requires_grad_(True)
    y = gnn.GCNAggregate.apply(g, xt, "mean")
    gy = to_device(features(n, 64, "f32", 30), "f32")
    y.backward(gy)
    assert torch.equal(y.detach(), gnn.gcn_forward(g, xt.detach(), "mean"))
    assert torch.equal(xt.grad, gnn.gcn_backward(g, gy, "mean"))


def test_spmm_rejects_bad_arguments():
    import graph_neural_network_gb300 as gnn
    rp, ci = workload.erdos_renyi(64, 4.0, 1)
    g = device_graph(dict(row_ptr=rp, col=ci))
    with pytest.raises(gnn.GnnError) as ex:
        gnn.gcn_forward(g, torch.zeros((64, 3), device="cuda"), "sum")   # 12 bytes per row
    assert ex.value.status == 2
    with pytest.raises(gnn.GnnError) as ex:
        gnn.gcn_forward(g, torch.zeros((64, 1024), device="cuda"), "sum")  # 4 KiB rows
    assert ex.value.status == 2
    x = torch.zeros((64, 16), device="cuda")
    small = torch.empty(16, dtype=torch.uint8, device="cuda")
    with pytest.raises(gnn.GnnError) as ex:
        gnn.gcn_forward(g, x, "sym", ws=small)
    assert ex.value.status == 4
