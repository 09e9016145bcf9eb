"""GATv2 attention: the CUDA path against the fp64 oracle on the same seeded
inputs, element by element: out, lse, dxl, dxr, datt over every bucket path,
shape and dtype."""
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


def inputs(n, H, D, dtype, seed):
    xl = workload.normal_f32(seed, 1, (n, H, D), 1.0)
    xr = workload.normal_f32(seed, 5, (n, H, D), 1.0)
    dout = workload.normal_f32(seed, 4, (n, H, D), 1.0)
    att = workload.normal_f32(seed, 2, (H, D), 0.1)
    if dtype == "bf16":
        xl, xr, dout = (workload.f32_to_bf16_bits(x) for x in (xl, xr, dout))
    return xl, xr, att, dout


def run(rp, ci, H, D, dtype, tiling=None, seed=3, slope=0.2, graph=None):
    import graph_neural_network_gb300 as gnn
    n = len(rp) - 1
    xl, xr, att, dout = inputs(n, H, D, dtype, seed)
    g = graph or device_graph(dict(row_ptr=np.asarray(rp, np.int32),
                                   col=np.asarray(ci, np.int32)), tiling)
    XL, XR, G = (to_device(x, dtype) for x in (xl, xr, dout))
    A = torch.from_numpy(att).cuda()
    out, lse = gnn.gatv2_forward(g, XL, XR, A, slope)
    dxl, dxr, datt = gnn.gatv2_backward(g, XL, XR, A, slope, lse, G)
    torch.cuda.synchronize()
    gnn.check_device_error(g)
    return (xl, xr, att, dout), dict(out=out, lse=lse, dxl=dxl, dxr=dxr, datt=datt), g


def check(rp, ci, H, D, dtype, tiling=None, seed=3, slope=0.2, what=""):
    (xl, xr, att, dout), got, g = run(rp, ci, H, D, dtype, tiling, seed, slope)
    f = oracle.gatv2_forward(rp, ci, xl, xr, att, slope, with_mag=True)
    b = oracle.gatv2_backward(rp, ci, xl, xr, att, slope, dout, with_mag=True)
    assert_close(to_f64(got["out"]), f["out"], dtype, f["out_mag"], what + " out")
    assert_close(to_f64(got["lse"]), f["lse"], "f32", None, what + " lse")
    assert_close(to_f64(got["dxl"]), b["dxl"], dtype, b["dxl_mag"], what + " dxl")
    assert_close(to_f64(got["dxr"]), b["dxr"], dtype, b["dxr_mag"], what + " dxr")
    assert_close(to_f64(got["datt"]), b["datt"], dtype, b["datt_mag"], what + " datt")
    return got


@pytest.mark.parametrize("tiling", TILINGS, ids=lambda t: "t%d_%d_%d" % t)
@pytest.mark.parametrize("dtype", ["f32", "bf16"])
def test_gatv2_bucket_thresholds(dtype, tiling):
    rp, ci = testgraphs.with_in_degrees(THRESHOLD_DEGREES, n_nodes=2500, seed=7)
    check(rp, ci, 4, 8 if dtype == "f32" else 16, dtype, tiling, what=f"thr {tiling}")


SHAPES = [(1, 4, "f32"), (3, 4, "f32"), (4, 32, "f32"), (1, 128, "f32"), (2, 8, "bf16"),
          (8, 16, "bf16"), (1, 128, "bf16"), (4, 64, "bf16"), (1, 256, "bf16")]


@pytest.mark.parametrize("shape", SHAPES, ids=lambda s: "H%d_D%d_%s" % s)
def test_gatv2_shapes(shape):
    H, D, dtype = shape
    rp, ci = testgraphs.with_in_degrees([0, 5, 70, 300], n_nodes=700, seed=H * 100 + D)
    check(rp, ci, H, D, dtype, (8, 64, 16), seed=17, what=f"shape {shape}")


@pytest.mark.parametrize("dtype", ["f32", "bf16"])
def test_gatv2_power_law_default_tiling(dtype):
    rp, ci = workload.chung_lu(30_000, 2.1, 20.0, 6_000.0, 13)
    check(rp, ci, 4, 32 if dtype == "f32" else 64, dtype, what="chung-lu")


def test_gatv2_slope_and_reproducibility():
    rp, ci = workload.chung_lu(20_000, 2.1, 15.0, 4_000.0, 29)
    check(rp, ci, 2, 16, "f32", slope=1.0, what="slope 1")
    # the forward's score writes LeakyReLU(z) as (1 + s)/2 z + (1 - s)/2 |z|, for any slope
    check(rp, ci, 2, 16, "f32", slope=1.5, what="slope 1.5")
    check(rp, ci, 2, 16, "bf16", slope=-0.3, what="slope -0.3")
    check(rp, ci, 2, 16, "f32", slope=0.0, what="slope 0")
    a = check(rp, ci, 2, 16, "f32", seed=9, what="run 1")
    b = check(rp, ci, 2, 16, "f32", seed=9, what="run 2")
    for k in a:
        assert torch.equal(a[k], b[k]), k


def test_gatv2_autograd_and_limits():
    import graph_neural_network_gb300 as gnn
    rp, ci = workload.erdos_renyi(300, 6.0, 3)
    g = device_graph(dict(row_ptr=rp, col=ci))
    (xl, xr, att, dout), got, _ = run(rp, ci, 2, 16, "f32", graph=g)
    XL = to_device(xl, "f32").requires_grad_(True)
    XR = to_device(xr, "f32").requires_grad_(True)
    A = torch.from_numpy(att).cuda().requires_grad_(True)
    y = gnn.GATv2Aggregate.apply(g, XL, XR, A, 0.2)
    y.backward(to_device(dout, "f32"))
    assert torch.equal(y.detach(), got["out"])
    assert torch.equal(XL.grad, got["dxl"]) and torch.equal(XR.grad, got["dxr"])
    assert torch.equal(A.grad, got["datt"])
    with pytest.raises(gnn.GnnError) as ex:   # rows above 512 bytes are not supported
        z = torch.zeros((300, 2, 128), device="cuda")
        gnn.gatv2_forward(g, z, z, torch.zeros((2, 128), device="cuda"))
    assert ex.value.status == 2
