"""Graph-transformer attention: the CUDA path against the fp64 oracle on the
same seeded inputs, element by element: out, lse, dq, dkey, dval over every
bucket path, shape and dtype."""
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
    arrs = [workload.normal_f32(seed, s, (n, H, D), 1.0) for s in (1, 5, 6, 4)]
    if dtype == "bf16":
        arrs = [workload.f32_to_bf16_bits(x) for x in arrs]
    return arrs   # q, key, val, dout


def run(rp, ci, H, D, dtype, tiling=None, seed=3, graph=None):
    import graph_neural_network_gb300 as gnn
    n = len(rp) - 1
    q, k, v, dout = inputs(n, H, D, dtype, seed)
    g = graph or device_graph(dict(row_ptr=np.asarray(rp, np.int32),
                                   col=np.asarray(ci, np.int32)), tiling)
    Q, K, Vt, G = (to_device(x, dtype) for x in (q, k, v, dout))
    out, lse = gnn.transformer_forward(g, Q, K, Vt)
    dq, dk, dv = gnn.transformer_backward(g, Q, K, Vt, lse, G)
    torch.cuda.synchronize()
    gnn.check_device_error(g)
    return (q, k, v, dout), dict(out=out, lse=lse, dq=dq, dkey=dk, dval=dv)


def check(rp, ci, H, D, dtype, tiling=None, seed=3, what=""):
    (q, k, v, dout), got = run(rp, ci, H, D, dtype, tiling, seed)
    scale = D ** -0.5
    f = oracle.gt_forward(rp, ci, q, k, v, scale, with_mag=True)
    b = oracle.gt_backward(rp, ci, q, k, v, scale, dout, with_mag=True)
    assert_close(to_f64(got["out"]), f["out"], dtype, f["out_mag"], what + " out")
    assert_close(to_f64(got["lse"]), f["lse"], "f32", None, what + " lse")
    for key in ("dq", "dkey", "dval"):
        assert_close(to_f64(got[key]), b[key], dtype, b[key + "_mag"], f"{what} {key}")
    return got


@pytest.mark.parametrize("tiling", TILINGS, ids=lambda t: "t%d_%d_%d" % t)
@pytest.mark.parametrize("dtype", ["f32", "bf16"])
def test_transformer_bucket_thresholds(dtype, tiling):
    rp, ci = testgraphs.with_in_degrees(THRESHOLD_DEGREES, n_nodes=2500, seed=7)
    check(rp, ci, 4, 8 if dtype == "f32" else 16, dtype, tiling, what=f"thr {tiling}")


SHAPES = [(1, 4, "f32"), (3, 4, "f32"), (4, 32, "f32"), (1, 128, "f32"), (2, 8, "bf16"),
          (8, 16, "bf16"), (1, 128, "bf16"), (4, 64, "bf16"), (1, 256, "bf16")]


@pytest.mark.parametrize("shape", SHAPES, ids=lambda s: "H%d_D%d_%s" % s)
def test_transformer_shapes(shape):
    H, D, dtype = shape
    rp, ci = testgraphs.with_in_degrees([0, 5, 70, 300], n_nodes=700, seed=H * 100 + D)
    check(rp, ci, H, D, dtype, (8, 64, 16), seed=17, what=f"shape {shape}")


@pytest.mark.parametrize("dtype", ["f32", "bf16"])
def test_transformer_power_law_default_tiling(dtype):
    rp, ci = workload.chung_lu(30_000, 2.1, 20.0, 6_000.0, 13)
    check(rp, ci, 4, 32 if dtype == "f32" else 64, dtype, what="chung-lu")


def test_transformer_reproducible_and_autograd():
    import graph_neural_network_gb300 as gnn
    rp, ci = workload.chung_lu(20_000, 2.1, 15.0, 4_000.0, 29)
    a = check(rp, ci, 2, 16, "f32", seed=9, what="run 1")
    b = check(rp, ci, 2, 16, "f32", seed=9, what="run 2")
    for key in a:
        assert torch.equal(a[key], b[key]), key
    g = device_graph(dict(row_ptr=rp, col=ci))
    (q, k, v, dout), got = run(rp, ci, 2, 16, "f32", seed=9, graph=g)
    Q, K, Vt = (to_device(x, "f32").requires_grad_(True) for x in (q, k, v))
    y = gnn.TransformerAggregate.apply(g, Q, K, Vt, 0.25)
    y.backward(to_device(dout, "f32"))
    assert torch.equal(y.detach(), got["out"])
    assert torch.equal(Q.grad, got["dq"]) and torch.equal(K.grad, got["dkey"])
    assert torch.equal(Vt.grad, got["dval"])
