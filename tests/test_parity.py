"""CUDA path vs the fp64 oracle on the same seeded inputs, element by element:
out, lse, dh, da_src, da_dst over every bucket path, shape and dtype."""
import numpy as np
import pytest
import torch

import workload
from workload import testgraphs
from gpu_util import (assert_close, compare, device_graph, make_case, run_gpu, run_oracle,
                      to_device, to_f64)

pytestmark = pytest.mark.gpu

SHAPES = [  # (H, D, dtype): row vectors rv = H * D * size / 16
    (1, 4, "f32"), (1, 16, "f32"), (3, 4, "f32"), (4, 32, "f32"), (2, 128, "f32"),
    (8, 64, "f32"), (2, 8, "bf16"), (6, 8, "bf16"), (8, 16, "bf16"), (1, 128, "bf16"),
    (4, 64, "bf16"), (12, 32, "bf16"), (1, 256, "bf16"),
]
TILINGS = [(64, 4096, 2048), (1024, 4096, 2048), (8, 64, 16), (0, 0, 1)]
THRESHOLD_DEGREES = [0, 1, 2, 3, 7, 8, 9, 15, 16, 17, 63, 64, 65, 127, 128, 129, 257, 1000, 2049,
                     4096, 4097]


def test_config1_tiny_erdos_renyi():
    w = workload.CONFIGS[1]
    rp, ci = workload.make_graph(w)
    case = make_case(rp, ci, w.H, w.D, w.dtype, w.seed, w.slope)
    compare(run_gpu(case), run_oracle(case), w.dtype, what="cfg1")


@pytest.mark.parametrize("tiling", TILINGS, ids=lambda t: "t%d_%d_%d" % t)
@pytest.mark.parametrize("dtype", ["f32", "bf16"])
def test_bucket_thresholds(tiling, dtype):
    """In-degrees at every threshold +-1 (zero in-degree, multi-edges, hubs of
    one, two and many chunks, ragged last chunks), Zipf sources so that the
    CSC side has hubs too."""
    rp, ci = testgraphs.with_in_degrees(THRESHOLD_DEGREES, n_nodes=2500, seed=7)
    case = make_case(rp, ci, 4, 16 if dtype == "bf16" else 8, dtype, 11)
    compare(run_gpu(case, tiling), run_oracle(case), dtype, what=f"thresholds {tiling}")


@pytest.mark.parametrize("shape", SHAPES, ids=lambda s: "H%d_D%d_%s" % s)
def test_shapes(shape):
    H, D, dtype = shape
    rp, ci = testgraphs.with_in_degrees([0, 5, 70, 300], n_nodes=700, seed=H * 100 + D)
    case = make_case(rp, ci, H, D, dtype, 17)
    compare(run_gpu(case, (8, 64, 16)), run_oracle(case), dtype, what=f"shape {shape}")


@pytest.mark.parametrize("dtype", ["f32", "bf16"])
def test_uniform_graph_default_tiling(dtype):
    rp, ci = workload.uniform(20_000, 16, 5)
    case = make_case(rp, ci, 4, 32 if dtype == "f32" else 64, dtype, 5)
    compare(run_gpu(case), run_oracle(case), dtype, what="uniform")


def test_power_law_default_tiling():
    rp, ci = workload.chung_lu(50_000, 2.1, 20.0, 10_000.0, 13)
    case = make_case(rp, ci, 8, 16, "bf16", 13)
    compare(run_gpu(case), run_oracle(case), "bf16", what="chung-lu")


@pytest.mark.parametrize("dtype", ["f32", "bf16"])
def test_single_neighbour_is_a_copy(dtype):
    """One in-neighbour: alpha = 1 and out_i = h_j exactly (bitwise)."""
    rp, ci = testgraphs.ring(1000)
    case = make_case(rp, ci, 2, 32, dtype, 23)
    gpu = run_gpu(case)
    h = case["h"] if dtype == "f32" else workload.bf16_bits_to_f32(case["h"])
    assert np.array_equal(gpu["out"], h[ci].astype(np.float64))
    compare(gpu, run_oracle(case), dtype, what="ring")


def test_equal_scores_give_the_mean():
    rp, ci = testgraphs.with_in_degrees([1, 2, 3, 50, 5000], n_nodes=600, seed=29)
    case = make_case(rp, ci, 2, 16, "f32", 29)
    case["a_src"][:] = 0
    case["a_dst"][:] = 0
    gpu = run_gpu(case, (8, 64, 16))
    deg = np.diff(rp)
    ok = deg > 0
    mean = np.add.reduceat(case["h"][ci].astype(np.float64), rp[:-1][ok], axis=0) / deg[ok][:, None, None]
    assert_close(gpu["out"][ok], mean, "f32", None, "mean")
    assert np.allclose(gpu["lse"][ok], np.log(deg[ok])[:, None], rtol=1e-6)


def test_isolated_nodes_and_empty_edge_set():
    rp, ci = testgraphs.isolated(50)
    case = make_case(rp, ci, 2, 16, "f32", 31)
    gpu = run_gpu(case)
    assert np.all(gpu["out"] == 0.0) and np.all(np.isneginf(gpu["lse"]))
    assert np.all(gpu["dh"] == 0.0)
    assert np.all(gpu["da_src"] == 0.0) and np.all(gpu["da_dst"] == 0.0)


@pytest.mark.parametrize("tiling", [(64, 4096, 2048), (8, 64, 16)], ids=str)
def test_bitwise_deterministic(tiling):
    rp, ci = testgraphs.with_in_degrees(THRESHOLD_DEGREES, n_nodes=3000, seed=37)
    case = make_case(rp, ci, 4, 32, "bf16", 37)
    a = run_gpu(case, tiling)
    for _ in range(2):
        b = run_gpu(case, tiling)
        for k in ("out", "lse", "dh", "da_src", "da_dst"):
            assert np.array_equal(a[k], b[k], equal_nan=True), k


@pytest.mark.parametrize("dtype", ["f32", "bf16"])
def test_hub_of_1e5_equal_scores_is_the_mean(dtype):
    """One destination with 100,000 distinct in-neighbours and all scores
    equal (a_src = a_dst = 0): out is the fp64 mean of the neighbour rows and
    lse = ln(100,000), within the plain tolerance, in the default tiling (a
    hub of 49 chunks merged in chunk order), and bitwise the same over three
    runs."""
    deg = 100_000
    n = deg + 1
    # node 0 gathers from every other node; the others keep one self-loop
    rp = np.concatenate([[0], deg + np.arange(n, dtype=np.int64)]).astype(np.int32)
    ci = np.concatenate([np.arange(1, n), np.arange(1, n)]).astype(np.int32)
    D = 32 if dtype == "f32" else 64
    case = make_case(rp, ci, 2, D, dtype, 53)
    case["a_src"][:] = 0
    case["a_dst"][:] = 0
    runs = [run_gpu(case, backward=False) for _ in range(3)]
    assert runs[0]["graph"].stats()["csr"]["hub_chunks"] == 49
    h = case["h"] if dtype == "f32" else workload.bf16_bits_to_f32(case["h"])
    mean = h[1:].astype(np.float64).mean(axis=0)
    assert_close(runs[0]["out"][0], mean, dtype, None, f"hub mean {dtype}", strict=True)
    assert_close(runs[0]["lse"][0], np.full(2, np.log(deg)), "f32", None, f"hub lse {dtype}",
                 strict=True)
    for r in runs[1:]:
        assert np.array_equal(r["out"], runs[0]["out"]) and np.array_equal(r["lse"], runs[0]["lse"])


def test_side_stream_matches_default_stream():
    rp, ci = testgraphs.with_in_degrees(THRESHOLD_DEGREES, n_nodes=2000, seed=41)
    case = make_case(rp, ci, 2, 32, "f32", 41)
    a = run_gpu(case, (8, 64, 16))
    s = torch.cuda.Stream()
    with torch.cuda.stream(s):
        b = run_gpu(case, (8, 64, 16), stream=s)
    for k in ("out", "lse", "dh", "da_src", "da_dst"):
        assert np.array_equal(a[k], b[k]), k


@pytest.mark.parametrize("dtype", ["f32", "bf16"])
def test_backward_reusing_the_forward_scores_is_bitwise_the_same(dtype):
    import graph_neural_network_gb300 as gnn
    rp, ci = testgraphs.with_in_degrees(THRESHOLD_DEGREES, n_nodes=2000, seed=47)
    D = 32 if dtype == "f32" else 64
    case = make_case(rp, ci, 2, D, dtype, 47)
    g = device_graph(case, (8, 64, 16))
    h, dout = to_device(case["h"], dtype), to_device(case["dout"], dtype)
    a_s = torch.from_numpy(case["a_src"]).cuda()
    a_d = torch.from_numpy(case["a_dst"]).cuda()
    ws = g.workspace(2, D, h.dtype)
    out, lse = gnn.gat_forward(g, h, a_s, a_d, 0.2, ws=ws)
    ref = gnn.gat_backward(g, h, a_s, a_d, 0.2, lse, dout)  # its own workspace
    got = gnn.gat_backward(g, h, a_s, a_d, 0.2, lse, dout, ws=ws, reuse_scores=True)
    for name, a, b in zip(("dh", "da_src", "da_dst"), ref, got):
        assert torch.equal(a, b), name


def test_autograd_function():
    import graph_neural_network_gb300 as gnn
    rp, ci = testgraphs.with_in_degrees([4, 90, 3], n_nodes=300, seed=43)
    case = make_case(rp, ci, 2, 16, "f32", 43)
    g = run_gpu(case, backward=False)["graph"]
    h = to_device(case["h"], "f32").requires_grad_(True)
    a_s = torch.from_numpy(case["a_src"]).cuda().requires_grad_(True)
    a_d = torch.from_numpy(case["a_dst"]).cuda().requires_grad_(True)
    out = gnn.GATAggregate.apply(g, h, a_s, a_d, 0.2)
    out.backward(to_device(case["dout"], "f32"))
    ref = run_oracle(case)
    assert_close(out.detach().cpu().numpy(), ref["out"], "f32", ref["out_mag"], "autograd out")
    assert_close(h.grad.cpu().numpy(), ref["dh"], "f32", ref["dh_mag"], "autograd dh",
                 kink=ref["dh_kink"])
    assert_close(a_s.grad.cpu().numpy(), ref["da_src"], "f32", ref["da_src_mag"], "da_src",
                 kink=ref["da_src_kink"])
    assert_close(a_d.grad.cpu().numpy(), ref["da_dst"], "f32", ref["da_dst_mag"], "da_dst",
                 kink=ref["da_dst_kink"])


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
def test_rows_off_32_byte_boundaries_take_16_byte_vectors(dtype):
    """Heads of 64 bytes or more run with 32-byte lane vectors when the rows
    start on 32-byte boundaries, else with 16-byte ones; both against the
    oracle, on the same graph."""
    import graph_neural_network_gb300 as gnn
    rp, ci = testgraphs.with_in_degrees(THRESHOLD_DEGREES, n_nodes=2500, seed=59)
    D = 32 if dtype == "f32" else 64
    case = make_case(rp, ci, 2, D, dtype, 59)
    ref = run_oracle(case)
    g = device_graph(case, (8, 64, 16))
    a_s = torch.from_numpy(case["a_src"]).cuda()
    a_d = torch.from_numpy(case["a_dst"]).cuda()
    for h, dout in ((to_device(case["h"], dtype), to_device(case["dout"], dtype)),
                    (_offset_copy(case["h"], dtype), _offset_copy(case["dout"], dtype))):
        out, lse = gnn.gat_forward(g, h, a_s, a_d, 0.2)
        dh, da_s, da_d = gnn.gat_backward(g, h, a_s, a_d, 0.2, lse, dout)
        torch.cuda.synchronize()
        gpu = dict(out=to_f64(out), lse=to_f64(lse), dh=to_f64(dh), da_src=to_f64(da_s),
                   da_dst=to_f64(da_d))
        compare(gpu, ref, dtype, what=f"offset {h.data_ptr() % 32}")


def _positive(seed, stream, shape):
    """Values in (0.75, 1.25): 1 + tanh(x) / 4 of seeded normals."""
    return (1.0 + 0.25 * np.tanh(workload.normal_f32(seed, stream, shape, 1.0))).astype(np.float32)


@pytest.mark.parametrize("dtype", ["f32", "bf16"])
def test_attention_gradients_without_cancellation(dtype):
    """da_src and da_dst held to the plain atol + rtol bound, with no float32
    summation term, on inputs whose sums do not cancel.  Every destination
    has two in-edges: from an A node with a positive row and from a B node
    with a zero row.  Rows, dout and a_src are positive and a_dst negative,
    so z > 0 on the A edge and z < 0 on the B edge, at least 0.25 from the
    kink; then de > 0 on every A edge and the terms of da_src (de h_a) are all
    positive, and those of da_dst (de (1 - slope) h_i per destination) too.
    The A nodes' out-degrees follow a Zipf law, so the source pass runs CSC
    hubs of several chunks as well as light and mid nodes.  A dropped or
    doubled contribution to either sum fails the plain bound."""
    n_a, n_b, n_c = 2000, 2000, 30000
    rp, ci = testgraphs.paired_sources(n_a, n_b, n_c, seed=71)
    n = len(rp) - 1
    H, D = 2, (16 if dtype == "f32" else 32)
    h = _positive(71, 1, (n, H, D))
    h[n_a:n_a + n_b] = 0.0
    dout = _positive(71, 4, (n, H, D))
    a_s = np.full((H, D), 2.0 / D, np.float32)     # a_src . h_a in (1.5, 2.5)
    a_d = np.full((H, D), -0.5 / D, np.float32)    # a_dst . h_i in (-0.625, -0.375)
    if dtype == "bf16":
        h = workload.f32_to_bf16_bits(h)
        dout = workload.f32_to_bf16_bits(dout)
    case = dict(row_ptr=rp, col=ci, h=h, dout=dout, a_src=a_s, a_dst=a_d, H=H, D=D,
                dtype=dtype, slope=0.2)
    # the construction, in float64: z = a_dst.h_i + a_src.h_j is at least 0.25 on every
    # A edge and at most -0.25 on every B edge (per head)
    hf = workload.bf16_bits_to_f32(h) if dtype == "bf16" else h
    sc_src = np.einsum("nkd,kd->nk", hf.astype(np.float64), a_s.astype(np.float64))
    sc_dst = np.einsum("nkd,kd->nk", hf.astype(np.float64), a_d.astype(np.float64))
    dst = np.repeat(np.arange(n), np.diff(rp))
    z = sc_dst[dst] + sc_src[ci]
    assert np.all(z[0::2] >= 0.25) and np.all(z[1::2] <= -0.25)
    ref = run_oracle(case)
    assert np.all(ref["da_src"] > 0) and np.all(ref["da_dst"] > 0)
    assert not np.any(ref["da_src_kink"]) and not np.any(ref["da_dst_kink"])
    g = device_graph(case, None)
    assert g.stats()["csc"]["hubs"] >= 2
    gpu = run_gpu(case, graph=g)
    compare(gpu, ref, dtype, what=f"no cancellation {dtype}")
    for k in ("da_src", "da_dst"):
        assert_close(gpu[k], ref[k], dtype, None, f"no cancellation {dtype} {k}", strict=True)
