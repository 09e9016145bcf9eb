"""Error paths of the compute entry points.  No fault is provoked: the bad
arguments are rejected by host-side checks before a kernel launches, and the
timeout case is a bounded device wait that runs out and reports a status."""
import pytest
import torch

from workload import testgraphs
from gpu_util import device_graph, make_case, to_device

pytestmark = pytest.mark.gpu


@pytest.fixture(scope="module")
def setup():
    rp, ci = testgraphs.with_in_degrees([3, 90, 2], n_nodes=200, seed=1)
    case = make_case(rp, ci, 2, 16, "f32", 1)
    return case, device_graph(case, (8, 64, 16))


def test_unsupported_shapes(setup):
    import graph_neural_network_gb300 as gnn
    case, g = setup
    for H, D, dt in [(2, 6, torch.float32), (2, 24, torch.bfloat16), (1, 256, torch.float32),
                     (64, 16, torch.float32)]:
        h = torch.zeros(g.n, H, D, dtype=dt, device="cuda")
        with pytest.raises(gnn.GnnError) as ex:
            gnn.gat_forward(g, h, torch.zeros(H, D, device="cuda"), torch.zeros(H, D, device="cuda"))
        assert ex.value.status == 2


def test_misaligned_features(setup):
    import graph_neural_network_gb300 as gnn
    case, g = setup
    flat = torch.zeros(g.n * 2 * 16 + 1, device="cuda")
    h = flat[1:].view(g.n, 2, 16)
    with pytest.raises(gnn.GnnError) as ex:
        gnn.gat_forward(g, h, torch.zeros(2, 16, device="cuda"), torch.zeros(2, 16, device="cuda"))
    assert ex.value.status == 1


def test_workspace_too_small(setup):
    import graph_neural_network_gb300 as gnn
    case, g = setup
    h = to_device(case["h"], "f32")
    a = torch.zeros(2, 16, device="cuda")
    small = torch.empty(256, dtype=torch.uint8, device="cuda")
    out, lse = gnn.gat_forward(g, h, a, a)
    with pytest.raises(gnn.GnnError) as ex:
        gnn.gat_backward(g, h, a, a, 0.2, lse, h, ws=small)
    assert ex.value.status == 4


def test_workspace_has_no_edge_by_head_term():
    """Workspace grows with N * H and the hub chunks, never with E * H."""
    import workload
    rp, ci = workload.chung_lu(30_000, 2.1, 40.0, 5_000.0, 3)
    case = make_case(rp, ci, 8, 16, "bf16", 3)
    g = device_graph(case)
    st = g.stats()
    n, e, H, D = st["n"], st["e"], 8, 16
    ws = g.workspace_bytes(H, D, torch.bfloat16)
    sms = torch.cuda.get_device_properties(g.device).multi_processor_count
    blocks = min(8 * sms, max(1, -(-n // 128)))   # attention-gradient partial-sum blocks
    # per node and head: a 16-byte record, ds_src, and the two score halves
    bound = (28 * n * H + 16 * st["csr"]["hub_chunks"] * H
             + 4 * st["csc"]["hub_chunks"] * H * (D + 1) + 16 * blocks * H * D + 9 * 256)
    assert ws <= bound
    assert ws < 4 * e * H / 2


def test_peak_memory_has_no_edge_by_head_term():
    """Device memory the forward + backward calls take beyond their inputs
    and outputs (workspace and any temporary of the binding), as torch's
    allocator records it, stays far below one float per edge and head."""
    import graph_neural_network_gb300 as gnn
    import workload
    rp, ci = workload.chung_lu(200_000, 2.1, 50.0, 20_000.0, 11)
    H, D = 8, 16
    case = make_case(rp, ci, H, D, "bf16", 5)
    h = to_device(case["h"], "bf16")
    dout = to_device(case["dout"], "bf16")
    a_s = torch.from_numpy(case["a_src"]).cuda()
    a_d = torch.from_numpy(case["a_dst"]).cuda()
    g = device_graph(case)
    torch.cuda.synchronize()
    torch.cuda.reset_peak_memory_stats()
    base = torch.cuda.memory_allocated()
    out, lse = gnn.gat_forward(g, h, a_s, a_d, 0.2)
    dh, da_s, da_d = gnn.gat_backward(g, h, a_s, a_d, 0.2, lse, dout)
    torch.cuda.synchronize()
    peak = torch.cuda.max_memory_allocated() - base
    outputs = sum(t.numel() * t.element_size() for t in (out, lse, dh, da_s, da_d))
    e = len(case["col"])
    assert peak - outputs < 4 * e * H / 4, (peak - outputs, 4 * e * H)


def test_bounded_wait_reports_timeout_and_context_survives(setup):
    """A device wait that nothing completes gives up after its poll limit and
    the host reads GNN_ERR_TIMEOUT; the context stays usable (no fault, no
    hang)."""
    import graph_neural_network_gb300 as gnn
    from graph_neural_network_gb300 import _native
    from gpu_util import compare, run_gpu, run_oracle
    rp, ci = testgraphs.with_in_degrees([0, 3, 70, 300, 3000], n_nodes=600, seed=5)
    case = make_case(rp, ci, 2, 16, "f32", 5)
    g = device_graph(case)
    lib = _native.load()
    assert lib.gnn_wait_selftest(g.handle, 1000, None) == _native.OK
    with pytest.raises(gnn.GnnError) as ex:
        gnn.check_device_error(g)
    assert ex.value.status == _native.ERR_TIMEOUT
    assert gnn.check_device_error(g) == 0          # the status word was cleared
    compare(run_gpu(case, graph=g), run_oracle(case), "f32", what="after a timeout")
