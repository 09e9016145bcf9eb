"""gnn_graph_prepare on the GPU: CSC transpose and degree buckets against a
host construction (integer results, compared exactly)."""
import numpy as np
import pytest
import torch

import workload
from workload import testgraphs
from gpu_util import device_graph, make_case

pytestmark = pytest.mark.gpu


def host_csc(rp, ci):
    n = len(rp) - 1
    dst = np.repeat(np.arange(n, dtype=np.int32), np.diff(rp))
    order = np.argsort(ci, kind="stable")           # stable: rows ascending per column
    col_ptr = np.zeros(n + 1, np.int64)
    col_ptr[1:] = np.cumsum(np.bincount(ci, minlength=n))
    return col_ptr.astype(np.int32), dst[order]


def host_buckets(ptr, tiling):
    light_max, cta_max, chunk = tiling
    deg = np.diff(ptr)
    light = np.nonzero(deg <= light_max)[0]
    light = light[np.argsort(-deg[light], kind="stable")]   # descending degree, ties by id
    mid = np.nonzero((deg > light_max) & (deg <= cta_max))[0]
    hub = np.nonzero(deg > cta_max)[0]
    items, hubs, slot = [], [], 0
    for v in hub:
        nch = -(-int(deg[v]) // chunk)
        hubs.append((v, slot, nch, 0))
        for c in range(nch):
            b = int(ptr[v]) + c * chunk
            items.append((v, b, min(int(ptr[v + 1]), b + chunk), slot))
            slot += 1
    for v in mid:
        items.append((v, int(ptr[v]), int(ptr[v + 1]), -1))
    return light, np.array(items, np.int64).reshape(-1, 4), np.array(hubs, np.int64).reshape(-1, 4)


GRAPHS = {
    "er512": lambda: workload.make_graph(workload.CONFIGS[1]),
    "thresholds": lambda: testgraphs.with_in_degrees(
        [0, 1, 7, 8, 9, 63, 64, 65, 100, 4096, 4097, 9000], n_nodes=3000, seed=3),
    "isolated": lambda: testgraphs.isolated(37),
    "star_out": lambda: testgraphs.star_out(5000, extra=2),
    "rmat12": lambda: workload.rmat(12, 16, 0.57, 0.19, 0.19, 9),
}
TILINGS = [(64, 4096, 2048), (1024, 4096, 2048), (8, 64, 16), (0, 0, 1)]


@pytest.mark.parametrize("tiling", TILINGS, ids=lambda t: "t%d_%d_%d" % t)
@pytest.mark.parametrize("name", sorted(GRAPHS))
def test_prepare_matches_host(name, tiling):
    rp, ci = GRAPHS[name]()
    case = make_case(rp, ci, 1, 16, "f32", 1)
    g = device_graph(case, tiling)
    arr = {k: v.cpu().numpy() for k, v in g.arrays().items()}
    col_ptr, row_idx = host_csc(rp, ci)
    assert np.array_equal(arr["col_ptr"], col_ptr)
    assert np.array_equal(arr["row_idx"], row_idx)
    st = g.stats()
    for d, ptr in (("csr", rp), ("csc", col_ptr)):
        light, items, hubs = host_buckets(ptr, tiling)
        assert np.array_equal(arr[f"{d}_light"], light)
        assert np.array_equal(arr[f"{d}_items"].astype(np.int64), items)
        assert np.array_equal(arr[f"{d}_hubs"].astype(np.int64), hubs)
        assert st[d]["max_deg"] == (int(np.diff(ptr).max()) if len(ptr) > 1 else 0)


def test_prepare_is_deterministic():
    rp, ci = workload.rmat(14, 16, 0.57, 0.19, 0.19, 2)
    case = make_case(rp, ci, 1, 16, "f32", 1)
    a = device_graph(case).arrays()
    b = device_graph(case).arrays()
    for k in a:
        assert torch.equal(a[k], b[k]), k


@pytest.mark.parametrize("bad", ["first", "decreasing", "last", "col_high", "col_negative"])
def test_invalid_csr_rejected(bad):
    import graph_neural_network_gb300 as gnn
    rp, ci = testgraphs.with_in_degrees([3, 2, 4, 1], seed=1)
    rp = rp.copy(); ci = ci.copy()
    if bad == "first":
        rp[0] = 1
    elif bad == "decreasing":
        rp[2] = rp[1] - 1
    elif bad == "last":
        rp[-1] += 1
    elif bad == "col_high":
        ci[3] = len(rp) - 1
    else:
        ci[0] = -1
    with pytest.raises(gnn.GnnError) as ex:
        gnn.Graph(torch.from_numpy(rp).cuda(), torch.from_numpy(ci).cuda())
    assert ex.value.status == 3


def test_empty_graph():
    import graph_neural_network_gb300 as gnn
    g = gnn.Graph(torch.zeros(1, dtype=torch.int32, device="cuda"),
                  torch.zeros(0, dtype=torch.int32, device="cuda"))
    st = g.stats()
    assert st["n"] == 0 and st["e"] == 0


def auto_light_max(e, sm_count, cta_max):
    """The automatic light threshold as documented for gnn_tiling: E / (SMs * 512)
    rounded to a power of two (on a log scale), within [64, 1024], at most
    cta_max_deg."""
    per = e / (sm_count * 512.0)
    t = 64
    while t < 1024 and per >= t * 2 ** 0.5:
        t *= 2
    return min(t, cta_max)


@pytest.mark.parametrize("scale,ef", [(10, 8), (16, 16), (19, 32)])
def test_automatic_light_threshold(scale, ef):
    """The default tiling picks the light threshold from the edge count and the
    SM count, and the buckets follow it exactly."""
    rp, ci = workload.rmat(scale, ef, 0.57, 0.19, 0.19, scale)
    case = make_case(rp, ci, 1, 16, "f32", 1)
    g = device_graph(case)                       # default tiling: automatic threshold
    sm = torch.cuda.get_device_properties(0).multi_processor_count
    want = auto_light_max(len(ci), sm, 4096)
    st = g.stats()
    assert st["light_max_deg"] == want and st["cta_max_deg"] == 4096
    arr = {k: v.cpu().numpy() for k, v in g.arrays().items()}
    col_ptr, _ = host_csc(rp, ci)
    for d, ptr in (("csr", rp), ("csc", col_ptr)):
        light, items, hubs = host_buckets(ptr, (want, 4096, 2048))
        assert np.array_equal(arr[f"{d}_light"], light)
        assert np.array_equal(arr[f"{d}_items"].astype(np.int64), items)
        assert np.array_equal(arr[f"{d}_hubs"].astype(np.int64), hubs)


def test_automatic_light_threshold_capped_by_cta_bound():
    """An automatic light threshold never exceeds cta_max_deg."""
    rp, ci = testgraphs.with_in_degrees([0, 1, 7, 8, 9, 15, 16, 17, 40, 100], n_nodes=1500, seed=5)
    case = make_case(rp, ci, 1, 16, "f32", 1)
    g = device_graph(case, (-1, 16, 8))
    st = g.stats()
    assert st["light_max_deg"] == 16 and st["cta_max_deg"] == 16
    arr = {k: v.cpu().numpy() for k, v in g.arrays().items()}
    col_ptr, _ = host_csc(rp, ci)
    for d, ptr in (("csr", rp), ("csc", col_ptr)):
        light, items, hubs = host_buckets(ptr, (16, 16, 8))
        assert np.array_equal(arr[f"{d}_light"], light)
        assert np.array_equal(arr[f"{d}_items"].astype(np.int64), items)
        assert np.array_equal(arr[f"{d}_hubs"].astype(np.int64), hubs)
