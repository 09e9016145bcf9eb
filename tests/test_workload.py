"""The seeded input generators: structure of the graphs they draw."""
import numpy as np
import pytest

import workload


def _check_csr(rp, ci):
    n = len(rp) - 1
    assert rp[0] == 0 and np.all(np.diff(rp) >= 1)
    assert ci.min() >= 0 and ci.max() < n
    for i in range(0, n, max(1, n // 500)):
        row = ci[rp[i]:rp[i + 1]]
        assert np.all(np.diff(row) > 0), "rows sorted, no duplicates"
        assert i in row, "self-loop present"


def test_er_config_shape():
    rp, ci = workload.make_graph(workload.CONFIGS[1])
    _check_csr(rp, ci)
    assert len(rp) - 1 == 512
    assert 7.0 < len(ci) / 512 - 1 < 9.5          # avg in-degree 8 plus the self-loop


def test_uniform_degree_exact():
    rp, ci = workload.uniform(5000, 16, 7)
    _check_csr(rp, ci)
    assert np.all(np.diff(rp) == 17)


def test_chung_lu_heavy_tail_and_cap():
    rp, ci = workload.chung_lu(200_000, 2.1, 20.0, 5_000.0, 9)
    _check_csr(rp, ci)
    indeg = np.diff(rp)
    assert indeg.max() <= 5_001
    assert indeg.max() > 50 * np.median(indeg)     # power-law tail
    outdeg = np.bincount(ci, minlength=len(rp) - 1)
    assert outdeg.max() > 50 * np.median(outdeg)


def test_rmat_dedup_and_skew():
    rp, ci = workload.rmat(14, 8, 0.57, 0.19, 0.19, 3)
    _check_csr(rp, ci)
    assert len(rp) - 1 == 1 << 14
    assert len(ci) < (1 << 14) * 9                 # duplicates removed


def test_generators_deterministic():
    a = workload.chung_lu(20_000, 2.3, 10.0, 1e9, 5)
    b = workload.chung_lu(20_000, 2.3, 10.0, 1e9, 5)
    assert np.array_equal(a[0], b[0]) and np.array_equal(a[1], b[1])
    x = workload.normal_f32(1, 2, (1000,))
    y = workload.normal_f32(1, 2, (1000,))
    assert np.array_equal(x, y)
    assert not np.array_equal(x, workload.normal_f32(1, 3, (1000,)))


def test_rcm_is_permutation_and_relabel_preserves_edges():
    rp, ci = workload.rmat(12, 8, 0.57, 0.19, 0.19, 4)
    rp, ci = workload.permute_random(rp, ci, 4)
    new_id = workload.rcm_order(rp, ci)
    assert np.array_equal(np.sort(new_id), np.arange(len(rp) - 1))
    rp2, ci2 = workload.relabel(rp, ci, new_id)
    assert len(ci2) == len(ci)
    # the edge set maps through new_id
    dst = np.repeat(np.arange(len(rp) - 1), np.diff(rp))
    e1 = np.sort(new_id[dst].astype(np.int64) << 32 | new_id[ci])
    dst2 = np.repeat(np.arange(len(rp2) - 1), np.diff(rp2))
    e2 = np.sort(dst2.astype(np.int64) << 32 | ci2)
    assert np.array_equal(e1, e2)


def test_rcm_reduces_bandwidth():
    rp, ci = workload.rmat(12, 8, 0.57, 0.19, 0.19, 6)
    rp, ci = workload.permute_random(rp, ci, 6)
    dst = np.repeat(np.arange(len(rp) - 1), np.diff(rp))
    bw_random = np.abs(dst - ci).mean()
    rp2, ci2 = workload.relabel(rp, ci, workload.rcm_order(rp, ci))
    dst2 = np.repeat(np.arange(len(rp2) - 1), np.diff(rp2))
    assert np.abs(dst2 - ci2).mean() < 0.8 * bw_random


def test_normal_moments_and_bf16_rounding():
    x = workload.normal_f32(3, 1, (200_000,), 0.1)
    assert abs(x.mean()) < 2e-3 and abs(x.std() - 0.1) < 2e-3
    b = workload.f32_to_bf16_bits(x)
    y = workload.bf16_bits_to_f32(b)
    rel = np.abs(y - x) / np.maximum(np.abs(x), 1e-30)
    assert rel.max() <= 2.0 ** -8
    # exact for values already representable
    assert np.array_equal(workload.f32_to_bf16_bits(y), b)


@pytest.mark.parametrize("idx", [1, 2])
def test_features_shapes(idx):
    w = workload.CONFIGS[idx]
    h, a_s, a_d, dout = workload.make_features(w, 100)
    assert h.shape == (100, w.H, w.D) and dout.shape == h.shape
    assert a_s.shape == (w.H, w.D) and a_d.shape == (w.H, w.D)


def test_hubs_then_rcm_order():
    rp, ci = workload.chung_lu(5_000, 2.1, 12.0, 1_500.0, 3)
    n = len(rp) - 1
    deg = np.diff(rp.astype(np.int64)) + np.bincount(ci, minlength=n)
    new_id = workload.hubs_then_rcm_order(rp, ci, 200)
    assert np.array_equal(np.sort(new_id), np.arange(n))       # a permutation
    order = np.argsort(new_id)                                  # old id by new id
    n_hub = int((deg > 200).sum())
    assert n_hub > 0
    assert np.all(deg[order[:n_hub]] > 200) and np.all(deg[order[n_hub:]] <= 200)
    assert np.all(np.diff(deg[order[:n_hub]]) <= 0)             # descending degree
    rcm = workload.rcm_order(rp, ci)
    assert np.all(np.diff(rcm[order[n_hub:]]) > 0)              # the rest keep RCM order
    rp2, ci2 = workload.relabel(rp, ci, new_id)
    assert len(ci2) == len(ci)
