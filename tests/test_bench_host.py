"""Host-side helpers of bench.py (CPU only): the bounded oracle sample, the
bytes model and the committed traffic records."""
import json
import os
import sys

import numpy as np

ROOT = os.path.dirname(os.path.dirname(os.path.abspath(__file__)))
sys.path.insert(0, ROOT)

import bench  # noqa: E402


def test_cpu_sample_is_a_csr_prefix():
    rp = np.array([0, 2, 5, 5, 9, 12], np.int32)
    ci = np.arange(12, dtype=np.int32) % 5
    srp, sci, m = bench.cpu_sample(rp, ci, 0.4)   # about 5 of 12 edges
    assert m == 2 and len(srp) == len(rp)
    assert list(srp) == [0, 2, 5, 5, 5, 5]       # rows past m keep no edges
    assert list(sci) == list(ci[:5])
    _, sci_all, m_all = bench.cpu_sample(rp, ci, 1.0)
    assert m_all == 5 and len(sci_all) == 12


def test_bytes_model_matches_its_definition():
    n, e, H, D, s = 1000, 17000, 4, 32, 4
    ab = bench.algorithmic_bytes(n, e, H, D, s)
    idx = 4 * (n + 1) + 4 * e
    assert ab["fwd_main"] == idx + s * e * H * D + s * n * H * D + 4 * n * H
    assert ab["bwd_dst_main"] == idx + s * e * H * D + 2 * s * n * H * D
    assert ab["bwd_src_main"] == idx + s * e * H * D + 2 * s * n * H * D


def test_traffic_records_name_existing_sources():
    with open(os.path.join(ROOT, "profiles", "traffic.json")) as f:
        rec = json.load(f)
    for wl, kernels in rec.items():
        if wl.startswith("_"):
            continue
        for k, entry in kernels.items():
            assert entry["bytes_per_launch"] > 0, (wl, k)
            for src in entry["sources"]:
                assert os.path.exists(os.path.join(ROOT, src)), src
            # a record is reported only while its sources hash to the recorded value
            got = bench.measured_traffic(wl, k)
            current = bench.source_hash([os.path.join(ROOT, p) for p in entry["sources"]])
            assert got == (entry["bytes_per_launch"] if current == entry["source_hash"] else None)


def test_oracle_sample_rate_stays_within_its_budget():
    import time
    w, rp, ci, h, a_s, a_d, dout = bench.load_workload(1)   # the 512-node graph
    t0 = time.perf_counter()
    rate, sample = bench.oracle_sample_rate(w, rp, ci, h, a_s, a_d, dout, budget_s=0.5,
                                            max_reps=5)
    assert time.perf_counter() - t0 < 5.0
    assert rate > 0 and "100.0% of E" in sample and "run(s)" in sample


def test_both_arms_print_the_same_config(capsys):
    args = bench.parse_args(["--impl", "reference", "--config", "1", "--steps", "1",
                             "--warmup", "0"])
    assert bench.run_reference(args, rank=0, world=1) == 0
    line = json.loads(capsys.readouterr().out)
    w, rp, ci, *_ = bench.load_workload(1)
    # the GPU arm prints workload_config(...) of the same workload and world
    assert line["config"] == bench.workload_config(w, rp, ci, 1)
    assert line["config"]["max_in_degree"] == int(np.diff(rp).max())
    assert "one thread" in line["cpu_baseline"]["sample"]


def test_default_workload_and_compact_lines():
    assert bench.DEFAULT_CONFIG == 5
    assert bench.sub_configs(bench.parse_args([])) == [3, 4, 6]
    assert bench.sub_configs(bench.parse_args(["--config", "2"])) == []
    assert bench.sub_configs(bench.parse_args(["--no-sub"])) == []
    assert bench.sub_configs(bench.parse_args(["--config", "2", "--sub", "3"])) == [3]
