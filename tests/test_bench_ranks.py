"""The multi-process path of bench.py on the CPU: two gloo ranks combine their
step times the way the GPU replicas do (max over ranks, whole-job
throughput), and the reference arm leaves the work to rank 0."""
import os
import socket
import sys

import pytest
import torch.multiprocessing as mp

ROOT = os.path.dirname(os.path.dirname(os.path.abspath(__file__)))


def _free_port():
    with socket.socket() as s:
        s.bind(("127.0.0.1", 0))
        return s.getsockname()[1]


def _rank(rank, world, port, out):
    sys.path.insert(0, ROOT)
    import torch.distributed as dist
    import bench
    dist.init_process_group("gloo", init_method=f"tcp://127.0.0.1:{port}", rank=rank,
                            world_size=world)
    try:
        # rank r took (r + 1) ms per step and 10 - r ms per forward
        ms, fwd = bench.max_over_ranks([rank + 1.0, 10.0 - rank], world, "cpu")
        out[rank] = (ms, fwd, bench.job_rate(3e6, world, ms))
        dist.barrier()
    finally:
        dist.destroy_process_group()


def test_ranks_take_the_slowest_replica():
    world, port = 2, _free_port()
    with mp.Manager() as m:
        out = m.dict()
        mp.spawn(_rank, args=(world, port, out), nprocs=world, join=True)
        res = dict(out)
    for r in range(world):
        ms, fwd, rate = res[r]
        assert ms == 2.0 and fwd == 10.0
        assert rate == pytest.approx(world * 3e6 / 2e-3 / 1e9)


def test_single_rank_is_the_identity():
    sys.path.insert(0, ROOT)
    import bench
    assert bench.max_over_ranks([1.5, 2.5], 1, "cpu") == [1.5, 2.5]
    assert bench.job_rate(2e9, 1, 1000.0) == pytest.approx(2.0)


def test_reference_arm_other_ranks_exit_without_work(capsys):
    sys.path.insert(0, ROOT)
    import bench
    args = bench.parse_args(["--impl", "reference"])
    assert bench.run_reference(args, rank=1, world=2) == 0
    assert capsys.readouterr().out == ""
