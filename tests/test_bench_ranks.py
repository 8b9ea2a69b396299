"""bench.py's multi-rank aggregation on CPU: two gloo ranks with different
step times report the slowest rank's time and all ranks' samples."""
import os
import socket
import sys

import pytest
import torch
import torch.distributed as dist
import torch.multiprocessing as mp

ROOT = os.path.dirname(os.path.dirname(os.path.abspath(__file__)))


def _free_port():
    with socket.socket() as s:
        s.bind(("127.0.0.1", 0))
        return s.getsockname()[1]


def _rank(rank, world, port, out):
    sys.path.insert(0, ROOT)
    import bench
    os.environ.update(MASTER_ADDR="127.0.0.1", MASTER_PORT=str(port))
    dist.init_process_group("gloo", rank=rank, world_size=world)
    local_ms = 100.0 + 50.0 * rank                     # rank 1 is the slow one
    job_ms = bench.max_over_ranks(local_ms, dist, torch.device("cpu"))
    rate = bench.whole_job_rate(world, 1_000_000, 10, job_ms)
    out[rank] = (job_ms, rate)
    dist.barrier()
    dist.destroy_process_group()


def test_two_gloo_ranks_take_the_slowest_time_and_all_samples():
    port = _free_port()
    with mp.Manager() as m:
        out = m.dict()
        mp.spawn(_rank, args=(2, port, out), nprocs=2, join=True)
        res = dict(out)
    for r in (0, 1):
        job_ms, rate = res[r]
        assert job_ms == pytest.approx(150.0)
        # 2 ranks x 10 steps x 1e6 samples in 0.15 s
        assert rate == pytest.approx(2 * 10 * 1e6 / 0.15 / 1e9)


def test_single_process_rate_needs_no_collective():
    sys.path.insert(0, ROOT)
    import bench
    assert bench.max_over_ranks(12.5) == 12.5
    assert bench.whole_job_rate(1, 16_908_288, 200, 400.0) == pytest.approx(8.454144)
