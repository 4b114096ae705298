"""The benchmark's multi-rank bookkeeping on CPU: two gloo ranks report
different step times; the job's step time is the slowest rank's, and the
whole-job throughput counts every rank's bytes over that time."""
import os
import socket

import pytest

torch = pytest.importorskip("torch")
import torch.distributed as dist  # noqa: E402
import torch.multiprocessing as mp  # noqa: E402


def _free_port() -> int:
    with socket.socket() as s:
        s.bind(("127.0.0.1", 0))
        return s.getsockname()[1]


def _rank(rank, world, port, out):
    os.environ.update(MASTER_ADDR="127.0.0.1", MASTER_PORT=str(port))
    dist.init_process_group("gloo", rank=rank, world_size=world)
    try:
        import bench

        ms = bench.slowest_rank_ms(1.0 + rank * 0.25, world)
        out[rank] = (ms, bench.whole_job_tbps(2e9, ms, world))
    finally:
        dist.destroy_process_group()


def test_two_gloo_ranks_take_the_slowest_rank():
    world = 2
    with mp.Manager() as man:
        out = man.dict()
        mp.spawn(_rank, args=(world, _free_port(), out), nprocs=world, join=True)
        res = dict(out)
    assert res[0][0] == res[1][0] == 1.25
    assert abs(res[0][1] - 2 * 2e9 / 1.25e-3 / 1e12) < 1e-12


def test_single_rank_needs_no_process_group():
    import bench

    assert bench.slowest_rank_ms(3.5, 1) == 3.5
    assert bench.whole_job_tbps(1e12, 1000.0, 1) == 1.0
