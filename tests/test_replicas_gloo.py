"""The N > 1 path of the benchmark (independent replicas, one per rank): the
job's time is the slowest rank's and its throughput counts every rank's
work.  Run as two gloo ranks on the CPU."""

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


def _rank_main(rank, world, port, times, out):
    import bench

    os.environ.update(MASTER_ADDR="127.0.0.1", MASTER_PORT=str(port), RANK=str(rank),
                      WORLD_SIZE=str(world))
    dist.init_process_group("gloo", rank=rank, world_size=world)
    try:
        got = bench.slowest_rank(dist, times[rank], "cpu")
        out[rank] = got
        dist.barrier()
    finally:
        dist.destroy_process_group()


def test_slowest_rank_and_replica_throughput_two_gloo_ranks():
    import bench

    times = {0: [1.5, 7.0], 1: [2.25, 3.0]}
    with mp.Manager() as m:
        out = m.dict()
        mp.spawn(_rank_main, args=(2, _free_port(), times, out), nprocs=2, join=True)
        res = dict(out)
    assert res[0] == res[1] == [2.25, 7.0]          # entry-wise max over ranks, on every rank
    # Two replicas of 1e12 FLOP each in 2.25 ms: 888.9 TFLOP/s for the job.
    assert abs(bench.replica_throughput(1e12, 2, 2.25) - 2e12 / 2.25e-3 / 1e12) < 1e-9
    assert bench.slowest_rank(None, [4.0, 5.0], "cpu") == [4.0, 5.0]
