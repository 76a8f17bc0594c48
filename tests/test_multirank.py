"""The N-GPU bench path runs independent replicas: per-rank timings are combined by a max over ranks
and the job throughput counts every replica's tokens. Checked with two gloo ranks on CPU."""
import os
import socket

import pytest
import torch.distributed as dist
import torch.multiprocessing as mp

import bench


def _free_port():
    with socket.socket() as s:
        s.bind(("127.0.0.1", 0))
        return s.getsockname()[1]


def _rank(rank, world, port, out):
    os.environ.update(MASTER_ADDR="127.0.0.1", MASTER_PORT=str(port))
    dist.init_process_group("gloo", rank=rank, world_size=world)
    try:
        mine = [10.0 + rank, 20.0 - rank, 5.0 * (rank + 1)]
        out[rank] = bench.max_over_ranks(mine, dist, "cpu")
        dist.barrier()
    finally:
        dist.destroy_process_group()


def test_max_over_two_gloo_ranks():
    world = 2
    port = _free_port()
    with mp.Manager() as m:
        out = m.dict()
        mp.spawn(_rank, args=(world, port, out), nprocs=world, join=True)
        got = dict(out)
    assert got[0] == got[1] == [11.0, 20.0, 10.0]


def test_single_rank_and_job_throughput():
    assert bench.max_over_ranks([1.0, 2.0]) == [1.0, 2.0]
    assert bench.job_tokens_per_s(1, 16384, 10.0) == pytest.approx(1638400.0)
    assert bench.job_tokens_per_s(4, 16384, 10.0) == pytest.approx(4 * 1638400.0)
