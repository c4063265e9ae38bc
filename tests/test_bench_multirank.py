"""The bench's multi-rank host logic on CPU: two gloo ranks on this host.

With N ranks the bench runs one replica batch per rank (sequences are
independent; no collective on the data path) and reports the whole job:
every rank's tokens over the slowest rank's time.  These tests run that
aggregation with world size 2 over gloo (127.0.0.1), no GPU.
"""
import os
import socket

import pytest
import torch.distributed as dist
import torch.multiprocessing as mp

import bench


def _free_port():
    s = socket.socket()
    s.bind(("127.0.0.1", 0))
    port = s.getsockname()[1]
    s.close()
    return port


def _rank_main(rank, world, port, times, out):
    os.environ.update(MASTER_ADDR="127.0.0.1", MASTER_PORT=str(port),
                      RANK=str(rank), WORLD_SIZE=str(world))
    dist.init_process_group("gloo", rank=rank, world_size=world)
    try:
        total = bench.max_over_ranks(dist, times[rank], "cpu")
        out[rank] = (total, bench.throughput(64, world, total, 10))
        dist.barrier()
    finally:
        dist.destroy_process_group()


@pytest.mark.parametrize("times", [(12.0, 15.0), (15.0, 12.0), (9.5, 9.5)])
def test_two_ranks_take_the_slowest_time(times):
    world = 2
    out = mp.Manager().dict()
    mp.spawn(_rank_main, args=(world, _free_port(), times, out), nprocs=world, join=True)
    slowest = max(times)
    for r in range(world):
        total, value = out[r]
        assert total == slowest
        # 64 tokens per rank per step, 10 steps: 128 tokens per slowest-step time
        assert value == pytest.approx(128 / (slowest / 10 / 1e3))


def test_single_rank_is_its_own_time():
    assert bench.max_over_ranks(None, 7.25, "cpu") == 7.25
    assert bench.throughput(64, 1, 10.0, 10) == pytest.approx(64e3)
