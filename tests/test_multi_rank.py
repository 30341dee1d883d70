"""bench.py's multi-rank logic on CPU with the gloo backend (world size 2):
the timed region's max over ranks, the whole-job value and per-replica seeds.
The path has no data exchange (replicas only), so this host logic is all
there is to test for N > 1."""
import os
import socket

import pytest
import torch
import torch.distributed as dist
import torch.multiprocessing as mp


def _free_port():
    with socket.socket() as s:
        s.bind(("127.0.0.1", 0))
        return s.getsockname()[1]


def _worker(rank, world, port, out):
    os.environ.update(MASTER_ADDR="127.0.0.1", MASTER_PORT=str(port), RANK=str(rank), WORLD_SIZE=str(world))
    import bench
    dist.init_process_group("gloo", rank=rank, world_size=world)
    try:
        local_time = [0.75, 1.25][rank]
        worst = bench.max_over_ranks(local_time, dist, torch.device("cpu"))
        seeds = [None] * world
        dist.all_gather_object(seeds, bench.replica_seed(rank))
        out[rank] = (worst, seeds, bench.dist_env())
    finally:
        dist.destroy_process_group()


def test_two_replicas_take_the_slowest_and_draw_distinct_batches():
    world = 2
    port = _free_port()
    manager = mp.Manager()
    out = manager.dict()
    mp.spawn(_worker, args=(world, port, out), nprocs=world, join=True)
    for rank in range(world):
        worst, seeds, env = out[rank]
        assert worst == 1.25
        assert len(set(seeds)) == world
        assert env[0] == world and env[1] == rank


def test_whole_job_value_scales_with_replicas():
    import bench
    one = bench.replica_value(17.6e12, 10, 1, 0.1)
    two = bench.replica_value(17.6e12, 10, 2, 0.1)
    assert two == pytest.approx(2 * one)
    assert one == pytest.approx(17.6e12 * 10 / 0.1 / 1e12)
