"""Host logic of the multi-GPU benchmark path (weak scaling over independent
heads, no collective on the data path), run as two gloo ranks on the CPU."""
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
    os.environ.update(MASTER_ADDR="127.0.0.1", MASTER_PORT=str(port), RANK=str(rank),
                      WORLD_SIZE=str(world), LOCAL_RANK=str(rank))
    import bench

    dist.init_process_group("gloo", rank=rank, world_size=world)
    try:
        r, w, lr = bench.dist_env()
        assert (r, w, lr) == (rank, world, rank)
        ms = 2.0 + rank  # rank 1 is the slowest
        mx = bench.max_over_ranks(ms, w)
        bench.barrier(w)
        value = bench.aggregate_value(1000, w, mx / 1e3)
        out[rank] = (bench.rank_seed(7, rank), mx, value)
    finally:
        dist.destroy_process_group()


def test_two_ranks_gloo():
    world = 2
    port = _free_port()
    with mp.Manager() as m:
        out = m.dict()
        mp.spawn(_worker, args=(world, port, out), nprocs=world, join=True)
        res = dict(out)
    seeds = {res[r][0] for r in range(world)}
    assert len(seeds) == world                      # each rank draws its own copy
    assert all(res[r][1] == 3.0 for r in range(world))   # max over ranks
    assert all(abs(res[r][2] - 2 * 1000 / 3e-3) < 1e-6 for r in range(world))


def test_single_rank_is_plain():
    import bench

    assert bench.max_over_ranks(1.5, 1) == 1.5
    assert bench.aggregate_value(10, 1, 0.5) == 20.0
