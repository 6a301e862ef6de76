"""The benchmark's multi-rank host logic on CPU (gloo, world size 2): each
rank runs an independent replica, the job time is the slowest rank's, and
the job throughput counts every rank's tokens."""
import os
import socket

import pytest
import torch
import torch.distributed as dist
import torch.multiprocessing as mp


def _free_port():
    s = socket.socket()
    s.bind(("127.0.0.1", 0))
    port = s.getsockname()[1]
    s.close()
    return port


def _worker(rank, world, port, out):
    os.environ.update(MASTER_ADDR="127.0.0.1", MASTER_PORT=str(port), RANK=str(rank),
                      WORLD_SIZE=str(world), LOCAL_RANK=str(rank))
    dist.init_process_group("gloo", rank=rank, world_size=world)
    import bench
    ms = 100.0 + 50.0 * rank          # rank 1 is the slow one
    got = bench.max_over_ranks(ms)
    tps = bench.job_tokens_per_s(1000, world, 10, got)
    w, r, lr = bench.dist_env()
    out[rank] = (got, tps, w, r, lr)
    dist.barrier()
    dist.destroy_process_group()


def test_two_rank_max_and_aggregate():
    world = 2
    mgr = mp.get_context("spawn").Manager()
    out = mgr.dict()
    mp.start_processes(_worker, args=(world, _free_port(), out), nprocs=world, join=True,
                       start_method="spawn")
    for rank in range(world):
        got, tps, w, r, lr = out[rank]
        assert got == 150.0
        assert tps == pytest.approx(1000 * 2 * 10 / 0.150)
        assert (w, r, lr) == (2, rank, rank)


def test_single_process_is_identity():
    import bench
    assert bench.max_over_ranks(12.5) == 12.5
