"""The multi-rank path of the benchmark (independent replicas, one per GPU):
the job's time is the slowest rank's, the throughput sums the replicas, and
each rank draws its own inputs.  Two gloo ranks on the CPU."""
import os
import socket

import numpy as np
import pytest
import torch
import torch.distributed as dist
import torch.multiprocessing as mp

import bench


def _free_port():
    s = socket.socket()
    s.bind(("127.0.0.1", 0))
    port = s.getsockname()[1]
    s.close()
    return port


def _rank_main(rank, world, port, out):
    os.environ.update(MASTER_ADDR="127.0.0.1", MASTER_PORT=str(port), RANK=str(rank), WORLD_SIZE=str(world))
    dist.init_process_group("gloo", rank=rank, world_size=world)
    try:
        local_ms = [120.0, 150.0][rank]                     # rank 1 is the slower replica
        dist.barrier()
        ms = bench.max_over_ranks(local_ms, dist, "cpu")
        value = bench.replica_throughput(world, 1, 1000, ms)
        idx, _ = bench.draw_routings(4, 384, 6, 1, seed=rank)
        gathered = [torch.zeros(4 * 6, dtype=torch.int64) for _ in range(world)]
        dist.all_gather(gathered, torch.from_numpy(idx.reshape(-1).astype(np.int64)))
        out[rank] = (ms, value, bool(torch.equal(gathered[0], gathered[1])))
    finally:
        dist.destroy_process_group()


def test_two_gloo_ranks_take_the_slowest_time_and_sum_replicas():
    world = 2
    with mp.Manager() as m:
        out = m.dict()
        mp.spawn(_rank_main, args=(world, _free_port(), out), nprocs=world, join=True)
        res = dict(out)
    for rank in range(world):
        ms, value, same_inputs = res[rank]
        assert ms == 150.0
        assert value == pytest.approx(2 * 1000 / 0.150)
        assert not same_inputs                              # each replica draws its own routing


def test_single_rank_needs_no_process_group():
    assert bench.max_over_ranks(12.5, None, "cpu") == 12.5
    assert bench.replica_throughput(1, 64, 10, 500.0) == pytest.approx(1280.0)
