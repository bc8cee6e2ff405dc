"""The N > 1 path of bench.py on CPU: two gloo ranks, each with its own independent problem,
aggregate to the slowest rank's time and the sum of the ranks' work (weak scaling)."""
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


def _rank(rank, world, port, out):
    os.environ.update(MASTER_ADDR="127.0.0.1", MASTER_PORT=str(port))
    dist.init_process_group("gloo", rank=rank, world_size=world)
    import bench
    elapsed, flops = bench.aggregate_over_ranks(10.0 + rank, 1e12 * (rank + 1), torch.device("cpu"), world)
    out[rank] = (elapsed, flops)
    dist.barrier()
    dist.destroy_process_group()


def test_two_ranks_take_max_time_and_sum_work():
    world = 2
    port = _free_port()
    with mp.Manager() as m:
        out = m.dict()
        mp.spawn(_rank, args=(world, port, out), nprocs=world, join=True)
        res = dict(out)
    for r in range(world):
        assert res[r] == (11.0, 3e12)


def test_single_rank_is_identity():
    import bench
    assert bench.aggregate_over_ranks(5.0, 2.0, torch.device("cpu"), 1) == (5.0, 2.0)
    assert bench.launches_per_step("topology") == 5 and bench.launches_per_step("dense") == 1
    assert bench.launches_per_step("topology-content") == 7
    assert bench.launches_per_step("segment:512") == 3 and bench.launches_per_step("density:0.1") == 1
