"""The N > 1 paths on CPU with gloo ranks: bench.py's aggregation (each rank its own independent
problem: the slowest rank's time, the sum of the ranks' work), and the exchange of the
lane-sharded schedule build (per-lane block sums gathered in global lane order)."""
import os
import socket

import numpy as np
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
    with mp.get_context("spawn").Manager() as m:
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


def _block_sums_np(k_lanes: torch.Tensor, block: int):
    """Sequential binary64 block sums (tokens ascending) of [lanes, S, D] 16-bit keys."""
    x = k_lanes.double().numpy()
    L, S, D = x.shape
    x = x.reshape(L, S // block, block, D)
    acc = np.zeros((L, S // block, D))
    for t in range(block):
        acc = acc + x[:, :, t, :]
    return acc


def _shard_rank(rank, world, port, cuts, out):
    os.environ.update(MASTER_ADDR="127.0.0.1", MASTER_PORT=str(port))
    dist.init_process_group("gloo", rank=rank, world_size=world)
    from topology_scheduled_gb300.distributed import gather_block_sums
    g = torch.Generator().manual_seed(11)
    k = torch.randn((7, 512, 32), generator=g).to(torch.bfloat16)  # every rank draws the same keys
    mine = torch.as_tensor(_block_sums_np(k[cuts[rank]:cuts[rank + 1]], 64))
    out[rank] = gather_block_sums(mine).numpy().tobytes()
    dist.barrier()
    dist.destroy_process_group()


@pytest.mark.parametrize("cuts", [(0, 4, 7), (0, 1, 7), (0, 7, 7)])
def test_lane_sharded_block_sums_gather_in_lane_order(cuts):
    """Uneven shards (one empty): every rank ends with all lanes' block sums in global lane
    order, bit for bit, and their ascending lane sum / (block * lanes) is the oracle's
    lane-mean centroid."""
    world = 2
    port = _free_port()
    with mp.get_context("spawn").Manager() as m:
        out = m.dict()
        mp.spawn(_shard_rank, args=(world, port, cuts, out), nprocs=world, join=True)
        res = dict(out)
    g = torch.Generator().manual_seed(11)
    k = torch.randn((7, 512, 32), generator=g).to(torch.bfloat16)
    full = _block_sums_np(k, 64)
    for r in range(world):
        assert res[r] == full.tobytes()
    import oracle
    acc = np.zeros(full.shape[1:])
    for lane in range(full.shape[0]):
        acc = acc + full[lane]
    assert np.array_equal(acc / (64 * 7), oracle.centroids(k, 64))
