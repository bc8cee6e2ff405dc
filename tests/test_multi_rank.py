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


def _sharded_driver_rank(rank, world, port, out):
    """bench.py's lane-sharded build driver on a gloo rank, with CPU stand-ins for the three
    library calls: this rank's block sums, the real exchange, and the oracle's schedule from
    the gathered sums."""
    os.environ.update(MASTER_ADDR="127.0.0.1", MASTER_PORT=str(port))
    dist.init_process_group("gloo", rank=rank, world_size=world)
    import bench
    import oracle
    from topology_scheduled_gb300.distributed import gather_block_sums
    from topology_scheduled_gb300.workloads import Workload
    w = Workload("t", 1, 3, 512, 32, torch.bfloat16, sink=1, local_radius=1, topk=2)
    # the whole problem is the ranks' shards in rank order; every rank draws all of them here
    g = torch.Generator().manual_seed(5)
    k_all = (torch.randn((world * w.lanes, w.S, w.D), generator=g) * 3).to(torch.bfloat16)
    k_mine = k_all[rank * w.lanes:(rank + 1) * w.lanes]

    def from_sums(every, rp, ci):
        full = every.numpy()
        acc = np.zeros(full.shape[1:])
        for lane in range(full.shape[0]):
            acc = acc + full[lane]
        sal, _ = oracle.salience(acc / (w.block * full.shape[0]))
        r, c = oracle.topology_csr(sal, w.sink, w.local_radius, w.topk)
        rp[:] = torch.as_tensor(r)
        ci[: len(c)] = torch.as_tensor(c)

    build = bench.lane_sharded_builder(
        w, k_mine, "topology",
        block_sums=lambda kk: torch.as_tensor(_block_sums_np(kk, w.block)),
        from_sums=from_sums,
        gather=lambda sums, counts: gather_block_sums(sums, counts=counts),
        world=world, rank=rank)
    rp = torch.zeros(w.nb + 1, dtype=torch.int32)
    ci = torch.full((oracle.max_nnz(w.nb, w.sink, w.local_radius, w.topk),), -1, dtype=torch.int32)
    build(rp, ci)
    out[rank] = (rp.numpy().tobytes(), ci.numpy()[: int(rp[-1])].tobytes())
    dist.barrier()
    dist.destroy_process_group()


def test_lane_sharded_bench_driver_builds_the_oracle_schedule():
    """Two gloo ranks run bench.py's lane-sharded build driver: both end with the CSR the oracle
    builds from all lanes' keys at once."""
    world = 2
    port = _free_port()
    with mp.get_context("spawn").Manager() as m:
        out = m.dict()
        mp.spawn(_sharded_driver_rank, args=(world, port, out), nprocs=world, join=True)
        res = dict(out)
    import bench
    import oracle
    g = torch.Generator().manual_seed(5)
    k_all = (torch.randn((world * 3, 512, 32), generator=g) * 3).to(torch.bfloat16)
    rp, ci, _ = oracle.build_schedule(k_all, 64, 1, 1, 2)
    for r in range(world):
        got_rp = np.frombuffer(res[r][0], dtype=np.int32)
        got_ci = np.frombuffer(res[r][1], dtype=np.int32)
        assert bench.check_csr_equal(got_rp, got_ci, rp, ci)


def test_check_csr_equal_and_peak_choice():
    import bench
    rp, ci = np.array([0, 1, 3]), np.array([0, 0, 1, 99])
    assert bench.check_csr_equal(rp, ci, rp, ci[:3])
    assert not bench.check_csr_equal(rp, np.array([0, 1, 1]), rp, ci)
    assert not bench.check_csr_equal(np.array([0, 1, 2]), ci, rp, ci)
    peaks = {"bf16_tflops": 1900.0, "bf16_tflops_sustained": 1700.0, "hbm_gbs": 6800.0}
    assert bench.tensor_peak(peaks, "measured", 23.0)[0] == 1900.0
    assert bench.tensor_peak(peaks, "measured", 1500.0)[0] == 1700.0
