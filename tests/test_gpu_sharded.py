"""The schedule build in two halves (tsa_block_sums, tsa_build_schedule_from_sums), as a
lane-sharded build runs it: block sums of each shard of lanes, concatenated in lane order, give
the oracle's CSR and salience (fp64 CPU, Kruskal) bit for bit, and so the one-call build's.
One GPU plays every shard here; tests/test_gpu_lane_sharded_procs.py runs the shards in
separate processes with a real exchange."""
import numpy as np
import pytest
import torch

import oracle
import topology_scheduled_gb300 as tsa
from topology_scheduled_gb300.workloads import WORKLOADS, make_qkv

pytestmark = pytest.mark.gpu
DEV = "cuda"


def _csr(rp, ci):
    rp = rp.cpu().numpy()
    return rp, ci.cpu().numpy()[: rp[-1]]


@pytest.mark.parametrize("name", ["b4h16s8192", "b2h32s32768"])
@pytest.mark.parametrize("tie", ["index", "content"])
@pytest.mark.parametrize("cuts", [(0, 64), (0, 40, 64), (0, 1, 17, 63, 64)])
def test_sharded_build_equals_one_call(name, tie, cuts):
    w = WORKLOADS[name]
    _, k, _ = make_qkv(w, seed=0, device=DEV)
    k = k.reshape(w.lanes, w.S, w.D)
    rp, ci, sal = tsa.tsa_build_schedule(k, w.block, w.sink, w.local_radius, w.topk, salience=True,
                                         tie_break=tie)
    shards = [tsa.tsa_block_sums(k[a:b].contiguous(), w.block) for a, b in zip(cuts[:-1], cuts[1:])]
    sums = torch.cat(shards, dim=0).contiguous()
    rp2, ci2, sal2 = tsa.tsa_build_schedule_from_sums(sums, w.block, w.sink, w.local_radius, w.topk,
                                                      salience=True, tie_break=tie)
    assert tsa.tsa_last_device_status() == 0
    a, b = _csr(rp, ci), _csr(rp2, ci2)
    assert np.array_equal(a[0], b[0]) and np.array_equal(a[1], b[1])
    assert torch.equal(sal.view(torch.int64), sal2.view(torch.int64))
    # against the oracle on the same keys (computed once per workload and tie rule)
    orp, oci, osal = _oracle_schedule(name, tie, k)
    assert np.array_equal(b[0], orp) and np.array_equal(b[1], oci)
    assert np.array_equal(sal2.cpu().numpy().view(np.uint64), osal.view(np.uint64))


_ORACLE = {}


def _oracle_schedule(name, tie, k):
    if (name, tie) not in _ORACLE:
        w = WORKLOADS[name]
        _ORACLE[(name, tie)] = oracle.build_schedule(k.cpu(), w.block, w.sink, w.local_radius, w.topk, tie=tie)
    return _ORACLE[(name, tie)]


def test_block_sums_are_the_block_sums():
    """Sequential binary64 sums of each block's tokens (exact for these inputs: 64 bf16 values)."""
    g = torch.Generator().manual_seed(3)
    k = torch.randn((3, 256, 64), generator=g).to(torch.bfloat16)
    got = tsa.tsa_block_sums(k.to(DEV), 64).cpu().numpy()
    x = k.double().numpy().reshape(3, 4, 64, 64)
    ref = np.zeros((3, 4, 64))
    for t in range(64):
        ref = ref + x[:, :, t, :]
    assert np.array_equal(got, ref)


def test_host_errors():
    L = tsa.lib()
    k = torch.zeros((2, 256, 64), dtype=torch.float16, device=DEV)
    part = torch.zeros((2, 4, 64), dtype=torch.float64, device=DEV)
    assert L.tsa_block_sums(k.data_ptr(), 0, 2, 256, 64, 64, part.data_ptr() + 4, None) == 1  # misaligned
    assert L.tsa_block_sums(k.data_ptr(), 0, 2, 0, 64, 64, part.data_ptr(), None) == 1        # empty
    rp = torch.zeros(5, dtype=torch.int32, device=DEV)
    ci = torch.zeros(16, dtype=torch.int32, device=DEV)
    ws = torch.zeros(256, dtype=torch.uint8, device=DEV)
    st = L.tsa_build_schedule_from_sums(part.data_ptr(), 2, 256, 64, 64, 1, 1, 2, 0, rp.data_ptr(),
                                        ci.data_ptr(), ci.numel(), None, ws.data_ptr(), ws.numel(), None)
    assert st == 5  # workspace too small
    st = L.tsa_build_schedule_from_sums(part.data_ptr(), 2, 256, 64, 64, 1, 1, 2, 7, rp.data_ptr(),
                                        ci.data_ptr(), ci.numel(), None, ws.data_ptr(), ws.numel(), None)
    assert st == 1  # unknown tie rule
