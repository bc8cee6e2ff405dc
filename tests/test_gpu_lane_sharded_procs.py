"""The lane-sharded path end to end in two processes sharing the one GPU: each process holds a
contiguous run of the lanes (uneven cuts, one of them empty), computes its lanes' block sums on
the GPU, the sums are exchanged in lane order over gloo (through host memory), each process
builds the CSR from all of them and runs the attention on its own lanes.

Checked against the oracle (fp64 CPU, Kruskal): every process's CSR and salience equal the
oracle's bit for bit; each process's O equals, bit for bit, the single-process O of the same
lanes (the attention is independent per lane) and is within tolerance of the oracle on sampled
rows.  The processes' kernels never wait on one another: the exchange is a host collective
between launches."""
import datetime
import os
import socket

import numpy as np
import pytest
import torch
import torch.distributed as dist
import torch.multiprocessing as mp

import oracle
from topology_scheduled_gb300.workloads import WORKLOADS, Workload, make_qkv

pytestmark = pytest.mark.gpu

CASES = {
    "b4h16s8192": (WORKLOADS["b4h16s8192"], "index", (0, 23, 64)),
    # partial last block, bf16, D 128, content ties, an empty first shard
    "b1h5s3000": (Workload("b1h5s3000", 1, 5, 3000, 128, torch.bfloat16, "clustered_geometric", n_means=8,
                           span=200, sink=2, local_radius=3, topk=4), "content", (0, 0, 5)),
}
from _tol import assert_close  # noqa: E402


def _free_port():
    with socket.socket() as s:
        s.bind(("127.0.0.1", 0))
        return s.getsockname()[1]


def _proc(rank, world, port, case, outdir):
    os.environ.update(MASTER_ADDR="127.0.0.1", MASTER_PORT=str(port))
    dist.init_process_group("gloo", rank=rank, world_size=world, timeout=datetime.timedelta(seconds=180))
    import topology_scheduled_gb300 as tsa
    from topology_scheduled_gb300.distributed import build_schedule_lane_sharded
    torch.cuda.set_device(0)
    w, tie, cuts = CASES[case]
    q, k, v = (x.reshape(w.lanes, w.S, w.D) for x in make_qkv(w, seed=0, device="cpu"))
    lo, hi = cuts[rank], cuts[rank + 1]
    ql, kl, vl = (x[lo:hi].contiguous().to("cuda") for x in (q, k, v))
    rp, ci, sal = build_schedule_lane_sharded(kl, w.block, w.sink, w.local_radius, w.topk, tie_break=tie,
                                              salience=True)
    out = tsa.tsa_scheduled_attention(ql, kl, vl, rp, ci, w.scale) if hi > lo else ql
    status = tsa.tsa_last_device_status()
    rp_h = rp.cpu().numpy()
    np.savez(os.path.join(outdir, f"rank{rank}.npz"), rp=rp_h, ci=ci.cpu().numpy()[: rp_h[-1]],
             sal=sal.cpu().numpy(), out=out.cpu().view(torch.int16).numpy(), status=np.int64(status))
    dist.barrier()
    dist.destroy_process_group()


@pytest.mark.parametrize("case", sorted(CASES))
def test_two_processes_one_gpu(case, tmp_path):
    import topology_scheduled_gb300 as tsa
    w, tie, cuts = CASES[case]
    world = len(cuts) - 1
    mp.start_processes(_proc, args=(world, _free_port(), case, str(tmp_path)), nprocs=world, join=True,
                       start_method="spawn")
    q, k, v = (x.reshape(w.lanes, w.S, w.D) for x in make_qkv(w, seed=0, device="cpu"))
    orp, oci, osal = oracle.build_schedule(k, w.block, w.sink, w.local_radius, w.topk, tie=tie)
    # the single-process O over all lanes, on the oracle's CSR
    rp_d = torch.as_tensor(orp, device="cuda")
    ci_d = torch.as_tensor(oci if len(oci) else np.zeros(1, np.int32), device="cuda")
    full = tsa.tsa_scheduled_attention(q.cuda(), k.cuda(), v.cuda(), rp_d, ci_d, w.scale).cpu()
    assert tsa.tsa_last_device_status() == 0
    rng = np.random.default_rng(1)
    for r in range(world):
        got = np.load(tmp_path / f"rank{r}.npz")
        assert int(got["status"]) == 0
        assert np.array_equal(got["rp"], orp) and np.array_equal(got["ci"], oci)
        assert np.array_equal(got["sal"].view(np.uint64), osal.view(np.uint64))
        lo, hi = cuts[r], cuts[r + 1]
        if hi == lo:
            continue
        mine = torch.from_numpy(got["out"]).view(w.dtype)
        assert torch.equal(mine.view(torch.int16), full[lo:hi].contiguous().view(torch.int16))
        lanes = rng.integers(lo, hi, 96)
        toks = np.concatenate([np.arange(0, 32), np.arange(w.S - 32, w.S), rng.integers(0, w.S, 32)])
        ref = oracle.attention(q, k, v, orp, oci, w.block, w.scale, lanes=lanes.astype(np.int64),
                               tokens=toks.astype(np.int64), nthreads=8)
        sel = mine[torch.as_tensor(lanes - lo), torch.as_tensor(toks)].double().numpy()
        assert_close(sel, ref, w.dtype)
