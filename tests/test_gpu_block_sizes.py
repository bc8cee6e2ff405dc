"""Scheduled attention over CSRs of 32- and 128-token blocks, on the GPU, element by element
against the oracle at the same block (same tolerance as test_gpu_attention).  The kernel works
in 64-token key steps: a 128-token key block is walked as two of them, a pair of 32-token key
blocks shares one with a per-(query quarter, key half) mask.  The cases cover dense, topology
and random CSRs, lengths with a partial last block (and a last 128-block holding a single
64-token block), both dtypes and head dims, and the schedule builder feeding the kernel."""
import numpy as np
import pytest
import torch

import oracle
import topology_scheduled_gb300 as tsa
from test_gpu_attention import assert_close
from topology_scheduled_gb300.workloads import random_density_csr

pytestmark = pytest.mark.gpu
DEV = "cuda"


def _run(q, k, v, rp, ci, scale, block):
    rp_d = torch.as_tensor(np.asarray(rp), dtype=torch.int32, device=DEV)
    ci_d = torch.as_tensor(np.asarray(ci) if len(ci) else np.zeros(1, np.int32), dtype=torch.int32, device=DEV)
    out, lse = tsa.tsa_scheduled_attention_fwd(q.to(DEV), k.to(DEV), v.to(DEV), rp_d, ci_d, scale, block=block)
    assert tsa.tsa_last_device_status() == 0
    return out.cpu(), lse.cpu()


@pytest.mark.parametrize("L,S,D,dtype", [(1, 1024, 64, torch.float16), (2, 2048, 128, torch.bfloat16),
                                         (3, 1000, 64, torch.bfloat16), (1, 130, 128, torch.float16),
                                         (2, 4096 + 64, 128, torch.float16)])
@pytest.mark.parametrize("kind", ["dense", "topology", "random"])
@pytest.mark.parametrize("block", [32, 128])
def test_block_matches_oracle(L, S, D, dtype, kind, block):
    g = torch.Generator().manual_seed(S + D + L)
    q, k, v = (torch.randn((L, S, D), generator=g).to(dtype) for _ in range(3))
    nb = -(-S // block)
    if kind == "dense":
        rp, ci = oracle.dense_causal_csr(nb)
    elif kind == "topology":
        rp, ci, _ = oracle.build_schedule(k, block, 1, 1, 2)
    else:
        rp, ci = random_density_csr(nb, 0.3, S)
    scale = D ** -0.5
    out, lse = _run(q, k, v, rp, ci, scale, block)
    ref, ref_lse = oracle.attention(q, k, v, rp, ci, block, scale, nthreads=8, return_lse=True)
    assert_close(out.double().numpy(), ref, dtype)
    u = 2.0 ** -11 if dtype == torch.float16 else 2.0 ** -8
    fin = np.isfinite(ref_lse)
    assert np.array_equal(np.isfinite(lse.double().numpy()), fin)
    assert np.abs(lse.double().numpy()[fin] - ref_lse[fin]).max() <= u


@pytest.mark.parametrize("block", [32, 128])
def test_schedule_from_the_builder(block):
    g = torch.Generator().manual_seed(2)
    L, S, D = 4, 4096, 64
    q, k, v = (torch.randn((L, S, D), generator=g).to(torch.float16) for _ in range(3))
    rp, ci = tsa.tsa_build_schedule(k.to(DEV), block, 1, 2, 3)
    orp, oci, _ = oracle.build_schedule(k, block, 1, 2, 3)
    assert np.array_equal(rp.cpu().numpy(), orp) and np.array_equal(ci.cpu().numpy()[: orp[-1]], oci)
    out = tsa.tsa_scheduled_attention(q.to(DEV), k.to(DEV), v.to(DEV), rp, ci, D ** -0.5, block=block)
    assert tsa.tsa_last_device_status() == 0
    ref = oracle.attention(q, k, v, orp, oci, block, D ** -0.5, nthreads=8)
    assert_close(out.cpu().double().numpy(), ref, torch.float16)


def test_other_blocks_unsupported():
    x = torch.zeros((1, 256, 64), dtype=torch.float16, device=DEV)
    rp, ci = tsa.tsa_dense_causal_csr(256, 16)
    with pytest.raises(tsa.TsaError):
        tsa.tsa_scheduled_attention(x, x.clone(), x.clone(), rp, ci, 0.125, block=16)
