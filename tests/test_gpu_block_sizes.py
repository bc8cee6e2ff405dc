"""Scheduled attention over CSRs of 32- and 128-token blocks, on the GPU, element by element
against the oracle at the same block (same tolerance as test_gpu_attention).  The kernel works
in 64-token key steps: a 128-token key block is walked as two of them, a pair of 32-token key
blocks shares one with a per-(query quarter, key half) mask.  The cases cover dense, topology
and random CSRs, lengths with a partial last block (and a last 128-block holding a single
64-token block), both dtypes and head dims, and the schedule builder feeding the kernel.  The
backward pass takes 128-token CSRs (expanded to 64-token blocks on the GPU) and refuses
32-token ones."""
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


@pytest.mark.parametrize("L,S,D,dtype", [(1, 1024, 64, torch.float16), (2, 1000, 128, torch.bfloat16),
                                         (1, 130, 128, torch.float16), (2, 4096 + 64, 64, torch.bfloat16)])
@pytest.mark.parametrize("kind", ["dense", "topology", "random", "holes"])
def test_backward_block128_matches_oracle(L, S, D, dtype, kind):
    """dQ, dK, dV over a CSR of 128-token blocks (expanded on the GPU to the 64-token CSR with
    the same allowed keys) against the oracle at block 128, test_gpu_backward's tolerance."""
    from test_gpu_backward import ETA, U, _bounds, _close
    g = torch.Generator().manual_seed(S + 7 * D + L)
    q, k, v, dO = (torch.randn((L, S, D), generator=g).to(dtype) for _ in range(4))
    nb = -(-S // 128)
    if kind == "dense":
        rp, ci = oracle.dense_causal_csr(nb)
    elif kind == "topology":
        rp, ci, _ = oracle.build_schedule(k, 128, 1, 1, 2)
    elif kind == "random":
        rp, ci = random_density_csr(nb, 0.3, S)
    else:  # an empty row, a row without its diagonal, the last row holding only its diagonal
        rng = np.random.default_rng(S)
        rows = [sorted(set(rng.choice(i + 1, size=rng.integers(1, i + 2), replace=False).tolist()))
                for i in range(nb)]
        rows[min(1, nb - 1)] = []
        if nb > 2:
            rows[2] = [0]
        rows[-1] = [nb - 1]
        rp = np.zeros(nb + 1, np.int32)
        rp[1:] = np.cumsum([len(r) for r in rows])
        ci = np.array([j for r in rows for j in r], np.int32)
    scale = D ** -0.5
    rpd = torch.as_tensor(np.asarray(rp), dtype=torch.int32, device=DEV)
    cid = torch.as_tensor(np.asarray(ci) if len(ci) else np.zeros(1, np.int32), dtype=torch.int32, device=DEV)
    O, lse = tsa.tsa_scheduled_attention_fwd(q.to(DEV), k.to(DEV), v.to(DEV), rpd, cid, scale, block=128)
    grads = tsa.tsa_scheduled_attention_backward(q.to(DEV), k.to(DEV), v.to(DEV), O, dO.to(DEV), lse, rpd, cid,
                                                 scale, block=128)
    assert tsa.tsa_last_device_status() == 0
    refs = oracle.attention_backward(q, k, v, dO, rp, ci, 128, scale, nthreads=8)
    bounds = _bounds(q, k, v, dO, rp, ci, scale, U[dtype], ETA[dtype], block=128)
    for name, got, ref, b in zip(("dQ", "dK", "dV"), grads, refs, bounds):
        _close(got, ref, U[dtype], f"{kind} {name}", b, ETA[dtype])


def test_backward_block128_bad_schedule_is_reported():
    x = torch.zeros((1, 256, 64), dtype=torch.float16, device=DEV)
    lse = torch.zeros((1, 256), dtype=torch.float32, device=DEV)
    rp = torch.tensor([0, 1, 3], dtype=torch.int32, device=DEV)
    ci = torch.tensor([1, 0, 1], dtype=torch.int32, device=DEV)  # row 0 names block 1 > 0
    tsa.tsa_scheduled_attention_backward(x, x, x, x, x, lse, rp, ci, 0.125, block=128)
    assert tsa.tsa_last_device_status() == 8  # TSA_ERR_BAD_SCHEDULE


def test_backward_block32_is_unsupported():
    x = torch.zeros((1, 256, 64), dtype=torch.float16, device=DEV)
    lse = torch.zeros((1, 256), dtype=torch.float32, device=DEV)
    rp, ci = tsa.tsa_dense_causal_csr(256, 32)
    with pytest.raises(tsa.TsaError) as e:
        tsa.tsa_scheduled_attention_backward(x, x, x, x, x, lse, rp, ci, 0.125, block=32)
    assert e.value.status == 2


def test_autograd_block128_equals_explicit_calls():
    from topology_scheduled_gb300.autograd import scheduled_attention
    g = torch.Generator().manual_seed(9)
    L, S, D = 2, 640, 64
    q, k, v, dO = (torch.randn((L, S, D), generator=g).to(torch.bfloat16).to(DEV) for _ in range(4))
    rp, ci = tsa.tsa_dense_causal_csr(S, 128)
    qa, ka, va = (x.clone().requires_grad_(True) for x in (q, k, v))
    out = scheduled_attention(qa, ka, va, rp, ci, 0.125, block=128)
    out.backward(dO)
    O, lse = tsa.tsa_scheduled_attention_fwd(q, k, v, rp, ci, 0.125, block=128)
    dq, dk, dv = tsa.tsa_scheduled_attention_backward(q, k, v, O, dO, lse, rp, ci, 0.125, block=128)
    assert torch.equal(out, O)
    assert torch.equal(qa.grad, dq) and torch.equal(ka.grad, dk) and torch.equal(va.grad, dv)
