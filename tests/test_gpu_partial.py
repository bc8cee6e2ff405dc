"""Sequences whose length is not a multiple of 64 (a partial last block), on the GPU.

Schedule builder and dense CSR: bit-exact against the oracle (nb = ceil(S / 64), the last
block's centroid averages the tokens it holds).  Attention: element by element against the
oracle within the tolerance of test_gpu_attention (2e-3 fp16, 1e-2 bf16; the bound plus half an
output ulp where the format is coarser), every lane compared, so a partial block that wrote past its lane's last
row into the next lane would show; rows past the last lane's end and log-sum-exp entries past
the end stay untouched.  Backward: dQ, dK, dV against the oracle within test_gpu_backward's
tolerance, with the same untouched-tail check.
"""
import numpy as np
import pytest
import torch

import oracle
import topology_scheduled_gb300 as tsa
from test_gpu_attention import assert_close
from test_gpu_backward import ETA, U, _bounds, _close, _schedule

pytestmark = pytest.mark.gpu
DEV = "cuda"


def _qkv(L, S, D, dtype, seed):
    g = torch.Generator().manual_seed(seed)
    return [torch.randn((L, S, D), generator=g).to(dtype) for _ in range(3)]


@pytest.mark.parametrize("L,S,D,dtype", [(1, 100, 64, torch.float16), (3, 1000, 128, torch.bfloat16),
                                         (2, 4133, 64, torch.bfloat16), (1, 8191, 128, torch.float16)])
@pytest.mark.parametrize("tie", ["index", "content"])
def test_builder_bit_exact(L, S, D, dtype, tie):
    _, k, _ = _qkv(L, S, D, dtype, S)
    rp, ci, sal = tsa.tsa_build_schedule(k.to(DEV), 64, 2, 1, 3, salience=True, tie_break=tie)
    assert tsa.tsa_last_device_status() == 0
    orp, oci, osal = oracle.build_schedule(k, 64, 2, 1, 3, tie=tie)
    nb = -(-S // 64)
    assert rp.numel() == nb + 1
    got_rp = rp.cpu().numpy()
    assert np.array_equal(got_rp, orp)
    assert np.array_equal(ci.cpu().numpy()[: got_rp[-1]], oci)
    assert np.array_equal(sal.cpu().numpy().view(np.int64), osal.view(np.int64))


@pytest.mark.parametrize("S", [1, 63, 65, 1000])
def test_dense_csr(S):
    rp, ci = tsa.tsa_dense_causal_csr(S, 64)
    orp, oci = oracle.dense_causal_csr(-(-S // 64))
    assert np.array_equal(rp.cpu().numpy(), orp) and np.array_equal(ci.cpu().numpy(), oci)


def _attention(q, k, v, rp, ci, scale, rows_extra=64):
    """Run into an output / lse buffer with sentinel rows past the end."""
    L, S, D = q.shape
    big = torch.full((L * S + rows_extra, D), 7.0, dtype=q.dtype, device=DEV)
    lse_big = torch.full((L * S + rows_extra,), 7.0, dtype=torch.float32, device=DEV)
    out = big[: L * S].view(L, S, D)
    lse = lse_big[: L * S].view(L, S)
    rp_d = torch.as_tensor(np.asarray(rp), dtype=torch.int32, device=DEV)
    ci_d = torch.as_tensor(np.asarray(ci) if len(ci) else np.zeros(1, np.int32), dtype=torch.int32, device=DEV)
    tsa.tsa_scheduled_attention_fwd(q.to(DEV), k.to(DEV), v.to(DEV), rp_d, ci_d, scale, out=out, lse=lse)
    assert tsa.tsa_last_device_status() == 0
    assert bool((big[L * S:] == 7.0).all()) and bool((lse_big[L * S:] == 7.0).all())
    return out.cpu(), lse.cpu()


@pytest.mark.parametrize("L,S,D,dtype", [(1, 100, 64, torch.float16), (3, 1000, 128, torch.bfloat16),
                                         (4, 130, 128, torch.float16), (2, 4133, 64, torch.bfloat16),
                                         (1, 8191, 128, torch.bfloat16),
                                         # one query block, partial: one token, and 63 tokens
                                         (1, 1, 64, torch.float16), (3, 63, 128, torch.bfloat16)])
@pytest.mark.parametrize("kind", ["dense", "topology"])
def test_attention_matches_oracle(L, S, D, dtype, kind):
    q, k, v = _qkv(L, S, D, dtype, S + D)
    nb = -(-S // 64)
    if kind == "dense":
        rp, ci = oracle.dense_causal_csr(nb)
    else:
        rp, ci, _ = oracle.build_schedule(k, 64, 1, 2, 3)
    scale = D ** -0.5
    out, lse = _attention(q, k, v, rp, ci, scale)
    ref, ref_lse = oracle.attention(q, k, v, rp, ci, 64, scale, nthreads=8, return_lse=True)
    assert_close(out.double().numpy(), ref, dtype)
    u = 2.0 ** -11 if dtype == torch.float16 else 2.0 ** -8
    assert np.abs(lse.double().numpy() - ref_lse).max() <= u


@pytest.mark.parametrize("L,S,D,dtype,kind", [(1, 100, 64, torch.float16, "dense"),
                                              (2, 33, 64, torch.float16, "dense"),
                                                (3, 1000, 128, torch.bfloat16, "random"),
                                                (2, 4133, 64, torch.bfloat16, "holes"),
                                                (2, 130, 128, torch.float16, "dense"),
                                                (1, 8191, 128, torch.bfloat16, "random")])
def test_backward_matches_oracle(L, S, D, dtype, kind):
    """dQ, dK, dV with a partial last block, every lane against the oracle; rows past the last
    lane's end stay untouched (a partial block is stored row by row, not as a 64-row box)."""
    q, k, v = _qkv(L, S, D, dtype, 3 * S + D)
    g = torch.Generator().manual_seed(S)
    dO = torch.randn((L, S, D), generator=g).to(dtype)
    nb = -(-S // 64)
    rp, ci = _schedule(kind, nb, seed=L)
    scale = D ** -0.5
    rpd, cid = torch.as_tensor(rp, device=DEV), torch.as_tensor(ci, device=DEV)
    O, lse = tsa.tsa_scheduled_attention_fwd(q.to(DEV), k.to(DEV), v.to(DEV), rpd, cid, scale)
    bufs = [torch.full((L * S + 64, D), 7.0, dtype=dtype, device=DEV) for _ in range(3)]
    grads = [b[: L * S].view(L, S, D) for b in bufs]
    tsa.tsa_scheduled_attention_backward(q.to(DEV), k.to(DEV), v.to(DEV), O, dO.to(DEV), lse, rpd, cid,
                                         scale, dq=grads[0], dk=grads[1], dv=grads[2])
    assert tsa.tsa_last_device_status() == 0
    for b in bufs:
        assert bool((b[L * S:] == 7.0).all())
    refs = oracle.attention_backward(q, k, v, dO, rp, ci, 64, scale, nthreads=8)
    bounds = _bounds(q, k, v, dO, rp, ci, scale, U[dtype], ETA[dtype])
    for name, got, ref, b in zip(("dQ", "dK", "dV"), grads, refs, bounds):
        _close(got, ref, U[dtype], f"{kind} {name}", b, ETA[dtype])
