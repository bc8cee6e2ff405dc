"""Pins for the oracle's backward pass and log-sum-exp.

What pins what:
* gradients -- torch autograd in fp64 through a dense-mask formulation of the same attention
  (scores masked with -inf outside the CSR / causal set, torch softmax, matmuls), on dense,
  diagonal-only, random and empty-row schedules, f16 and bf16 inputs;
* invariants of the chain rule: shifting every key by one vector leaves each softmax row
  unchanged, so the key gradients sum to zero; each softmax row sums to one, so the value
  gradients sum to the upstream gradient of the rows that have keys; a query with a single
  allowed key has an exactly zero query gradient;
* log-sum-exp -- scipy.special.logsumexp over the same masked scores, -inf for rows without
  keys, and scale * <q, k> for single-key rows;
* a sequence whose length is not a multiple of the block (a partial last block): the same
  autograd comparison with the mask cut at S.
"""
import numpy as np
import pytest
import torch
from scipy.special import logsumexp

import oracle


def _mask(row_ptr, col_idx, S, block):
    nb = -(-S // block)  # a partial last block counts
    M = np.zeros((S, S), dtype=bool)
    for i in range(nb):
        for j in col_idx[row_ptr[i]:row_ptr[i + 1]]:
            M[i * block:(i + 1) * block, j * block:(j + 1) * block] = True
    return M & np.tril(np.ones((S, S), dtype=bool))


def _autograd(Q, K, V, dO, M, scale):
    q, k, v = (x.double().clone().requires_grad_(True) for x in (Q, K, V))
    s = scale * q @ k.transpose(-1, -2)
    m = torch.as_tensor(M)
    has = m.any(dim=-1, keepdim=True)
    s = s.masked_fill(~m, float("-inf")).masked_fill(~has, 0.0)
    p = torch.softmax(s, dim=-1) * has
    o = p @ v
    (o * dO.double()).sum().backward()
    return q.grad.numpy(), k.grad.numpy(), v.grad.numpy(), s.detach().numpy()


def _schedules(nb, seed):
    rng = np.random.default_rng(seed)
    dense = oracle.dense_causal_csr(nb)
    diag = (np.arange(nb + 1, dtype=np.int32), np.arange(nb, dtype=np.int32))
    rows = [sorted(set(rng.choice(i + 1, size=rng.integers(1, i + 2), replace=False).tolist()))
            for i in range(nb)]
    rows[1] = []  # an empty row
    rows[2] = [0]  # a row without its diagonal block
    rp = np.zeros(nb + 1, np.int32)
    rp[1:] = np.cumsum([len(r) for r in rows])
    rand = (rp, np.array([j for r in rows for j in r], np.int32))
    return {"dense": dense, "diagonal": diag, "random": rand}


@pytest.mark.parametrize("dtype", [torch.float16, torch.bfloat16])
@pytest.mark.parametrize("kind", ["dense", "diagonal", "random"])
def test_gradients_equal_autograd(dtype, kind):
    g = torch.Generator().manual_seed(21)
    L, S, D, block, scale = 2, 192, 16, 32, 0.3
    Q, K, V, dO = (torch.randn((L, S, D), generator=g).to(dtype) for _ in range(4))
    rp, ci = _schedules(S // block, 4)[kind]
    dq, dk, dv = oracle.attention_backward(Q, K, V, dO, rp, ci, block, scale, nthreads=2)
    rq, rk, rv, _ = _autograd(Q, K, V, dO, _mask(rp, ci, S, block), scale)
    for got, ref in ((dq, rq), (dk, rk), (dv, rv)):
        assert np.abs(got - ref).max() <= 1e-10 * max(1.0, np.abs(ref).max())


def test_gradient_invariants():
    g = torch.Generator().manual_seed(22)
    L, S, D, block, scale = 3, 256, 8, 64, 0.5
    Q, K, V, dO = (torch.randn((L, S, D), generator=g).to(torch.bfloat16) for _ in range(4))
    for kind, (rp, ci) in _schedules(S // block, 5).items():
        dq, dk, dv = oracle.attention_backward(Q, K, V, dO, rp, ci, block, scale, nthreads=3)
        M = _mask(rp, ci, S, block)
        has = M.any(axis=1)
        assert np.abs(dk.sum(axis=1)).max() <= 1e-11, kind
        want = (dO.double().numpy() * has[None, :, None]).sum(axis=1)
        assert np.abs(dv.sum(axis=1) - want).max() <= 1e-11, kind
        single = M.sum(axis=1) == 1
        assert np.all(dq[:, single] == 0.0), kind


def test_lse_matches_logsumexp():
    g = torch.Generator().manual_seed(23)
    L, S, D, block, scale = 2, 256, 32, 64, 0.125
    Q, K, V = (torch.randn((L, S, D), generator=g).to(torch.float16) for _ in range(3))
    for kind, (rp, ci) in _schedules(S // block, 6).items():
        _, lse = oracle.attention(Q, K, V, rp, ci, block, scale, return_lse=True, nthreads=2)
        M = _mask(rp, ci, S, block)
        s = scale * np.einsum("lqd,lkd->lqk", Q.double().numpy(), K.double().numpy())
        ref = logsumexp(np.where(M[None], s, -np.inf), axis=-1)
        assert np.array_equal(np.isinf(lse), np.isinf(ref)), kind
        fin = np.isfinite(ref)
        assert np.abs(lse[fin] - ref[fin]).max() <= 1e-12, kind
        single = M.sum(axis=1) == 1  # one allowed key: lse is that key's scaled score
        only = np.where(M[None], s, -np.inf).max(axis=-1)
        assert np.abs(lse[:, single] - only[:, single]).max() <= 1e-12, kind


@pytest.mark.parametrize("S", [163, 129, 31])
@pytest.mark.parametrize("kind", ["dense", "random"])
def test_partial_last_block_gradients_equal_autograd(S, kind):
    g = torch.Generator().manual_seed(S)
    L, D, block, scale = 2, 16, 32, 0.3
    Q, K, V, dO = (torch.randn((L, S, D), generator=g).to(torch.bfloat16) for _ in range(4))
    nb = -(-S // block)
    if kind == "dense":
        rp, ci = oracle.dense_causal_csr(nb)
    else:
        rng = np.random.default_rng(S)
        rows = [sorted(set(rng.choice(i + 1, size=rng.integers(1, i + 2), replace=False).tolist()) | {i})
                for i in range(nb)]
        rp = np.zeros(nb + 1, np.int32)
        rp[1:] = np.cumsum([len(r) for r in rows])
        ci = np.array([j for r in rows for j in r], np.int32)
    dq, dk, dv = oracle.attention_backward(Q, K, V, dO, rp, ci, block, scale, nthreads=2)
    rq, rk, rv, _ = _autograd(Q, K, V, dO, _mask(rp, ci, S, block), scale)
    for got, ref in ((dq, rq), (dk, rk), (dv, rv)):
        assert got.shape == (L, S, D)
        assert np.abs(got - ref).max() <= 1e-10 * max(1.0, np.abs(ref).max())
