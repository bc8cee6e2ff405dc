"""Pins for the oracle's masked attention.

* The dense causal CSR reproduces full causal softmax attention: torch's
  scaled_dot_product_attention (fp64, CPU, is_causal) is the independent library routine.
* The diagonal-only schedule is causal attention inside each block (same routine per block).
* The pages' single-pass form (running maximum and denominator, rescale by
  exp(m_prev - m_new)) agrees with the two-pass form to 1e-12, the figure the PR mirror
  page's port note quotes for its f64 check against dense masked attention.
* An explicit dense [S, S] mask built from the CSR, with scipy's softmax, agrees on random
  schedules (a different formulation: whole-matrix masking instead of per-row gathering).
"""
import numpy as np
import pytest
import torch
from scipy.special import softmax

import oracle
from topology_scheduled_gb300.workloads import random_density_csr


def _qkv(L, S, D, dtype, seed):
    g = torch.Generator().manual_seed(seed)
    return [torch.randn((L, S, D), generator=g).to(dtype) for _ in range(3)]


@pytest.mark.parametrize("dtype", [torch.float16, torch.bfloat16])
@pytest.mark.parametrize("S,D,block", [(256, 64, 64), (192, 32, 32), (40, 8, 8)])
def test_dense_csr_is_full_causal_sdpa(dtype, S, D, block):
    q, k, v = _qkv(2, S, D, dtype, 1)
    rp, ci = oracle.dense_causal_csr(S // block)
    scale = 1.0 / np.sqrt(D)
    got = oracle.attention(q, k, v, rp, ci, block, scale)
    ref = torch.nn.functional.scaled_dot_product_attention(
        q.double(), k.double(), v.double(), is_causal=True, scale=scale).numpy()
    np.testing.assert_allclose(got, ref, rtol=0, atol=1e-12)


def test_diagonal_only_is_blockwise_causal():
    S, D, block = 256, 16, 64
    q, k, v = _qkv(1, S, D, torch.float16, 2)
    nb = S // block
    rp, ci = np.arange(nb + 1, dtype=np.int32), np.arange(nb, dtype=np.int32)
    got = oracle.attention(q, k, v, rp, ci, block, 0.25)
    for b in range(nb):
        sl = slice(b * block, (b + 1) * block)
        ref = torch.nn.functional.scaled_dot_product_attention(
            q[:, sl].double(), k[:, sl].double(), v[:, sl].double(), is_causal=True,
            scale=0.25).numpy()
        np.testing.assert_allclose(got[:, sl], ref, rtol=0, atol=1e-12)


def _dense_mask_reference(q, k, v, rp, ci, block, scale):
    Q, K, V = (x.double().numpy() for x in (q, k, v))
    L, S, D = Q.shape
    allowed = np.zeros((S, S), dtype=bool)
    for i in range(S // block):
        for j in ci[rp[i]:rp[i + 1]]:
            allowed[i * block:(i + 1) * block, j * block:(j + 1) * block] = True
    allowed &= np.tril(np.ones((S, S), dtype=bool))
    out = np.zeros_like(Q)
    for l in range(L):
        s = scale * Q[l] @ K[l].T
        s[~allowed] = -np.inf
        has = allowed.any(axis=1)
        p = np.zeros_like(s)
        p[has] = softmax(s[has], axis=1)
        out[l] = p @ V[l]
    return out


@pytest.mark.parametrize("density,seed", [(0.0, 0), (0.2, 1), (0.5, 2), (1.0, 3)])
def test_random_schedule_matches_dense_mask(density, seed):
    S, D, block = 320, 16, 32
    q, k, v = _qkv(2, S, D, torch.bfloat16, 10 + seed)
    rp, ci = random_density_csr(S // block, density, seed)
    got = oracle.attention(q, k, v, rp, ci, block, 0.3)
    ref = _dense_mask_reference(q, k, v, rp, ci, block, 0.3)
    np.testing.assert_allclose(got, ref, rtol=0, atol=1e-12)


def test_online_equals_two_pass():
    S, D, block = 512, 64, 64
    q, k, v = _qkv(2, S, D, torch.float16, 4)
    k = (k.float() * 3).to(torch.float16)  # wide score range so the running max moves often
    rp, ci = random_density_csr(S // block, 0.6, 4)
    a = oracle.attention(q, k, v, rp, ci, block, 0.125)
    b = oracle.attention(q, k, v, rp, ci, block, 0.125, online=True)
    assert np.max(np.abs(a - b)) <= 1e-12


def test_rows_subset_threads_and_degenerate_rows():
    S, D, block = 256, 32, 64
    q, k, v = _qkv(3, S, D, torch.bfloat16, 5)
    nb = S // block
    # row 2 empty: its tokens have no key and get O = 0
    rp = np.array([0, 1, 3, 3, 5], dtype=np.int32)
    ci = np.array([0, 0, 1, 1, 3], dtype=np.int32)
    full = oracle.attention(q, k, v, rp, ci, block, 0.2)
    assert np.all(full[:, 2 * block:3 * block] == 0)
    # token 0 attends to itself only
    np.testing.assert_array_equal(full[:, 0], v[:, 0].double().numpy())
    lanes = np.array([2, 0, 1, 2], dtype=np.int64)
    toks = np.array([255, 17, 64, 200], dtype=np.int64)
    for nt in (1, 3):
        sub = oracle.attention(q, k, v, rp, ci, block, 0.2, lanes=lanes, tokens=toks, nthreads=nt)
        np.testing.assert_array_equal(sub, full[lanes, toks])
    assert nb == 4
