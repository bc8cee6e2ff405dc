"""Pins for the oracle on sequences whose length is not a multiple of the block (a partial last
block).  Reading: nb = ceil(S / block); the last block holds the S - (nb - 1) * block tokens
that exist; its centroid averages those tokens; attention sees keys k < S only.

What pins what:
* centroids -- exact rational arithmetic on integer-valued keys (the sums are exact, so the
  centroid is the correctly rounded quotient of two integers), and piecewise-constant keys;
* attention -- the dense causal CSR reproduces torch's causal scaled-dot-product attention in
  fp64 on the S tokens; the diagonal-only CSR reproduces block-local causal attention with a
  short last block;
* schedule -- a partial last block whose n tokens (n dividing the block) are tiled to fill a
  full block has the same centroid (the sums are exact), hence the same CSR and salience.
"""
from fractions import Fraction

import numpy as np
import pytest
import torch

import oracle


@pytest.mark.parametrize("S,L", [(100, 1), (200, 3), (65, 2), (127, 1)])
def test_centroids_integer_keys_exact(S, L):
    g = torch.Generator().manual_seed(S + L)
    k = torch.randint(-40, 41, (L, S, 5), generator=g).to(torch.bfloat16)  # integers: exact in bf16
    C = oracle.centroids(k, 64)
    nb = -(-S // 64)
    assert C.shape == (nb, 5)
    x = k.to(torch.int64).numpy()
    for b in range(nb):
        lo, hi = 64 * b, min(64 * (b + 1), S)
        for d in range(5):
            total = int(x[:, lo:hi, d].sum())
            assert C[b, d] == float(Fraction(total, (hi - lo) * L)), (b, d)


def test_centroids_piecewise_constant():
    S = 64 * 3 + 7
    vals = np.array([1.5, -2.0, 0.25, 3.0])
    k = np.repeat(vals, 64)[:S]
    K = torch.tensor(np.tile(k[None, :, None], (2, 1, 4)), dtype=torch.bfloat16)
    C = oracle.centroids(K, 64)
    assert np.array_equal(C, np.repeat(vals[:, None], 4, axis=1))


def _sdpa_causal(Q, K, V, scale):
    q, k, v = (x.double() for x in (Q, K, V))
    return torch.nn.functional.scaled_dot_product_attention(q, k, v, is_causal=True, scale=scale).numpy()


@pytest.mark.parametrize("S,D,dtype", [(100, 16, torch.float16), (1000, 64, torch.bfloat16), (129, 32, torch.float16)])
def test_dense_csr_is_causal_attention(S, D, dtype):
    g = torch.Generator().manual_seed(S)
    Q, K, V = (torch.randn((2, S, D), generator=g).to(dtype) for _ in range(3))
    nb = -(-S // 64)
    rp, ci = oracle.dense_causal_csr(nb)
    got = oracle.attention(Q, K, V, rp, ci, 64, D ** -0.5, nthreads=4)
    ref = _sdpa_causal(Q, K, V, D ** -0.5)
    assert np.abs(got - ref).max() < 1e-12


def test_diagonal_csr_is_blockwise_causal_attention():
    S, D = 150, 16
    g = torch.Generator().manual_seed(5)
    Q, K, V = (torch.randn((1, S, D), generator=g).to(torch.float16) for _ in range(3))
    nb = -(-S // 64)
    rp = np.arange(nb + 1, dtype=np.int32)
    ci = np.arange(nb, dtype=np.int32)
    got = oracle.attention(Q, K, V, rp, ci, 64, 0.25)
    ref = np.concatenate([_sdpa_causal(Q[:, a:a + 64], K[:, a:a + 64], V[:, a:a + 64], 0.25)
                          for a in range(0, S, 64)], axis=1)
    assert np.abs(got - ref).max() < 1e-12


@pytest.mark.parametrize("n", [16, 32])
def test_partial_block_equals_tiled_full_block(n):
    g = torch.Generator().manual_seed(n)
    nb = 9
    S = 64 * (nb - 1) + n
    K = torch.randn((2, S, 32), generator=g).to(torch.bfloat16)
    tail = K[:, 64 * (nb - 1):]
    full = torch.cat([K[:, : 64 * (nb - 1)], tail.repeat(1, 64 // n, 1)], dim=1)
    assert np.array_equal(oracle.centroids(K, 64), oracle.centroids(full, 64))
    a = oracle.build_schedule(K, 64, 1, 1, 2)
    b = oracle.build_schedule(full, 64, 1, 1, 2)
    assert np.array_equal(a[0], b[0]) and np.array_equal(a[1], b[1])
    assert np.array_equal(a[2].view(np.int64), b[2].view(np.int64))
    assert np.count_nonzero(a[2] == 0) == 1 and a[0].shape[0] == nb + 1
