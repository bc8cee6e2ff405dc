"""GPU segment schedules vs the CPU oracle (bit-exact CSR), and scheduled attention over them:
parity with the oracle and, for block-aligned segments, with causal attention run segment by
segment (the zero schedule error the pages claim for segment boundaries)."""
import numpy as np
import pytest
import torch

import oracle
import topology_scheduled_gb300 as tsa

pytestmark = pytest.mark.gpu
DEV = "cuda"


def _np(rp, ci):
    rp = rp.cpu().numpy()
    return rp, ci.cpu().numpy()[: rp[-1]]


@pytest.mark.parametrize("S,block,seg,count", [(4096, 64, 512, 288), (4096, 64, 256, 160),
                                               (4096, 64, 4096, 2080)])
def test_fixed_segment_counts_of_the_pages(S, block, seg, count):
    rp, ci = _np(*tsa.tsa_fixed_segment_csr(S, block, seg))
    rp_o, ci_o = oracle.fixed_segment_csr(S, block, seg)
    assert np.array_equal(rp, rp_o) and np.array_equal(ci, ci_o)
    assert rp[-1] == count
    assert tsa.tsa_last_device_status() == 0


@pytest.mark.parametrize("S,block,seg", [(64, 64, 64), (640, 64, 192), (1024, 64, 100), (2048, 32, 7),
                                         (32768, 64, 1536), (65534 * 2, 2, 4096)])
def test_fixed_segments_bit_exact(S, block, seg):
    rp, ci = _np(*tsa.tsa_fixed_segment_csr(S, block, seg))
    if S <= 32768:
        rp_o, ci_o = oracle.fixed_segment_csr(S, block, seg)
        assert np.array_equal(rp, rp_o) and np.array_equal(ci, ci_o)
    else:  # nb 65534: check the closed form row by row
        nb, m = S // block, seg // block
        assert rp[-1] == tsa.tsa_fixed_segment_nnz(S, block, seg)
        for i in (0, 1, m - 1, m, nb // 2, nb - 1):
            assert list(ci[rp[i]:rp[i + 1]]) == list(range((i // m) * m, i + 1))
    assert tsa.tsa_last_device_status() == 0


@pytest.mark.parametrize("seed", range(8))
def test_random_token_starts_bit_exact(seed):
    rng = np.random.default_rng(seed)
    block = int(rng.choice([16, 64]))
    S = block * int(rng.integers(1, 80))
    p = float(rng.choice([0.0024, 0.01, 0.1]))
    starts = 1 + np.flatnonzero(rng.random(S - 1) < p)
    if seed == 3:
        starts = np.concatenate([[0], starts])  # an explicit start at token 0
    st = torch.as_tensor(starts.astype(np.int32), device=DEV)
    rp, ci = _np(*tsa.tsa_segment_csr(S, block, st))
    rp_o, ci_o = oracle.segment_csr(S, block, starts)
    assert np.array_equal(rp, rp_o) and np.array_equal(ci, ci_o)
    assert tsa.tsa_last_device_status() == 0


def test_segment_edge_cases():
    S, block = 512, 64
    empty = torch.zeros(0, dtype=torch.int32, device=DEV)
    rp, ci = _np(*tsa.tsa_segment_csr(S, block, empty))
    rp_o, ci_o = oracle.dense_causal_csr(S // block)
    assert np.array_equal(rp, rp_o) and np.array_equal(ci, ci_o)
    every = torch.arange(S, dtype=torch.int32, device=DEV)
    rp, ci = _np(*tsa.tsa_segment_csr(S, block, every))
    assert np.array_equal(rp, np.arange(9)) and np.array_equal(ci, np.arange(8))
    assert tsa.tsa_last_device_status() == 0


def test_bad_starts_use_the_valid_prefix_and_report():
    S, block = 1024, 64
    st = torch.tensor([130, 400, 390, 700], dtype=torch.int32, device=DEV)  # 390 out of order
    rp, ci = _np(*tsa.tsa_segment_csr(S, block, st))
    assert tsa.tsa_last_device_status() == 8  # TSA_ERR_BAD_SCHEDULE
    rp_o, ci_o = oracle.segment_csr(S, block, [130, 400])
    assert np.array_equal(rp, rp_o) and np.array_equal(ci, ci_o)
    st = torch.tensor([S], dtype=torch.int32, device=DEV)  # out of range
    rp, ci = _np(*tsa.tsa_segment_csr(S, block, st))
    assert tsa.tsa_last_device_status() == 8
    assert np.array_equal(rp, oracle.dense_causal_csr(S // block)[0])


def test_capacity_cut_is_reported():
    S, block = 1024, 64
    st = torch.zeros(0, dtype=torch.int32, device=DEV)
    rp, ci = tsa.tsa_segment_csr(S, block, st, col_cap=50)
    assert tsa.tsa_last_device_status() == 9  # TSA_ERR_DEVICE (capacity on the device)
    rp = rp.cpu().numpy()
    assert rp[-1] == 50 and np.all(np.diff(rp) >= 0)


@pytest.mark.parametrize("dtype,D", [(torch.float16, 64), (torch.bfloat16, 128)])
def test_attention_over_fixed_segments(dtype, D):
    """Block-aligned segments: GPU attention matches the oracle over the segment CSR and causal
    attention computed independently on each segment."""
    g = torch.Generator().manual_seed(5)
    L, S, seg = 2, 2048, 512
    Q, K, V = (torch.randn((L, S, D), generator=g).to(dtype) for _ in range(3))
    rp, ci = tsa.tsa_fixed_segment_csr(S, 64, seg)
    out = tsa.tsa_scheduled_attention(Q.to(DEV), K.to(DEV), V.to(DEV), rp, ci, 0.125)
    assert tsa.tsa_last_device_status() == 0
    got = out.cpu().double().numpy()
    rp_o, ci_o = oracle.fixed_segment_csr(S, 64, seg)
    ref = oracle.attention(Q, K, V, rp_o, ci_o, 64, 0.125, nthreads=8)
    tol = 2e-3 if dtype == torch.float16 else 1e-2
    assert np.abs(got - ref).max() <= tol
    # the segment-by-segment causal run on the GPU gives the same rows, bit for bit
    drp, dci = tsa.tsa_dense_causal_csr(seg, 64)
    for s0 in range(0, S, seg):
        sl = slice(s0, s0 + seg)
        part = tsa.tsa_scheduled_attention(Q[:, sl].contiguous().to(DEV), K[:, sl].contiguous().to(DEV),
                                           V[:, sl].contiguous().to(DEV), drp, dci, 0.125)
        assert torch.equal(part.cpu(), out[:, sl].cpu())


def test_attention_over_token_starts():
    """Starts inside blocks: the kernel runs the covering block schedule; parity with the oracle
    over the same CSR."""
    g = torch.Generator().manual_seed(6)
    L, S, D = 1, 4096, 64
    Q, K, V = (torch.randn((L, S, D), generator=g).to(torch.float16) for _ in range(3))
    starts = np.array([700, 1500, 1536, 3001], dtype=np.int32)
    rp, ci = tsa.tsa_segment_csr(S, 64, torch.as_tensor(starts, device=DEV))
    out = tsa.tsa_scheduled_attention(Q.to(DEV), K.to(DEV), V.to(DEV), rp, ci, 0.125)
    assert tsa.tsa_last_device_status() == 0
    rp_o, ci_o = oracle.segment_csr(S, 64, starts)
    ref = oracle.attention(Q, K, V, rp_o, ci_o, 64, 0.125, nthreads=8)
    assert np.abs(out.cpu().double().numpy() - ref).max() <= 2e-3
