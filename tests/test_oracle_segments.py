"""Pins for the oracle's segment schedules (fixed segments and arbitrary segment starts).

What pins what:
* the pages' printed block counts at S 4096 / block 64: 288 (512-token segments), 160
  (256-token segments), 2080 (one segment = dense) -- tests/golden/segment_counts.txt;
* the closed form of block-aligned fixed segments (row i = [segment start, i]);
* for arbitrary token starts, the row structure derived independently of the oracle's
  token-by-token union: row i runs from the block of the last start <= the block's first token
  to i;
* the random-boundary expectation in closed form against the oracle's mean over seeded draws,
  and the pages' 478 (mean of 200 draws) against that closed form;
* zero error of block-aligned segment schedules: the scheduled attention equals causal
  attention run on each segment separately.
"""
import os

import numpy as np
import pytest
import torch

import oracle

GOLDEN = os.path.join(os.path.dirname(__file__), "golden")


def _golden():
    fixed, random = [], []
    for line in open(os.path.join(GOLDEN, "segment_counts.txt")):
        if not line.strip() or line.startswith("#"):
            continue
        f = line.split()
        if f[0] == "random":
            random.append((int(f[1]), int(f[2]), float(f[3]), int(f[4]), float(f[5])))
        else:
            fixed.append(tuple(int(x) for x in f))
    return fixed, random


def test_fixed_segment_counts_match_pages():
    fixed, _ = _golden()
    assert len(fixed) == 3
    for S, block, seg, blocks in fixed:
        row_ptr, col_idx = oracle.fixed_segment_csr(S, block, seg)
        assert row_ptr[-1] == blocks == col_idx.size


@pytest.mark.parametrize("S,block,seg", [(4096, 64, 512), (1024, 64, 64), (2048, 32, 96),
                                         (640, 64, 192), (64, 64, 64)])
def test_block_aligned_fixed_segments_closed_form(S, block, seg):
    row_ptr, col_idx = oracle.fixed_segment_csr(S, block, seg)
    nb, m = S // block, seg // block
    assert row_ptr[0] == 0
    for i in range(nb):
        assert list(col_idx[row_ptr[i]:row_ptr[i + 1]]) == list(range((i // m) * m, i + 1))
    full, rest = divmod(nb, m)
    assert row_ptr[-1] == full * m * (m + 1) // 2 + rest * (rest + 1) // 2


def _rows_from_starts(S, block, starts):
    """Row i = [block of the last start <= block*i, i]: the earliest token of a query block has
    the earliest segment start, and every block from there to i holds an allowed key."""
    nb = S // block
    rows = []
    for i in range(nb):
        s = max([0] + [x for x in starts if x <= block * i])
        rows.append(list(range(s // block, i + 1)))
    return rows


@pytest.mark.parametrize("seed", range(6))
def test_token_starts_row_structure(seed):
    rng = np.random.default_rng(seed)
    S, block = 1024, 64
    starts = np.sort(rng.choice(np.arange(1, S), size=rng.integers(0, 12), replace=False))
    row_ptr, col_idx = oracle.segment_csr(S, block, starts)
    rows = _rows_from_starts(S, block, list(starts))
    assert row_ptr[-1] == sum(len(r) for r in rows)
    for i, r in enumerate(rows):
        assert list(col_idx[row_ptr[i]:row_ptr[i + 1]]) == r


def test_segment_special_cases():
    S, block = 512, 64
    nb = S // block
    dense = oracle.dense_causal_csr(nb)
    for starts in ([], [0]):
        rp, ci = oracle.segment_csr(S, block, starts)
        assert np.array_equal(rp, dense[0]) and np.array_equal(ci, dense[1])
    rp, ci = oracle.segment_csr(S, block, list(range(0, S, block)))  # every block its own segment
    assert np.array_equal(rp, np.arange(nb + 1)) and np.array_equal(ci, np.arange(nb))
    rp, ci = oracle.segment_csr(S, block, list(range(S)))  # every token its own segment
    assert np.array_equal(rp, np.arange(nb + 1)) and np.array_equal(ci, np.arange(nb))
    for bad in ([5, 5], [7, 3], [-1], [S]):
        with pytest.raises(ValueError):
            oracle.segment_csr(S, block, bad)


def _expected_random_blocks(S, block, p):
    """E[visited blocks] when each token t >= 1 starts a segment with probability p.

    Row i runs from block floor(s/block) to i, s the last start <= block*i.  s < block*m holds
    iff no token in [block*m, block*i] starts a segment, probability (1-p)^(block*(i-m)+1), so
    E[len(row i)] = 1 + sum_{d=0}^{i-1} (1-p)^(block*d+1).
    """
    nb = S // block
    return sum(1 + sum((1 - p) ** (block * d + 1) for d in range(i)) for i in range(nb))


def test_random_boundaries_mean_matches_closed_form_and_pages():
    _, random = _golden()
    (S, block, p, draws, printed), = random
    expect = _expected_random_blocks(S, block, p)
    rng = np.random.default_rng(2024)
    counts = []
    for _ in range(600):
        starts = 1 + np.flatnonzero(rng.random(S - 1) < p)
        counts.append(int(oracle.segment_csr(S, block, starts)[0][-1]))
    counts = np.array(counts, dtype=np.float64)
    sd = counts.std(ddof=1)
    # the oracle's Monte Carlo mean agrees with the closed form (4 standard errors)
    assert abs(counts.mean() - expect) < 4 * sd / np.sqrt(counts.size)
    # the pages' 200-draw mean is a draw from the same distribution (3 standard errors)
    assert abs(printed - expect) < 3 * sd / np.sqrt(draws)


@pytest.mark.parametrize("dtype", [torch.float16, torch.bfloat16])
def test_block_aligned_segments_have_zero_schedule_error(dtype):
    """Segments that start on block boundaries: scheduled attention over the segment CSR is
    causal attention within each segment, computed here segment by segment."""
    g = torch.Generator().manual_seed(11)
    L, S, D, block, seg = 2, 512, 16, 64, 192
    Q, K, V = (torch.randn((L, S, D), generator=g).to(dtype) for _ in range(3))
    rp, ci = oracle.fixed_segment_csr(S, block, seg)
    got = oracle.attention(Q, K, V, rp, ci, block, 0.25)
    want = np.empty_like(got)
    for s0 in range(0, S, seg):
        n = min(seg, S - s0)
        drp, dci = oracle.dense_causal_csr(n // block)
        sl = slice(s0, s0 + n)
        want[:, sl] = oracle.attention(Q[:, sl].contiguous(), K[:, sl].contiguous(),
                                       V[:, sl].contiguous(), drp, dci, block, 0.25)
    assert np.abs(got - want).max() <= 1e-12
