"""Pins for the oracle's schedule builder (centroids, distances, elder-rule salience, CSR).

What pins what:
* dense causal CSR -- the pages' printed block counts (tests/golden/dense_causal_counts.txt)
  and the closed form of the lower triangle;
* centroids -- torch's fp64 mean (f16 sums are exact in binary64, so every order agrees);
* distances -- exact integer arithmetic on integer points, and scipy's cdist;
* salience -- the hand-worked cases in tests/golden/elder_rule_examples.txt, "exactly one
  block scores zero", the H0 barcode by brute-force single linkage and by scipy's
  single-linkage dendrogram, and Prim's MST for the claim that MST edges suffice;
* topology CSR -- the hand-worked case, the special cases that reduce to the dense or the
  diagonal schedule, and the count bounds that contain the pages' 56/59 of 136 and 114 of 528.
"""
import itertools
import os

import numpy as np
import pytest
import torch
from scipy.cluster.hierarchy import linkage
from scipy.spatial.distance import cdist

import oracle

GOLDEN = os.path.join(os.path.dirname(__file__), "golden")


def _points_as_keys(points):
    """1-D points as a [1, n, 1] key tensor (block 1, one lane), exactly representable."""
    return torch.tensor(points, dtype=torch.float16).view(1, -1, 1)


# ---------------------------------------------------------------- dense CSR
def test_dense_counts_match_pages():
    rows = [l.split() for l in open(os.path.join(GOLDEN, "dense_causal_counts.txt"))
            if l.strip() and not l.startswith("#")]
    assert rows
    for seq, block, nb, dense in (map(int, r) for r in rows):
        assert seq // block == nb
        row_ptr, col_idx = oracle.dense_causal_csr(nb)
        assert row_ptr[-1] == dense == col_idx.size


@pytest.mark.parametrize("nb", [1, 2, 7, 256, 512])
def test_dense_layout_is_lower_triangle(nb):
    row_ptr, col_idx = oracle.dense_causal_csr(nb)
    assert row_ptr[0] == 0
    for i in range(nb):
        assert row_ptr[i + 1] - row_ptr[i] == i + 1
        assert list(col_idx[row_ptr[i]:row_ptr[i + 1]]) == list(range(i + 1))
    assert row_ptr[-1] == {256: 32896, 512: 131328}.get(nb, nb * (nb + 1) // 2)


# ---------------------------------------------------------------- centroids
@pytest.mark.parametrize("L,S,D,block", [(1, 128, 8, 64), (3, 96, 5, 32), (4, 64, 16, 1)])
def test_centroids_f16_equal_torch_mean(L, S, D, block):
    g = torch.Generator().manual_seed(3)
    K = (torch.randn((L, S, D), generator=g) * 3).to(torch.float16)
    got = oracle.centroids(K, block)
    ref = K.double().view(L, S // block, block, D).mean(dim=(0, 2)).numpy()
    assert np.array_equal(got, ref)


def test_centroids_bf16_exact_when_sums_are_exact():
    # small integers: every partial sum is exact, so the result is the rounded true mean
    g = torch.Generator().manual_seed(4)
    K = torch.randint(-50, 50, (3, 128, 6), generator=g).to(torch.bfloat16)
    got = oracle.centroids(K, 64)
    exact = K.double().view(3, 2, 64, 6).sum(dim=(0, 2)).numpy() / (3 * 64)
    assert np.array_equal(got, exact)


# ---------------------------------------------------------------- distances
def test_pairwise_d2_integer_points_exact():
    g = np.random.default_rng(5)
    C = g.integers(-1000, 1000, size=(9, 7)).astype(np.float64)
    D2 = oracle.pairwise_d2(C)
    for u, v in itertools.product(range(9), repeat=2):
        exact = sum(int(C[u, d] - C[v, d]) ** 2 for d in range(7))
        assert D2[u, v] == float(exact)


def test_pairwise_d2_matches_scipy_and_is_symmetric():
    g = np.random.default_rng(6)
    C = g.normal(size=(20, 64))
    D2 = oracle.pairwise_d2(C)
    assert np.array_equal(D2, D2.T)
    assert np.all(np.diag(D2) == 0)
    np.testing.assert_allclose(D2, cdist(C, C, "sqeuclidean"), rtol=1e-13, atol=1e-12)


def test_pairwise_d2_summation_order():
    """The stated binary64 order, written out with exact rationals (each fused multiply-add and
    each addition rounded once): 32 strided partial sums, then halving.  Coordinates spread over
    many binades so that a sequential sum rounds differently; D = 1, 31, 32, 33 and 100 cover
    empty, single-term and uneven partial sums."""
    from fractions import Fraction

    def fma(a, b, c):
        return float(Fraction(a) * Fraction(b) + Fraction(c))

    def add(a, b):
        return float(Fraction(a) + Fraction(b))

    g = np.random.default_rng(17)
    seq_differs = 0
    for D in (1, 31, 32, 33, 100):
        C = g.normal(size=(4, D)) * np.exp2(g.integers(-30, 30, size=(4, D)))
        D2 = oracle.pairwise_d2(C)
        for u, v in ((0, 1), (2, 3), (1, 3)):
            delta = [float(C[u, d] - C[v, d]) for d in range(D)]
            part = []
            for j in range(32):
                acc = 0.0
                for d in range(j, D, 32):
                    acc = fma(delta[d], delta[d], acc)
                part.append(acc)
            w = 16
            while w >= 1:
                part = [add(part[j], part[j + w]) for j in range(w)] + part[w:]
                w //= 2
            assert D2[u, v] == part[0] and D2[v, u] == part[0]
            seq = 0.0
            for d in range(D):
                seq = fma(delta[d], delta[d], seq)
            seq_differs += seq != part[0]
    assert seq_differs > 0  # the inputs do tell the two orders apart


# ---------------------------------------------------------------- salience
def _golden_elder():
    cases, csr = [], None
    lines = [l.split() for l in open(os.path.join(GOLDEN, "elder_rule_examples.txt"))
             if l.strip() and not l.startswith("#")]
    for i, l in enumerate(lines):
        if l[0] == "points":
            cases.append(([float(x) for x in l[1:]], [float(x) for x in lines[i + 1][1:]]))
        if l[0] == "csr":
            csr = ([int(x) for x in l[1:]], [int(x) for x in lines[i + 1][1:]],
                   [int(x) for x in lines[i + 2][1:]])
    return cases, csr


def test_elder_rule_hand_worked_cases():
    cases, _ = _golden_elder()
    assert len(cases) == 4
    for points, sal in cases:
        C = oracle.centroids(_points_as_keys(points), 1)
        got, _ = oracle.salience(C)
        assert list(got) == sal, points
        # the full builder reaches the same values through the key tensor
        _, _, got2 = oracle.build_schedule(_points_as_keys(points), 1, 0, 0, 0)
        assert list(got2) == sal


def _single_linkage_heights(C):
    """Brute force H0 barcode: merge the two closest clusters, O(n^3) per merge."""
    clusters = [[i] for i in range(len(C))]
    heights = []
    while len(clusters) > 1:
        best = None
        for a in range(len(clusters)):
            for b in range(a + 1, len(clusters)):
                d = min(float(np.sum((C[p] - C[q]) ** 2)) for p in clusters[a] for q in clusters[b])
                if best is None or d < best[0]:
                    best = (d, a, b)
        d, a, b = best
        heights.append(d)
        clusters[a] = clusters[a] + clusters[b]
        del clusters[b]
    return sorted(heights)


@pytest.mark.parametrize("seed", range(6))
def test_salience_is_h0_barcode_with_one_zero(seed):
    g = np.random.default_rng(seed)
    n = int(g.integers(2, 13))
    C = g.normal(size=(n, 4))
    sal, _ = oracle.salience(C)
    assert int(np.sum(sal == 0)) == 1
    nonzero = sorted(sal[sal != 0])
    np.testing.assert_allclose(nonzero, _single_linkage_heights(C), rtol=1e-12)
    # scipy's single-linkage dendrogram heights are Euclidean merge distances
    heights = np.sort(linkage(C, method="single", metric="euclidean")[:, 2])
    np.testing.assert_allclose(np.sqrt(nonzero), heights, rtol=1e-12)


def test_salience_multiset_is_permutation_invariant_but_not_per_block():
    # two equal-size ties: per-block values move with the order, the multiset does not
    pts = np.array([[0.0], [1.0], [10.0], [11.0]])
    base, _ = oracle.salience(pts)
    for perm in itertools.permutations(range(4)):
        sal, _ = oracle.salience(pts[list(perm)])
        assert sorted(sal) == sorted(base)
    moved, _ = oracle.salience(pts[[1, 0, 2, 3]])
    assert int(np.argmin(moved)) == 0 and moved[1] == 1.0  # block 0 keeps zero by index order


def _prim(D2):
    n = D2.shape[0]
    inside = [0]
    best = {v: (D2[0, v], 0) for v in range(1, n)}
    edges = set()
    while best:
        v = min(best, key=lambda x: (best[x][0], min(x, best[x][1]), max(x, best[x][1])))
        d, u = best.pop(v)
        edges.add((min(u, v), max(u, v)))
        inside.append(v)
        for w in best:
            if D2[v, w] < best[w][0]:
                best[w] = (D2[v, w], v)
    return edges


@pytest.mark.parametrize("seed", range(4))
def test_accepted_edges_are_the_mst(seed):
    g = np.random.default_rng(100 + seed)
    C = g.normal(size=(40, 16))
    _, (mu, mv, md) = oracle.salience(C)
    assert len(mu) == 39
    assert np.all(np.diff(md) >= 0)  # accepted in ascending order
    assert {(int(a), int(b)) for a, b in zip(mu, mv)} == _prim(oracle.pairwise_d2(C))


# ---------------------------------------------------------------- topology CSR
def test_topology_csr_hand_worked_case():
    cases, (params, row_ptr, col_idx) = _golden_elder()
    sal = np.array(cases[1][1])
    rp, ci = oracle.topology_csr(sal, *params)
    assert list(rp) == row_ptr and list(ci) == col_idx


@pytest.mark.parametrize("nb", [1, 5, 16, 33])
def test_topology_special_cases(nb):
    g = np.random.default_rng(nb)
    sal = g.random(nb)
    sal[g.integers(nb)] = 0.0
    dense = oracle.dense_causal_csr(nb)
    for args in [(0, nb - 1, 0), (0, 0, nb), (1, nb + 5, 3), (nb, 0, 0)]:
        rp, ci = oracle.topology_csr(sal, *args)
        assert np.array_equal(rp, dense[0]) and np.array_equal(ci, dense[1]), args
    rp, ci = oracle.topology_csr(sal, 0, 0, 0)
    assert np.array_equal(rp, np.arange(nb + 1)) and np.array_equal(ci, np.arange(nb))


def test_topology_rows_are_valid_and_within_bounds():
    # sink 1, local_radius 1, topk 2: 45 <= nnz <= 70 at 16 blocks (pages: 59 and 56 of 136),
    # 93 <= nnz <= 150 at 32 blocks (pages: 114 of 528)
    for nb, lo, hi in [(16, 45, 70), (32, 93, 150), (64, 189, 310)]:
        for seed in range(20):
            g = np.random.default_rng(seed)
            sal = g.random(nb) ** 3
            sal[g.integers(nb)] = 0.0
            rp, ci = oracle.topology_csr(sal, 1, 1, 2)
            assert lo <= rp[-1] <= hi
            assert rp[-1] <= oracle.max_nnz(nb, 1, 1, 2)
            for i in range(nb):
                row = ci[rp[i]:rp[i + 1]]
                assert np.all(np.diff(row) > 0) and row[0] == 0 and row[-1] == i
                top2 = sorted(range(i + 1), key=lambda j: (-sal[j], j))[:2]
                assert set(top2) <= set(row)
        assert lo <= {16: 56, 32: 114, 64: 189}[nb] <= hi


def test_topk_ties_go_to_lower_index():
    sal = np.array([0.0, 5.0, 5.0, 5.0, 1.0, 1.0])
    rp, ci = oracle.topology_csr(sal, 0, 0, 2)
    assert list(ci[rp[5]:rp[6]]) == [1, 2, 5]
    assert list(ci[rp[4]:rp[5]]) == [1, 2, 4]


def test_build_schedule_lane_mean_matches_pieces():
    g = torch.Generator().manual_seed(9)
    K = torch.randn((3, 512, 8), generator=g).to(torch.bfloat16)
    rp, ci, sal = oracle.build_schedule(K, 64, 1, 1, 2)
    C = oracle.centroids(K, 64)
    sal2, _ = oracle.salience(C)
    rp2, ci2 = oracle.topology_csr(sal2, 1, 1, 2)
    assert np.array_equal(sal, sal2) and np.array_equal(rp, rp2) and np.array_equal(ci, ci2)
