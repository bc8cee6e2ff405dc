"""Pins for the elder rule's two tie rules (block index and centroid content).

What pins what:
* hand-worked cases under both rules, including one where IEEE totalOrder (-0 before +0)
  decides -- tests/golden/tie_break_examples.txt;
* permutation equivariance of the content rule (the property the pages say the index rule
  lacks), bitwise, on random centroids and end to end from keys whose blocks are permuted;
* what both rules share: the H0 barcode (multiset of saliences), the MST edge set, exactly
  one zero, and the sum of saliences equal to the MST weight;
* bit-identical centroids, where the content rule falls back to the index rule.
"""
import os

import numpy as np
import pytest
import torch

import oracle

GOLDEN = os.path.join(os.path.dirname(__file__), "golden")


def _cases():
    cases, cur = [], None
    for line in open(os.path.join(GOLDEN, "tie_break_examples.txt")):
        if not line.strip() or line.startswith("#"):
            continue
        f = line.split()
        if f[0] == "points":
            cur = {"C": np.array([[float(x)] for x in f[1:]])}
            cases.append(cur)
        elif f[0] == "points2":
            cur = {"C": np.array([[float(v) for v in x.split(",")] for x in f[1:]])}
            cases.append(cur)
        else:
            cur[f[0]] = np.array([float(x) for x in f[1:]])
    return cases


def test_hand_worked_tie_cases():
    cases = _cases()
    assert len(cases) == 4
    for c in cases:
        for rule in ("index", "content"):
            sal, _ = oracle.salience(c["C"], tie=rule)
            assert np.array_equal(sal, c[rule]), (c["C"].tolist(), rule, sal)


def _random_centroids(seed, nb=40, D=3):
    rng = np.random.default_rng(seed)
    return rng.standard_normal((nb, D))


@pytest.mark.parametrize("seed", range(5))
def test_content_rule_is_permutation_equivariant(seed):
    C = _random_centroids(seed)
    sal, _ = oracle.salience(C, tie="content")
    rng = np.random.default_rng(100 + seed)
    index_moved = False
    for _ in range(4):
        perm = rng.permutation(C.shape[0])
        sal_p, _ = oracle.salience(C[perm], tie="content")
        assert np.array_equal(sal_p, sal[perm])
        sal_i, _ = oracle.salience(C, tie="index")
        sal_ip, _ = oracle.salience(C[perm], tie="index")
        index_moved |= not np.array_equal(sal_ip, sal_i[perm])
    # every first merge of two singletons is a size tie, so the index rule moves scores
    assert index_moved


@pytest.mark.parametrize("seed", range(5))
def test_rules_share_barcode_and_mst(seed):
    C = _random_centroids(seed, nb=33, D=4)
    res = {rule: oracle.salience(C, tie=rule) for rule in ("index", "content")}
    (si, (ui, vi, di)), (sc, (uc, vc, dc)) = res["index"], res["content"]
    assert np.array_equal(np.sort(si), np.sort(sc))
    assert {frozenset(e) for e in zip(ui, vi)} == {frozenset(e) for e in zip(uc, vc)}
    for s, d in ((si, di), (sc, dc)):
        assert np.count_nonzero(s == 0.0) == 1
        assert np.isclose(s.sum(), d.sum(), rtol=1e-12)


def test_identical_centroids_fall_back_to_index():
    C = np.ones((9, 3))
    si, _ = oracle.salience(C, tie="index")
    sc, _ = oracle.salience(C, tie="content")
    assert np.array_equal(si, sc) and not si.any()
    C = np.array([[2.0], [5.0], [2.0], [5.0], [2.0]])
    si, mi = oracle.salience(C, tie="index")
    sc, mc = oracle.salience(C, tie="content")
    assert np.array_equal(np.sort(si), np.sort(sc))


@pytest.mark.parametrize("dtype", [torch.float16, torch.bfloat16])
def test_end_to_end_block_permutation(dtype):
    """Moving whole key blocks (every lane) moves each centroid exactly, so the content-rule
    salience follows the blocks."""
    g = torch.Generator().manual_seed(9)
    L, nb, block, D = 3, 24, 8, 6
    K = torch.randn((L, nb * block, D), generator=g).to(dtype)
    perm = torch.randperm(nb, generator=g)
    Kp = K.view(L, nb, block, D)[:, perm].reshape(L, nb * block, D).contiguous()
    _, _, sal = oracle.build_schedule(K, block, 1, 1, 2, tie="content")
    _, _, sal_p = oracle.build_schedule(Kp, block, 1, 1, 2, tie="content")
    assert np.array_equal(sal_p, sal[perm.numpy()])
