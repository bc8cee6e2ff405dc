"""GPU schedule builder under the content tie rule vs the CPU oracle: bit-exact salience and
CSR, and the permutation equivariance the content rule exists for."""
import numpy as np
import pytest
import torch

import oracle
import topology_scheduled_gb300 as tsa
from topology_scheduled_gb300.workloads import WORKLOADS, make_qkv

pytestmark = pytest.mark.gpu
DEV = "cuda"


def _gpu(K, block, sink, r, topk, tie="content"):
    rp, ci, sal = tsa.tsa_build_schedule(K, block, sink, r, topk, salience=True, tie_break=tie)
    assert tsa.tsa_last_device_status() == 0
    rp = rp.cpu().numpy()
    return rp, ci.cpu().numpy()[: rp[-1]], sal.cpu().numpy()


def _ref(K, block, sink, r, topk, tie="content"):
    S, D = K.shape[-2], K.shape[-1]
    return oracle.build_schedule(K.detach().cpu().reshape(-1, S, D), block, sink, r, topk, tie=tie)


def _same(a, b):
    assert np.array_equal(a[2].view(np.uint64), b[2].view(np.uint64)), "salience bits differ"
    assert np.array_equal(a[0], b[0]) and np.array_equal(a[1], b[1]), "CSR differs"


@pytest.mark.parametrize("name", ["s1024", "s2048", "s4096", "b4h16s8192", "b2h32s32768"])
def test_content_rule_workloads(name):
    w = WORKLOADS[name]
    _, k, _ = make_qkv(w, seed=0, device=DEV)
    _same(_gpu(k, w.block, w.sink, w.local_radius, w.topk),
          _ref(k, w.block, w.sink, w.local_radius, w.topk))


def test_hand_worked_tie_cases_on_gpu():
    rows = [l.split() for l in open("tests/golden/tie_break_examples.txt")
            if l.strip() and not l.startswith("#")]
    n = 0
    for i, r in enumerate(rows):
        if r[0] == "points":
            pts = [[float(x)] for x in r[1:]]
        else:
            # 2-D cases pin signed-zero order on raw centroids; a centroid built from keys is
            # never -0 (its sum starts at +0, and +0 + -0 = +0), so they stay oracle-only
            continue
        k = torch.tensor(pts, dtype=torch.float16, device=DEV).view(1, len(pts), -1)
        for rule_row in rows[i + 1:i + 3]:
            _, _, got = _gpu(k, 1, 0, 0, 0, tie=rule_row[0])
            assert list(got) == [float(x) for x in rule_row[1:]], (pts, rule_row[0])
            n += 1
    assert n == 6


@pytest.mark.parametrize("seed", range(10))
def test_content_rule_random_and_ragged(seed):
    g = np.random.default_rng(seed)
    lanes, block = int(g.integers(1, 5)), int(g.choice([1, 2, 8, 64]))
    nb, D = int(g.integers(1, 90)), int(g.choice([1, 3, 8, 64, 128]))
    dtype = torch.float16 if seed % 2 else torch.bfloat16
    gen = torch.Generator().manual_seed(seed)
    k = torch.randn((lanes, nb * block, D), generator=gen)
    if seed % 3 == 0 and nb > 3:  # duplicated blocks: identical centroids fall back to the index
        k[:, block:2 * block] = k[:, 0:block]
        k[:, 3 * block:4 * block] = k[:, 0:block]
    if seed % 4 == 1:  # small integers: many equal distances and equal leading coordinates
        k = torch.randint(-2, 3, k.shape, generator=gen).float()
    if seed % 5 == 2:  # equal leading coordinates (the -0 keys sum to +0 centroids)
        k[:, :, 0] = 0.0
        k[:, : nb * block // 2, 0] = -0.0
    k = k.to(dtype).to(DEV)
    sink, r, topk = int(g.integers(0, 3)), int(g.integers(0, 4)), int(g.integers(0, 6))
    _same(_gpu(k, block, sink, r, topk), _ref(k, block, sink, r, topk))


@pytest.mark.parametrize("nb", [97, 512, 4096])
def test_content_rule_is_permutation_equivariant_on_gpu(nb):
    gen = torch.Generator().manual_seed(nb)
    L, block, D = 2, 4, 32
    k = torch.randn((L, nb * block, D), generator=gen).to(torch.bfloat16)
    perm = torch.randperm(nb, generator=gen)
    kp = k.view(L, nb, block, D)[:, perm].reshape(L, nb * block, D).contiguous()
    sal = _gpu(k.to(DEV), block, 1, 1, 2)[2]
    sal_p = _gpu(kp.to(DEV), block, 1, 1, 2)[2]
    assert np.array_equal(sal_p.view(np.uint64), sal[perm.numpy()].view(np.uint64))
    # the index rule gives the same barcode but moves the scores
    sal_i = _gpu(k.to(DEV), block, 1, 1, 2, tie="index")[2]
    sal_ip = _gpu(kp.to(DEV), block, 1, 1, 2, tie="index")[2]
    assert np.array_equal(np.sort(sal_i), np.sort(sal))
    assert not np.array_equal(sal_ip, sal_i[perm.numpy()])


def test_unknown_tie_rule_is_rejected():
    k = torch.zeros((1, 256, 64), dtype=torch.float16, device=DEV)
    with pytest.raises(ValueError):
        tsa.tsa_build_schedule(k, tie_break="size")
