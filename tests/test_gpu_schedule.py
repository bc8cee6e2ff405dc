"""GPU schedule builder vs the CPU oracle: bit-exact CSR and salience.

Covers the dense causal CSR, the topology schedule on every workload shape (single lane,
lane-mean over 64 lanes at S 8192 and S 32768), tiny and ragged inputs (D = 1, block = 1,
one block, ties from duplicated blocks), the largest accepted block count, and the invariant
that exactly one block has zero salience.
"""
import numpy as np
import pytest
import torch

import oracle
import topology_scheduled_gb300 as tsa
from topology_scheduled_gb300.workloads import WORKLOADS, make_qkv

pytestmark = pytest.mark.gpu
DEV = "cuda"


def _trim(rp, ci):
    rp = rp.cpu().numpy()
    return rp, ci.cpu().numpy()[: rp[-1]]


def _gpu_schedule(K, block, sink, r, topk):
    rp, ci, sal = tsa.tsa_build_schedule(K, block, sink, r, topk, salience=True)
    assert tsa.tsa_last_device_status() == 0
    rp, ci = _trim(rp, ci)
    return rp, ci, sal.cpu().numpy()


def _oracle_schedule(K, block, sink, r, topk):
    S, D = K.shape[-2], K.shape[-1]
    return oracle.build_schedule(K.detach().cpu().reshape(-1, S, D), block, sink, r, topk)


def _assert_same(gpu, ref, distinct=True):
    rp, ci, sal = gpu
    rp_o, ci_o, sal_o = ref
    assert np.array_equal(sal.view(np.uint64), sal_o.view(np.uint64)), "salience bits differ"
    assert np.array_equal(rp, rp_o), "row_ptr differs"
    assert np.array_equal(ci, ci_o), "col_idx differs"
    # exactly one block is never absorbed; coincident centroids add zero-distance merges
    assert int(np.sum(sal == 0)) == 1 if distinct else int(np.sum(sal == 0)) >= 1


@pytest.mark.parametrize("nb", [1, 2, 3, 16, 32, 64, 255, 512, 1025])
def test_dense_csr_bit_exact(nb):
    rp, ci = tsa.tsa_dense_causal_csr(nb * 64, 64)
    rp_o, ci_o = oracle.dense_causal_csr(nb)
    assert np.array_equal(rp.cpu().numpy(), rp_o)
    assert np.array_equal(ci.cpu().numpy(), ci_o)
    if nb in (16, 32, 64):
        assert int(rp_o[-1]) == {16: 136, 32: 528, 64: 2080}[nb]


@pytest.mark.parametrize("name", ["s1024", "s2048", "s4096"])
def test_topology_single_lane_workloads(name):
    w = WORKLOADS[name]
    _, k, _ = make_qkv(w, seed=0, device=DEV)
    gpu = _gpu_schedule(k, w.block, w.sink, w.local_radius, w.topk)
    ref = _oracle_schedule(k, w.block, w.sink, w.local_radius, w.topk)
    _assert_same(gpu, ref)
    nnz = int(gpu[0][-1])
    assert nnz <= tsa.tsa_schedule_max_nnz(w.S, w.block, w.sink, w.local_radius, w.topk)


@pytest.mark.parametrize("name", ["b4h16s8192", "b2h32s32768"])
def test_topology_lane_mean_workloads(name):
    w = WORKLOADS[name]
    _, k, _ = make_qkv(w, seed=0, device=DEV)
    gpu = _gpu_schedule(k, w.block, w.sink, w.local_radius, w.topk)
    ref = _oracle_schedule(k, w.block, w.sink, w.local_radius, w.topk)
    _assert_same(gpu, ref)


def _hand_cases():
    rows = [l.split() for l in open("tests/golden/elder_rule_examples.txt") if l.strip() and not l.startswith("#")]
    return [([float(x) for x in r[1:]], [float(x) for x in rows[i + 1][1:]])
            for i, r in enumerate(rows) if r[0] == "points"]


def test_hand_worked_elder_cases_on_gpu():
    for points, sal in _hand_cases():
        k = torch.tensor(points, dtype=torch.float16, device=DEV).view(1, -1, 1)
        _, _, got = _gpu_schedule(k, 1, 0, 0, 0)
        assert list(got) == sal


@pytest.mark.parametrize("seed", range(12))
def test_random_small_and_ragged(seed):
    g = np.random.default_rng(seed)
    lanes = int(g.integers(1, 5))
    block = int(g.choice([1, 2, 8, 64]))
    nb = int(g.integers(1, 70))
    D = int(g.choice([1, 3, 8, 64, 128]))
    dtype = torch.float16 if seed % 2 else torch.bfloat16
    gen = torch.Generator().manual_seed(seed)
    k = torch.randn((lanes, nb * block, D), generator=gen)
    if seed % 3 == 0 and nb > 3:  # duplicated blocks force distance ties
        k[:, block:2 * block] = k[:, 0:block]
        k[:, 3 * block:4 * block] = k[:, 0:block]
    if seed % 4 == 1:  # small integers: many exactly equal distances
        k = torch.randint(-2, 3, k.shape, generator=gen).float()
    k = k.to(dtype).to(DEV)
    sink, r, topk = int(g.integers(0, 3)), int(g.integers(0, 4)), int(g.integers(0, 6))
    _assert_same(_gpu_schedule(k, block, sink, r, topk), _oracle_schedule(k, block, sink, r, topk),
                 distinct=(seed % 3 != 0 and seed % 4 != 1 and D * block > 2))


@pytest.mark.parametrize("nb,dtype,jmax", [(40, torch.float16, 4), (300, torch.float16, 1024),
                                           (300, torch.bfloat16, 4)])
def test_distances_below_binary32_resolution(nb, dtype, jmax):
    """Blocks of two tokens, (2048, ...) and (j * 2^-14, ...): centroids 1024 + j * 2^-15, whose
    last bits lie below the binary32 resolution at 1024 (2^-13).  With j < 4 the rows collapse
    to a handful of binary32 values (and a few dozen binary64 ones, so exact ties abound); with
    j < 1024 they stay apart but a binary32 difference can be off by half its size.  Either way the binary32
    distance intervals cannot order the edges and the binary64 keys decide.  Every 7th block
    sits at -2048, so that some edges are excluded by their bounds.  Covers the per-pair
    interval kernel (nb < 256) and the tiled one."""
    D, block = 3, 2
    g = torch.Generator().manual_seed(nb + jmax)
    x = torch.zeros((1, nb * block, D))
    x[0, 0::2] = 2048.0
    x[0, 0::14] = -2048.0
    x[0, 1::2] = torch.randint(0, jmax, (nb, D), generator=g).float() * 2.0 ** -14
    k = x.to(dtype)
    assert torch.equal(k.float(), x)  # every key exact in the key format
    kd = k.to(DEV)
    _assert_same(_gpu_schedule(kd, block, 1, 2, 4), _oracle_schedule(kd, block, 1, 2, 4), distinct=False)


@pytest.mark.parametrize("spread", [0, 16, 24, 60])
def test_lane_sum_integer_path_and_fallback(spread):
    """Lane means over 5 lanes whose keys differ in scale by up to 2^spread.  At 0 and 16 the
    block sums of all lanes fit 53 bits at their common lowest bit in every column, so the lane
    sum is exact and the GPU adds integers; at 24 about a quarter of the columns do (a mix of
    both paths in one launch); at 60 none do and it adds in binary64 lane by lane.  Either way
    the CSR and the salience equal the oracle's bit for bit."""
    g = torch.Generator().manual_seed(100 + spread)
    lanes, nb, D = 5, 20, 8
    x = torch.randn((lanes, nb * 64, D), generator=g)
    x = x * torch.pow(2.0, torch.tensor([0.0, spread, -spread / 2, spread / 3, 1.0])).view(lanes, 1, 1)
    k = x.to(torch.bfloat16).to(DEV)
    _assert_same(_gpu_schedule(k, 64, 1, 2, 3), _oracle_schedule(k, 64, 1, 2, 3))


def _fuzz_keys(seed):
    """Seeded keys for the builder fuzz test: one of several distributions that stress the
    binary32 distance intervals (near-ties, coincident blocks, magnitudes on both sides of the
    2^+-60 limits where a block's intervals become [0, +inf])."""
    g = np.random.default_rng(1000 + seed)
    lanes = int(g.integers(1, 4))
    block = int(g.choice([1, 4, 16, 64]))
    nb = int(g.integers(2, 90))
    D = int(g.choice([1, 2, 5, 16, 64, 128]))
    kind = seed % 6
    dtype = torch.bfloat16 if (seed // 6) % 2 == 0 else torch.float16
    shape = (lanes, nb * block, D)
    if kind == 0:    # iid Gaussian
        x = g.normal(size=shape)
    elif kind == 1:  # few clusters with small noise: many near-equal distances
        means = g.normal(scale=2.0, size=(4, D))
        x = means[g.integers(0, 4, size=nb)].repeat(block, axis=0)[None] + g.normal(scale=1e-2, size=shape)
    elif kind == 2:  # blocks repeated exactly: zero distances and exact ties
        base = g.normal(size=(lanes, 3 * block, D))
        x = np.concatenate([base] * (nb // 3 + 1), axis=1)[:, : nb * block]
    elif kind == 3:  # heavy tails
        x = g.standard_t(1.5, size=shape)
    elif kind == 4:  # large magnitudes: around 2^60 in bf16, near the top of the f16 range
        if dtype == torch.bfloat16:
            x = g.normal(size=shape) * (2.0 ** g.integers(55, 66))
        else:
            x = np.clip(g.normal(size=shape) * 3e4, -6e4, 6e4)
    else:            # tiny magnitudes around 2^-60 (f16 flushes them to zero or subnormals)
        x = g.normal(size=shape) * (2.0 ** -g.integers(55, 66))
    sink, r, topk = int(g.integers(0, 3)), int(g.integers(0, 3)), int(g.integers(0, 6))
    return torch.as_tensor(x, dtype=torch.float32).to(dtype), block, sink, r, topk, kind


@pytest.mark.parametrize("seed", range(48))
def test_builder_fuzz_against_oracle(seed):
    """Random shapes and distributions: the GPU schedule (built on binary32 distance intervals
    with exact binary64 keys where they decide) equals the oracle's bit for bit."""
    k, block, sink, r, topk, kind = _fuzz_keys(seed)
    assert torch.isfinite(k.float()).all()
    kd = k.to(DEV)
    _assert_same(_gpu_schedule(kd, block, sink, r, topk), _oracle_schedule(kd, block, sink, r, topk),
                 distinct=False)


@pytest.mark.parametrize("D,dtype", [(1000, torch.bfloat16), (1024, torch.float16), (1024, torch.bfloat16)])
def test_widest_head_dim(D, dtype):
    """The builder's widest head dimension (1024; the distance intervals' error budget is sized
    for it) and a width that is not a multiple of 32: bit-exact CSR and salience, with keys
    drawn around 8 cluster means so that many distances nearly tie."""
    g = torch.Generator().manual_seed(D)
    nb, block, lanes = 60, 4, 2
    means = torch.randn((8, D), generator=g)
    which = torch.randint(0, 8, (nb,), generator=g)
    x = means[which].repeat_interleave(block, dim=0)[None].repeat(lanes, 1, 1)
    x = x + 0.01 * torch.randn((lanes, nb * block, D), generator=g)
    kd = x.to(dtype).to(DEV)
    _assert_same(_gpu_schedule(kd, block, 1, 2, 4), _oracle_schedule(kd, block, 1, 2, 4), distinct=False)


def test_largest_block_count():
    nb = 4096
    gen = torch.Generator().manual_seed(7)
    k = torch.randn((1, nb * 4, 16), generator=gen).to(torch.bfloat16).to(DEV)
    _assert_same(_gpu_schedule(k, 4, 2, 3, 5), _oracle_schedule(k, 4, 2, 3, 5))


def test_special_cases_reduce_to_dense_and_diagonal():
    gen = torch.Generator().manual_seed(11)
    k = torch.randn((2, 40 * 64, 64), generator=gen).to(torch.float16).to(DEV)
    rp, ci, _ = _gpu_schedule(k, 64, 0, 39, 0)
    rp_o, ci_o = oracle.dense_causal_csr(40)
    assert np.array_equal(rp, rp_o) and np.array_equal(ci, ci_o)
    rp, ci, _ = _gpu_schedule(k, 64, 0, 0, 0)
    assert np.array_equal(rp, np.arange(41)) and np.array_equal(ci, np.arange(40))


def test_host_errors_with_device_tensors():
    k = torch.randn((1, 256, 64), device=DEV).to(torch.float16)
    with pytest.raises(tsa.TsaError) as e:
        tsa.tsa_build_schedule(k, 64, 1, 1, 2, col_idx=torch.empty(3, dtype=torch.int32, device=DEV))
    assert e.value.status == 5
    L = tsa.lib()
    rp = torch.empty(5, dtype=torch.int32, device=DEV)
    ci = torch.empty(10, dtype=torch.int32, device=DEV)
    ws = torch.empty(tsa.tsa_build_schedule_workspace_bytes(1, 256, 64, 64), dtype=torch.uint8, device=DEV)
    host_k = torch.randn((1, 256, 64)).to(torch.float16)
    st = L.tsa_build_schedule(host_k.data_ptr(), 0, 1, 256, 64, 64, 1, 1, 2, rp.data_ptr(), ci.data_ptr(),
                              10, None, ws.data_ptr(), ws.numel(), None)
    assert st == 3


@pytest.mark.parametrize("dtype", [torch.bfloat16, torch.float16])
def test_centroid_sums_with_extreme_exponents(dtype):
    """Keys spread over ~75 binades (subnormals, values outside the integer window, widely
    spread columns): the block sums must still equal the sequential binary64 sums."""
    g = torch.Generator().manual_seed(5)
    lanes, nb, D = 3, 24, 64
    x = torch.randn((lanes, nb * 64, D), generator=g)
    hi = 30 if dtype == torch.bfloat16 else 13
    e = torch.randint(-45, hi, x.shape, generator=g).float()
    x = x * torch.pow(2.0, e)
    x[:, :64, :8] = 1e-30  # columns of tiny values only (f16: zero, bf16: below the window)
    k = x.to(dtype).to(DEV)
    _assert_same(_gpu_schedule(k, 64, 1, 2, 3), _oracle_schedule(k, 64, 1, 2, 3), distinct=False)


@pytest.mark.parametrize("dtype", [torch.bfloat16, torch.float16])
@pytest.mark.parametrize("lanes,S", [(1, 1000), (16, 40000 - 23)])
def test_block_sums_small_and_large_grids(dtype, lanes, S):
    """Block sums against the sequential binary64 sum (tokens ascending) on a few CTAs (one
    64-row block in flight per thread) and on a many-wave grid (a ring of 8-row chunks), with
    columns whose exponents spread past the fast paths' bounds and a partial last block."""
    D, block = 64, 64
    g = torch.Generator().manual_seed(lanes + S)
    x = torch.randn((lanes, S, D), generator=g)
    lo_e, hi_e = (-24, 12) if dtype == torch.bfloat16 else (-20, 8)
    x = x * torch.pow(2.0, torch.randint(lo_e, hi_e, (lanes, S, D), generator=g).float())
    k = x.to(dtype)
    got = tsa.tsa_block_sums(k.to(DEV), block).cpu().numpy()
    nb = -(-S // block)
    xd = np.zeros((lanes, nb * block, D))
    xd[:, :S] = k.double().numpy()
    xd = xd.reshape(lanes, nb, block, D)
    ref = np.zeros((lanes, nb, D))
    for t in range(block):
        ref = ref + xd[:, :, t, :]  # padding rows add +0.0, which leaves a sum unchanged
    assert np.array_equal(got, ref)
