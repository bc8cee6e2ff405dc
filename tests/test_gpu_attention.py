"""GPU scheduled attention vs the fp64 CPU oracle, element by element.

Tolerance (max abs error against the unrounded fp64 oracle): 2e-3 for fp16 and 1e-2 for
bf16 inputs/outputs, fp32 accumulation on the GPU -- except for outputs whose magnitude makes
the dtype's own spacing coarser than that, which must be within the bound plus half an ulp of
the output format, and never more than one ulp (tests/_tol.py).

Small cases cover every schedule shape the kernel meets -- dense, diagonal-only, random
density, topology, rows without their diagonal, empty rows, odd block counts (a query-block
pair with one block), several lanes, both head dims and both dtypes.  Full-size workloads
(S 1024 .. 32768, up to 64 lanes) are compared on sampled rows in the same launch
configuration the benchmark times.
"""
import numpy as np
import pytest
import torch

import oracle
import topology_scheduled_gb300 as tsa
from topology_scheduled_gb300.workloads import WORKLOADS, make_qkv, random_density_csr

pytestmark = pytest.mark.gpu
DEV = "cuda"
from _tol import TOL, assert_close  # noqa: E402,F401


def _run(q, k, v, rp, ci, scale):
    rp_d = torch.as_tensor(np.asarray(rp), dtype=torch.int32, device=DEV)
    ci_d = torch.as_tensor(np.asarray(ci) if len(ci) else np.zeros(1, np.int32), dtype=torch.int32, device=DEV)
    out = tsa.tsa_scheduled_attention(q.to(DEV), k.to(DEV), v.to(DEV), rp_d, ci_d, scale)
    assert tsa.tsa_last_device_status() == 0
    return out.cpu()


def _compare_full(q, k, v, rp, ci, scale):
    out = _run(q, k, v, rp, ci, scale)
    S, D = q.shape[-2], q.shape[-1]
    ref = oracle.attention(q.reshape(-1, S, D), k.reshape(-1, S, D), v.reshape(-1, S, D), rp, ci, 64, scale,
                           nthreads=8)
    return assert_close(out.reshape(-1, S, D).double().numpy(), ref, q.dtype)


def _qkv(L, S, D, dtype, seed, kscale=1.0):
    g = torch.Generator().manual_seed(seed)
    q = torch.randn((L, S, D), generator=g).to(dtype)
    k = (torch.randn((L, S, D), generator=g) * kscale).to(dtype)
    v = torch.randn((L, S, D), generator=g).to(dtype)
    return q, k, v


CASES = [(1, 128, 64), (1, 192, 64), (3, 256, 128), (2, 320, 128), (1, 64, 64), (2, 1024, 64)]


@pytest.mark.parametrize("dtype", [torch.float16, torch.bfloat16])
@pytest.mark.parametrize("L,S,D", CASES)
def test_dense_schedule(dtype, L, S, D):
    q, k, v = _qkv(L, S, D, dtype, S + D)
    rp, ci = oracle.dense_causal_csr(S // 64)
    _compare_full(q, k, v, rp, ci, D ** -0.5)


@pytest.mark.parametrize("dtype", [torch.float16, torch.bfloat16])
@pytest.mark.parametrize("L,S,D", CASES)
def test_diagonal_only(dtype, L, S, D):
    q, k, v = _qkv(L, S, D, dtype, 1 + S)
    nb = S // 64
    _compare_full(q, k, v, np.arange(nb + 1, dtype=np.int32), np.arange(nb, dtype=np.int32), D ** -0.5)


@pytest.mark.parametrize("density", [0.1, 0.5])
@pytest.mark.parametrize("D,dtype", [(64, torch.float16), (128, torch.bfloat16)])
def test_random_density(density, D, dtype):
    S = 1536
    q, k, v = _qkv(2, S, D, dtype, 5, kscale=2.0)
    rp, ci = random_density_csr(S // 64, density, 3)
    _compare_full(q, k, v, rp, ci, D ** -0.5)


def test_rows_without_diagonal_and_empty_rows():
    S, D = 512, 64
    q, k, v = _qkv(2, S, D, torch.float16, 9)
    # rows: 0 {0}, 1 {} , 2 {0}, 3 {1,2}, 4 {4}, 5 {}, 6 {0,3,6}, 7 {2,5}
    rows = [[0], [], [0], [1, 2], [4], [], [0, 3, 6], [2, 5]]
    rp = np.zeros(9, np.int32)
    rp[1:] = np.cumsum([len(r) for r in rows])
    ci = np.array([j for r in rows for j in r], np.int32)
    _compare_full(q, k, v, rp, ci, 0.125)


def test_wide_score_range_exercises_rescaling():
    S, D = 2048, 128
    q, k, v = _qkv(1, S, D, torch.bfloat16, 21, kscale=6.0)
    rp, ci = oracle.dense_causal_csr(S // 64)
    _compare_full(q, k, v, rp, ci, D ** -0.5)


@pytest.mark.parametrize("dtype,growth", [(torch.float16, 4.0), (torch.bfloat16, 8.0)])
def test_running_maximum_grows_past_the_rescale_threshold(dtype, growth):
    """Key block j scaled by growth * (j + 1): each block's row maxima exceed the previous ones
    by more than the lazy-rescale threshold (2^15 for f16, 2^30 for bf16), so the kernel must
    rescale O and the denominator many times along every dense row."""
    S, D = 1024, 64
    g = torch.Generator().manual_seed(77)
    q = torch.randn((2, S, D), generator=g)
    kscale = growth * (torch.arange(S) // 64 + 1).float().view(1, S, 1)
    k = torch.randn((2, S, D), generator=g) * kscale
    v = torch.randn((2, S, D), generator=g)
    q, k, v = (x.to(dtype) for x in (q, k, v))
    rp, ci = oracle.dense_causal_csr(S // 64)
    _compare_full(q, k, v, rp, ci, D ** -0.5)


def test_four_dim_input_and_dtype_preserved():
    g = torch.Generator().manual_seed(3)
    q, k, v = (torch.randn((2, 3, 256, 64), generator=g).to(torch.bfloat16) for _ in range(3))
    rp, ci = oracle.dense_causal_csr(4)
    out = tsa.tsa_scheduled_attention(q.to(DEV), k.to(DEV), v.to(DEV), torch.as_tensor(rp, device=DEV),
                                      torch.as_tensor(ci, device=DEV))
    assert out.shape == q.shape and out.dtype == torch.bfloat16
    ref = oracle.attention(q, k, v, rp, ci, 64, 0.125)
    assert_close(out.cpu().double().numpy().reshape(ref.shape), ref, torch.bfloat16)


def test_bad_schedule_is_reported_not_read():
    S, D = 256, 64
    q, k, v = _qkv(1, S, D, torch.float16, 2)
    rp = torch.tensor([0, 1, 3, 5, 7], dtype=torch.int32, device=DEV)
    ci = torch.tensor([0, 0, 9, 0, 1, 3, 2], dtype=torch.int32, device=DEV)  # 9 > 1 and 3 before 2
    tsa.tsa_scheduled_attention(q.to(DEV), k.to(DEV), v.to(DEV), rp, ci, 0.125)
    assert tsa.tsa_last_device_status() == 8
    assert tsa.tsa_last_device_status() == 0  # read clears


def test_host_errors_with_device_tensors():
    q, k, v = (x.to(DEV) for x in _qkv(1, 128, 64, torch.float16, 1))
    rp, ci = tsa.tsa_dense_causal_csr(128)
    with pytest.raises(tsa.TsaError) as e:
        tsa.tsa_scheduled_attention(q, k, v, rp.cpu(), ci, 0.1)
    assert e.value.status == 3
    with pytest.raises(tsa.TsaError) as e:
        tsa.tsa_scheduled_attention(q, k, v, rp, ci, 0.1, out=q)
    assert e.value.status == 1


# ---------------------------------------------------------------- full-size workloads
def _sample_rows(L, S, rng, n_lanes=3, n_random=192):
    lanes = rng.choice(L, size=min(L, n_lanes), replace=False)
    toks = [np.arange(0, 64), np.arange(S - 64, S), np.arange(S // 2, S // 2 + 64)]
    ls, ts = [], []
    for l in lanes:
        t = np.concatenate(toks + [rng.integers(0, S, n_random)])
        ls.append(np.full(t.shape, l))
        ts.append(t)
    return np.concatenate(ls).astype(np.int64), np.concatenate(ts).astype(np.int64)


def _full_size(w, rp_d, ci_d, q, k, v):
    out = tsa.tsa_scheduled_attention(q, k, v, rp_d, ci_d, w.scale)
    assert tsa.tsa_last_device_status() == 0
    rp = rp_d.cpu().numpy()
    ci = ci_d.cpu().numpy()[: rp[-1]]
    S, D = w.S, w.D
    lanes, toks = _sample_rows(w.lanes, S, np.random.default_rng(0))
    qh, kh, vh = (x.cpu().reshape(-1, S, D) for x in (q, k, v))
    ref = oracle.attention(qh, kh, vh, rp, ci, 64, w.scale, lanes=lanes, tokens=toks, nthreads=16)
    got = out.reshape(-1, S, D)[torch.as_tensor(lanes, device=out.device), torch.as_tensor(toks, device=out.device)]
    err = assert_close(got.cpu().double().numpy(), ref, w.dtype)
    assert torch.isfinite(out).all()
    return err


@pytest.mark.parametrize("name", ["s1024", "s2048", "s4096"])
def test_single_lane_workloads_topology_and_dense(name):
    w = WORKLOADS[name]
    q, k, v = make_qkv(w, seed=0, device=DEV)
    rp, ci = tsa.tsa_build_schedule(k, w.block, w.sink, w.local_radius, w.topk)
    _full_size(w, rp, ci, q, k, v)
    rp, ci = tsa.tsa_dense_causal_csr(w.S, w.block)
    _full_size(w, rp, ci, q, k, v)


@pytest.mark.parametrize("name", ["b4h16s8192", "b2h32s32768"])
def test_lane_mean_workloads(name):
    w = WORKLOADS[name]
    q, k, v = make_qkv(w, seed=0, device=DEV)
    rp, ci = tsa.tsa_build_schedule(k, w.block, w.sink, w.local_radius, w.topk)
    _full_size(w, rp, ci, q, k, v)


@pytest.mark.parametrize("density", [0.02, 0.05, 0.10, 0.25, 0.50, 1.0])
def test_density_sweep_workload(density):
    w = WORKLOADS["b1h32s16384"]
    q, k, v = make_qkv(w, seed=0, device=DEV)
    rp, ci = random_density_csr(w.nb, density, 0)
    if density == 1.0:
        assert rp[-1] == 32896
    _full_size(w, torch.as_tensor(rp, device=DEV), torch.as_tensor(ci, device=DEV), q, k, v)
