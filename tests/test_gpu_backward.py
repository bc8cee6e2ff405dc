"""GPU backward pass (and the forward's log-sum-exp) vs the CPU oracle.

Tolerances come from the arithmetic: P and dS are rounded to the input dtype before they enter
the tensor cores and the gradients are rounded to it at the end, each a relative error of at
most u/2 (u = 2^-8 for bf16, 2^-11 for f16); accumulation is fp32.  Delta = <dO, O> uses the
stored (rounded) O, which adds up to u/2 |dO||O| per row; where one key dominates a row,
dP - Delta nearly cancels and that term is a visible share of dS.  A gradient element is
accepted within 3u of its tensor's largest magnitude, and the rms error must stay below 2u of
the rms value.  The log-sum-exp sums the rounded P of the forward, so it is accepted within u.
"""
import numpy as np
import pytest
import torch

import oracle
import topology_scheduled_gb300 as tsa
from topology_scheduled_gb300.autograd import scheduled_attention
from topology_scheduled_gb300.workloads import WORKLOADS, make_qkv, random_density_csr

pytestmark = pytest.mark.gpu
DEV = "cuda"
U = {torch.float16: 2.0 ** -11, torch.bfloat16: 2.0 ** -8}


def _close(got, ref, u, what):
    got = got.detach().cpu().double().numpy().reshape(ref.shape)
    err = np.abs(got - ref)
    m = np.abs(ref).max()
    assert err.max() <= 3 * u * max(m, 1e-30), f"{what}: max err {err.max():.3g} vs max {m:.3g}"
    assert np.sqrt((err ** 2).mean()) <= 2 * u * np.sqrt((ref ** 2).mean()) + 1e-30, f"{what}: rms"


def _schedule(kind, nb, seed=0):
    if kind == "dense":
        return oracle.dense_causal_csr(nb)
    if kind == "diagonal":
        return np.arange(nb + 1, dtype=np.int32), np.arange(nb, dtype=np.int32)
    if kind == "random":
        return random_density_csr(nb, 0.3, seed)
    if kind == "holes":  # an empty row, a row without its diagonal block, a one-block row
        rng = np.random.default_rng(seed)
        rows = [sorted(set(rng.choice(i + 1, size=rng.integers(1, i + 2), replace=False).tolist()))
                for i in range(nb)]
        rows[1], rows[2], rows[-1] = [], [0], [nb - 1]
        rp = np.zeros(nb + 1, np.int32)
        rp[1:] = np.cumsum([len(r) for r in rows])
        return rp, np.array([j for r in rows for j in r], np.int32)
    raise ValueError(kind)


def _run(Q, K, V, dO, rp, ci, scale):
    rpd, cid = torch.as_tensor(rp, device=DEV), torch.as_tensor(ci, device=DEV)
    O, lse = tsa.tsa_scheduled_attention_fwd(Q.to(DEV), K.to(DEV), V.to(DEV), rpd, cid, scale)
    grads = tsa.tsa_scheduled_attention_backward(Q.to(DEV), K.to(DEV), V.to(DEV), O, dO.to(DEV), lse,
                                                 rpd, cid, scale)
    assert tsa.tsa_last_device_status() == 0
    return O, lse, grads


CASES = [(1, 256, 64, torch.float16, "dense"), (1, 256, 64, torch.bfloat16, "diagonal"),
         (2, 512, 64, torch.float16, "random"), (2, 512, 128, torch.bfloat16, "random"),
         (1, 1024, 128, torch.bfloat16, "dense"), (2, 640, 64, torch.bfloat16, "holes"),
         (1, 576, 128, torch.float16, "holes"), (3, 192, 128, torch.float16, "dense")]


@pytest.mark.parametrize("L,S,D,dtype,kind", CASES)
def test_backward_matches_oracle(L, S, D, dtype, kind):
    g = torch.Generator().manual_seed(S + D)
    Q, K, V, dO = (torch.randn((L, S, D), generator=g).to(dtype) for _ in range(4))
    rp, ci = _schedule(kind, S // 64, seed=L)
    scale = D ** -0.5
    _, lse, (dq, dk, dv) = _run(Q, K, V, dO, rp, ci, scale)
    _, rl = oracle.attention(Q, K, V, rp, ci, 64, scale, return_lse=True, nthreads=8)
    got_l = lse.cpu().double().numpy()
    assert np.array_equal(np.isinf(got_l), np.isinf(rl))
    fin = np.isfinite(rl)
    assert np.abs(got_l[fin] - rl[fin]).max() <= U[dtype]
    rq, rk, rv = oracle.attention_backward(Q, K, V, dO, rp, ci, 64, scale, nthreads=8)
    for name, got, ref in (("dQ", dq, rq), ("dK", dk, rk), ("dV", dv, rv)):
        _close(got, ref, U[dtype], f"{kind} {name}")


def test_wide_score_range_and_4d_input():
    g = torch.Generator().manual_seed(7)
    B, H, S, D = 2, 2, 384, 64
    Q = (torch.randn((B, H, S, D), generator=g) * 3).to(torch.bfloat16)
    K = (torch.randn((B, H, S, D), generator=g) * 3).to(torch.bfloat16)
    V, dO = (torch.randn((B, H, S, D), generator=g).to(torch.bfloat16) for _ in range(2))
    rp, ci = _schedule("random", S // 64, seed=3)
    _, _, (dq, dk, dv) = _run(Q, K, V, dO, rp, ci, 0.125)
    rq, rk, rv = oracle.attention_backward(Q.reshape(-1, S, D), K.reshape(-1, S, D), V.reshape(-1, S, D),
                                           dO.reshape(-1, S, D), rp, ci, 64, 0.125, nthreads=4)
    for name, got, ref in (("dQ", dq, rq), ("dK", dk, rk), ("dV", dv, rv)):
        assert got.shape == (B, H, S, D)
        _close(got, ref, U[torch.bfloat16], name)


def test_autograd_wrapper():
    g = torch.Generator().manual_seed(8)
    L, S, D = 2, 256, 64
    Q, K, V, dO = (torch.randn((L, S, D), generator=g).to(torch.float16) for _ in range(4))
    rp, ci = _schedule("random", S // 64, seed=5)
    q, k, v = (x.to(DEV).requires_grad_(True) for x in (Q, K, V))
    out = scheduled_attention(q, k, v, torch.as_tensor(rp, device=DEV), torch.as_tensor(ci, device=DEV), 0.125)
    out.backward(dO.to(DEV))
    assert tsa.tsa_last_device_status() == 0
    rq, rk, rv = oracle.attention_backward(Q, K, V, dO, rp, ci, 64, 0.125, nthreads=2)
    for name, got, ref in (("dQ", q.grad, rq), ("dK", k.grad, rk), ("dV", v.grad, rv)):
        _close(got, ref, U[torch.float16], name)


@pytest.mark.parametrize("name", ["b4h16s8192", "b2h32s32768"])
def test_full_size_topology_properties(name):
    """Whole workload through the topology schedule.  Exact identities of the gradient hold at
    any size: shifting every key leaves each softmax row unchanged (key gradients sum to zero per
    lane), and softmax rows sum to one (value gradients sum to the upstream gradient).  On
    b4h16s8192 two sampled lanes are also compared with the oracle element by element."""
    w = WORKLOADS[name]
    q, k, v = make_qkv(w, seed=0, device=DEV)
    rp, ci = tsa.tsa_build_schedule(k, w.block, w.sink, w.local_radius, w.topk)
    g = torch.Generator(device=DEV).manual_seed(1)
    dO = torch.randn(q.shape, generator=g, device=DEV).to(q.dtype)
    O, lse = tsa.tsa_scheduled_attention_fwd(q, k, v, rp, ci, w.scale)
    dq, dk, dv = tsa.tsa_scheduled_attention_backward(q, k, v, O, dO, lse, rp, ci, w.scale)
    assert tsa.tsa_last_device_status() == 0
    L, S, D = w.lanes, w.S, w.D
    u = U[q.dtype]
    dk_sum = dk.reshape(L, S, D).double().sum(dim=1)
    dk_scale = dk.reshape(L, S, D).double().abs().sum(dim=1)
    assert (dk_sum.abs() <= 4 * u * dk_scale + 1e-6).all()
    dv_sum = dv.reshape(L, S, D).double().sum(dim=1)
    do_sum = dO.reshape(L, S, D).double().sum(dim=1)  # every row has keys (the diagonal)
    dv_scale = dv.reshape(L, S, D).double().abs().sum(dim=1)
    assert ((dv_sum - do_sum).abs() <= 4 * u * dv_scale + 1e-6).all()
    assert torch.isfinite(dq).all() and torch.isfinite(lse).all()
    if name == "b4h16s8192":
        rph = rp.cpu().numpy()
        cih = ci.cpu().numpy()[: rph[-1]]
        for lane in (0, L - 1):
            sl = lambda t: t.reshape(L, S, D)[lane:lane + 1].cpu()  # noqa: E731
            rq, rk, rv = oracle.attention_backward(sl(q), sl(k), sl(v), sl(dO), rph, cih, 64, w.scale)
            for nm, got, ref in (("dQ", sl(dq), rq), ("dK", sl(dk), rk), ("dV", sl(dv), rv)):
                _close(got, ref, u, f"lane {lane} {nm}")


def test_bad_schedule_is_reported():
    g = torch.Generator().manual_seed(9)
    L, S, D = 1, 256, 64
    Q, K, V, dO = (torch.randn((L, S, D), generator=g).to(torch.float16).to(DEV) for _ in range(4))
    rp = torch.tensor([0, 1, 3, 5, 7], dtype=torch.int32, device=DEV)
    ci = torch.tensor([0, 0, 1, 2, 1, 0, 3], dtype=torch.int32, device=DEV)  # row 2 out of order
    O, lse = tsa.tsa_scheduled_attention_fwd(Q, K, V, rp, ci, 0.125)
    assert tsa.tsa_last_device_status() == 8
    tsa.tsa_scheduled_attention_backward(Q, K, V, O, dO, lse, rp, ci, 0.125)
    assert tsa.tsa_last_device_status() == 8


def test_host_errors():
    L, S, D = 1, 256, 64
    x = torch.zeros((L, S, D), dtype=torch.float16, device=DEV)
    rp, ci = tsa.tsa_dense_causal_csr(S, 64)
    lse = torch.zeros((L, S), dtype=torch.float32, device=DEV)
    L_ = tsa.lib()
    ws = torch.empty(16, dtype=torch.uint8, device=DEV)
    st = L_.tsa_scheduled_attention_backward(x.data_ptr(), x.data_ptr(), x.data_ptr(), x.data_ptr(),
                                             x.data_ptr(), lse.data_ptr(), rp.data_ptr(), ci.data_ptr(),
                                             ci.numel(), x.data_ptr(), x.data_ptr(), x.data_ptr(), 0, 1, 1,
                                             S, D, 64, 0.125, ws.data_ptr(), ws.numel(), None)
    assert st == 1  # outputs alias inputs
    dq, dk, dv = (torch.empty_like(x) for _ in range(3))
    st = L_.tsa_scheduled_attention_backward(x.data_ptr(), x.data_ptr(), x.data_ptr(), x.data_ptr(),
                                             x.data_ptr(), lse.data_ptr(), rp.data_ptr(), ci.data_ptr(),
                                             ci.numel(), dq.data_ptr(), dk.data_ptr(), dv.data_ptr(), 0, 1, 1,
                                             S, D, 64, 0.125, ws.data_ptr(), ws.numel(), None)
    assert st == 5  # workspace too small
    assert tsa.tsa_attention_backward_workspace_bytes(1, 64 * 8193, 64, 10) == 0
