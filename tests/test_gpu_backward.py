"""GPU backward pass (and the forward's log-sum-exp) vs the CPU oracle.

Tolerances come from the arithmetic, element by element.  With r the unit roundoff of the
input dtype (2^-8 for bf16, 2^-11 for f16) and fp32 accumulation (a sum of n terms is off by at
most n 2^-24 times the sum of their magnitudes):
  * P = exp(scale s - lse) uses the forward's log-sum-exp (within r of the oracle's, checked
    below) and is rounded to the input dtype before the tensor cores: |dP_err| <= 2r P, plus
    the score's own fp32 error, scale D 2^-24 (|Q| |K|^T);
  * Delta = <dO, O> uses the stored O, whose error is at most r|O| (rounding) plus 2r (P |V|)
    (the forward's rounded P): |Delta_err| <= sum_d |dO| (r|O| + 2r P|V|);
  * dS = P o (dP - Delta) is rounded to the input dtype (r |dS|), and dP = dO V^T carries
    D 2^-24 (|dO| |V|^T);
  * dQ = scale dS K, dK = scale dS^T Q and dV = P^T dO are fp32 sums of those terms, rounded
    to the input dtype at the end (r |grad|).
Each gradient element must lie within 1.5x the bound these terms give for it, and the rms
error must stay below 2r of the rms value.  The log-sum-exp sums the rounded P of the
forward, so it is accepted within r.
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
# half the spacing of the dtype's subnormals: the absolute rounding error of a value below the
# smallest normal (2^-14 in f16, 2^-126 in bf16)
ETA = {torch.float16: 2.0 ** -25, torch.bfloat16: 2.0 ** -134}


def _allowed(rp, ci, S, block=64):
    """Boolean [S, S] mask of the keys each query may see: its CSR row's blocks, keys <= query."""
    M = np.zeros((S, S), dtype=bool)
    for i in range(len(rp) - 1):
        for j in ci[rp[i]:rp[i + 1]]:
            M[i * block:(i + 1) * block, j * block:(j + 1) * block] = True
    return M & np.tril(np.ones((S, S), dtype=bool))


def _bounds(Q, K, V, dO, rp, ci, scale, r, eta, block=64, rows=512):
    """Per-element error bounds of dQ, dK, dV (see the module docstring), [L, S, D] each."""
    Qn, Kn, Vn, dOn = (x.double().numpy().reshape((-1,) + tuple(x.shape[-2:])) for x in (Q, K, V, dO))
    L, S, D = Qn.shape
    O, lse = oracle.attention(Q.reshape(L, S, D), K.reshape(L, S, D), V.reshape(L, S, D), rp, ci, block, scale,
                              return_lse=True, nthreads=8)
    M = _allowed(rp, ci, S, block)
    acc = 2.0 ** -24
    bq, bk, bv = (np.zeros((L, S, D)) for _ in range(3))
    for l in range(L):
        aQ, aK, aV, adO = np.abs(Qn[l]), np.abs(Kn[l]), np.abs(Vn[l]), np.abs(dOn[l])
        for q0 in range(0, S, rows):
            sl = slice(q0, min(S, q0 + rows))
            m = M[sl]
            fin = np.isfinite(lse[l, sl])[:, None]
            z = np.where(m & fin, scale * (Qn[l, sl] @ Kn[l].T) - np.where(fin, lse[l, sl, None], 0.0), -np.inf)
            P = np.exp(z)
            dP = dOn[l, sl] @ Vn[l].T
            delta = (dOn[l, sl] * O[l, sl]).sum(1)
            dS = P * (dP - delta[:, None])
            eP = P * (2 * r + scale * D * acc * (aQ[sl] @ aK.T)) + eta * m
            eDelta = (adO[sl] * (r * np.abs(O[l, sl]) + 2 * r * (P @ aV))).sum(1)
            edP = D * acc * (adO[sl] @ aV.T)
            edS = eP * np.abs(dP - delta[:, None]) + P * (eDelta[:, None] + edP) + r * np.abs(dS) + eta * m
            n = S * acc
            bq[l, sl] = scale * ((edS + n * np.abs(dS)) @ aK)
            bk[l] += scale * ((edS + n * np.abs(dS)).T @ aQ[sl])
            bv[l] += (eP + n * P).T @ adO[sl]
    return bq, bk, bv


def _close(got, ref, r, what, bound, eta):
    """Element by element within the smaller of two bounds: 1.5x the derived bound plus the
    output's own rounding, and 3r of the tensor's largest magnitude."""
    got = got.detach().cpu().double().numpy().reshape(ref.shape)
    err = np.abs(got - ref)
    lim = np.minimum(1.5 * (bound.reshape(ref.shape) + r * np.abs(ref) + eta), 3 * r * np.abs(ref).max()) + 1e-30
    worst = np.unravel_index(np.argmax(err / lim), err.shape)
    assert (err <= lim).all(), (f"{what}: {int((err > lim).sum())} elements over the bound; worst err "
                                f"{err[worst]:.3g} vs bound {lim[worst]:.3g} (ref {ref[worst]:.3g})")
    assert np.sqrt((err ** 2).mean()) <= 2 * r * np.sqrt((ref ** 2).mean()) + 1e-30, f"{what}: rms"


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
    bounds = _bounds(Q, K, V, dO, rp, ci, scale, U[dtype], ETA[dtype])
    for name, got, ref, b in zip(("dQ", "dK", "dV"), (dq, dk, dv), (rq, rk, rv), bounds):
        _close(got, ref, U[dtype], f"{kind} {name}", b, ETA[dtype])


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
    bounds = _bounds(Q, K, V, dO, rp, ci, 0.125, U[torch.bfloat16], ETA[torch.bfloat16])
    for name, got, ref, b in zip(("dQ", "dK", "dV"), (dq, dk, dv), (rq, rk, rv), bounds):
        assert got.shape == (B, H, S, D)
        _close(got, ref, U[torch.bfloat16], name, b, ETA[torch.bfloat16])


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
    bounds = _bounds(Q, K, V, dO, rp, ci, 0.125, U[torch.float16], ETA[torch.float16])
    for name, got, ref, b in zip(("dQ", "dK", "dV"), (q.grad, k.grad, v.grad), (rq, rk, rv), bounds):
        _close(got, ref, U[torch.float16], name, b, ETA[torch.float16])


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
            bounds = _bounds(sl(q), sl(k), sl(v), sl(dO), rph, cih, w.scale, u, ETA[q.dtype])
            for nm, got, ref, b in zip(("dQ", "dK", "dV"), (sl(dq), sl(dk), sl(dv)), (rq, rk, rv), bounds):
                _close(got, ref, u, f"lane {lane} {nm}", b, ETA[q.dtype])


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
