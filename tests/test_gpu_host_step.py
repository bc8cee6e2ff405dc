"""tsa_topology_attention_host: one forward step from host memory with the copies overlapped.
Its O and CSR must equal, bit for bit, those of the device-resident calls it chains
(tsa_build_schedule_ex and tsa_scheduled_attention on the same inputs), for every lane-chunk
size (one lane per chunk, uneven chunks, the default, one chunk), both dtypes and head dims, a
partial last block, page-locked and pageable host memory; a device pointer given as host memory
is refused.  One case per dtype is also compared directly with the oracle (fp64 CPU): the CSR
bit for bit, O on every row within the attention tolerance."""
import numpy as np
import pytest
import torch

import oracle
import topology_scheduled_gb300 as tsa
from _tol import assert_close

pytestmark = pytest.mark.gpu
DEV = "cuda"


def _inputs(L, S, D, dtype, seed, pinned=True):
    g = torch.Generator().manual_seed(seed)
    xs = [torch.randn((L, S, D), generator=g).to(dtype) for _ in range(3)]
    return [x.pin_memory() for x in xs] if pinned else xs


def _device_path(hq, hk, hv, block, sink, r, topk, tie):
    q, k, v = (x.to(DEV) for x in (hq, hk, hv))
    rp, ci = tsa.tsa_build_schedule(k, block, sink, r, topk, tie_break=tie)
    out = tsa.tsa_scheduled_attention(q, k, v, rp, ci, q.shape[-1] ** -0.5, block=block)
    return out.cpu(), rp.cpu(), ci.cpu()


@pytest.mark.parametrize("L,S,D,dtype,block,chunk", [(1, 1024, 64, torch.float16, 64, 0),
                                                     (8, 2048, 128, torch.bfloat16, 64, 1),
                                                     (7, 1000, 64, torch.bfloat16, 64, 3),
                                                     (6, 4096, 128, torch.float16, 128, 0),
                                                     (5, 2048, 64, torch.float16, 32, 99)])
@pytest.mark.parametrize("tie", ["index", "content"])
def test_equals_device_path(L, S, D, dtype, block, chunk, tie):
    hq, hk, hv = _inputs(L, S, D, dtype, S + L)
    out, rp, ci = tsa.tsa_topology_attention_host(hq, hk, hv, block, 1, 2, 3, tie_break=tie, lane_chunk=chunk)
    torch.cuda.synchronize()
    assert tsa.tsa_last_device_status() == 0
    ref, rrp, rci = _device_path(hq, hk, hv, block, 1, 2, 3, tie)
    assert torch.equal(rp.cpu(), rrp)
    n = int(rrp[-1])
    assert torch.equal(ci.cpu()[:n], rci[:n])
    assert torch.equal(out.view(torch.int16), ref.view(torch.int16))


def test_pageable_host_memory():
    hq, hk, hv = _inputs(3, 1536, 64, torch.bfloat16, 11, pinned=False)
    out = torch.empty_like(hq)  # pageable output too
    tsa.tsa_topology_attention_host(hq, hk, hv, 64, 2, 1, 2, out=out, lane_chunk=2)
    torch.cuda.synchronize()
    ref, _, _ = _device_path(hq, hk, hv, 64, 2, 1, 2, "index")
    assert torch.equal(out.view(torch.int16), ref.view(torch.int16))


def test_device_pointer_as_host_is_refused():
    hq, hk, hv = _inputs(1, 256, 64, torch.float16, 3)
    bad = hk.to(DEV)
    L = tsa.lib()
    bufs = [torch.empty(hq.shape, dtype=hq.dtype, device=DEV) for _ in range(4)]
    rp = torch.empty(5, dtype=torch.int32, device=DEV)
    ci = torch.empty(64, dtype=torch.int32, device=DEV)
    ws = torch.empty(tsa.tsa_build_schedule_workspace_bytes(1, 256, 64, 64), dtype=torch.uint8, device=DEV)
    out = torch.empty(hq.shape, dtype=hq.dtype, pin_memory=True)
    st = L.tsa_topology_attention_host(hq.data_ptr(), bad.data_ptr(), hv.data_ptr(), out.data_ptr(), 0, 1, 1,
                                       256, 64, 64, 1, 1, 2, 0, 0.125, *[b.data_ptr() for b in bufs],
                                       rp.data_ptr(), ci.data_ptr(), ci.numel(), ws.data_ptr(), ws.numel(), 0, None)
    assert st == 1


@pytest.mark.parametrize("L,S,D,dtype,block,tie", [(6, 2048, 128, torch.bfloat16, 64, "index"),
                                                    (5, 1000, 64, torch.float16, 64, "content")])
def test_equals_oracle(L, S, D, dtype, block, tie):
    hq, hk, hv = _inputs(L, S, D, dtype, 7 * S + L)
    hk = (hk.float() * 2.5).to(dtype)  # wider spread of the key-block centroids
    out, rp, ci = tsa.tsa_topology_attention_host(hq, hk, hv, block, 2, 2, 3, tie_break=tie, lane_chunk=2)
    torch.cuda.synchronize()
    assert tsa.tsa_last_device_status() == 0
    orp, oci, _ = oracle.build_schedule(hk, block, 2, 2, 3, tie=tie)
    rp = rp.cpu().numpy()
    assert np.array_equal(rp, orp) and np.array_equal(ci.cpu().numpy()[: rp[-1]], oci)
    ref = oracle.attention(hq, hk, hv, orp, oci, block, D ** -0.5, nthreads=8)
    assert_close(out.double().numpy(), ref, dtype)
