"""tsa_build_schedule_noalloc against tsa_build_schedule, through the C ABI.

The allocation-free entry point exists for callers that have no device allocator of their
own (a plugin inside an application that already reserved the device memory for its pool,
or a loop that cannot afford cudaMalloc's device-wide synchronization).  Its scratch is a
fixed 16 MiB array inside the library, shared by every call on a device.

Checked here: two calls in a row on different inputs (so a stale scratch from the first
call would show in the second) each give the same CSR and salience, bit for bit, as the
workspace entry point on the same keys -- bit-exactness is the bar every schedule test in
this suite uses -- and a workload whose scratch need exceeds the array is refused with
TSA_ERR_CAPACITY before any launch.  This file is collected last on purpose.
"""
import ctypes

import numpy as np
import pytest
import torch

import topology_scheduled_gb300 as tsa
from topology_scheduled_gb300.workloads import WORKLOADS, make_qkv

pytestmark = pytest.mark.gpu
DEV = "cuda"
SCRATCH_BYTES = 16 << 20
TSA_ERR_CAPACITY = 5


def _noalloc(k, w):
    """One call of tsa_build_schedule_noalloc; returns (row_ptr, col_idx[:nnz], salience)."""
    L = tsa.lib()
    lanes = w.lanes
    cap = tsa.tsa_schedule_max_nnz(w.S, w.block, w.sink, w.local_radius, w.topk)
    row_ptr = torch.full((w.nb + 1,), -7, dtype=torch.int32, device=DEV)
    col_idx = torch.full((cap,), -7, dtype=torch.int32, device=DEV)
    sal = torch.full((w.nb,), -1.0, dtype=torch.float64, device=DEV)
    stream = torch.cuda.current_stream().cuda_stream
    st = L.tsa_build_schedule_noalloc(k.data_ptr(), tsa.TSA_F16 if k.dtype == torch.float16 else tsa.TSA_BF16,
                                      lanes, w.S, w.D, w.block, w.sink, w.local_radius, w.topk,
                                      row_ptr.data_ptr(), col_idx.data_ptr(), cap, sal.data_ptr(), stream)
    assert st == 0, tsa.STATUS_NAMES.get(st, st)
    assert tsa.tsa_last_device_status() == 0
    rp = row_ptr.cpu().numpy()
    return rp, col_idx.cpu().numpy()[: rp[-1]], sal.cpu().numpy()


def _with_workspace(k, w):
    rp, ci, sal = tsa.tsa_build_schedule(k, w.block, w.sink, w.local_radius, w.topk, salience=True)
    assert tsa.tsa_last_device_status() == 0
    rp = rp.cpu().numpy()
    return rp, ci.cpu().numpy()[: rp[-1]], sal.cpu().numpy()


def test_noalloc_matches_workspace_entry_point_on_two_calls_in_a_row():
    first, second = WORKLOADS["b4h16s8192"], WORKLOADS["s4096"]
    for w in (first, second):
        assert 0 < tsa.tsa_build_schedule_workspace_bytes(w.lanes, w.S, w.D, w.block) <= SCRATCH_BYTES
    k1 = make_qkv(first, seed=3, device=DEV)[1]
    k2 = make_qkv(second, seed=4, device=DEV)[1]
    for k, w in ((k1, first), (k2, second)):
        got = _noalloc(k, w)
        ref = _with_workspace(k, w)
        assert np.array_equal(got[0], ref[0])
        assert np.array_equal(got[1], ref[1])
        assert np.array_equal(got[2].view(np.uint64), ref[2].view(np.uint64))


def test_noalloc_refuses_workloads_beyond_its_scratch():
    w = WORKLOADS["b2h32s32768"]
    assert tsa.tsa_build_schedule_workspace_bytes(w.lanes, w.S, w.D, w.block) > SCRATCH_BYTES
    L = tsa.lib()
    k = torch.empty((w.B, w.H, w.S, w.D), dtype=w.dtype, device=DEV)
    row_ptr = torch.empty(w.nb + 1, dtype=torch.int32, device=DEV)
    col_idx = torch.empty(8192, dtype=torch.int32, device=DEV)
    st = L.tsa_build_schedule_noalloc(k.data_ptr(), tsa.TSA_BF16, w.lanes, w.S, w.D, w.block, w.sink,
                                      w.local_radius, w.topk, row_ptr.data_ptr(), col_idx.data_ptr(),
                                      8192, None, ctypes.c_void_p(torch.cuda.current_stream().cuda_stream))
    assert st == TSA_ERR_CAPACITY
