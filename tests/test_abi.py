"""The C ABI library builds, loads and exports every entry point declared in include/tsa.h;
host-side argument checks that need no GPU return the documented status codes."""
import ctypes
import os
import re

import pytest

import topology_scheduled_gb300 as tsa
from topology_scheduled_gb300.binding import SIGNATURES

ROOT = os.path.dirname(os.path.dirname(os.path.abspath(__file__)))


def _declared():
    text = open(os.path.join(ROOT, "include", "tsa.h")).read()
    text = re.sub(r"/\*.*?\*/", "", text, flags=re.S)
    return sorted(set(re.findall(r"\b(tsa_[a-z_0-9]+)\s*\(", text)))


def test_every_declared_symbol_is_exported_and_bound():
    L = tsa.lib()
    names = _declared()
    assert len(names) == 19
    for n in names:
        assert hasattr(L, n), n
        assert n in SIGNATURES, n


def test_status_strings():
    L = tsa.lib()
    for code, name in tsa.STATUS_NAMES.items():
        assert L.tsa_status_string(code).decode() == name


def test_max_nnz_closed_form():
    # sum_i min(i+1, sink+r+1+topk): 70 at 16 blocks for (1,1,2), 150 at 32, 310 at 64
    assert tsa.tsa_schedule_max_nnz(1024, 64, 1, 1, 2) == 70
    assert tsa.tsa_schedule_max_nnz(2048, 64, 1, 1, 2) == 150
    assert tsa.tsa_schedule_max_nnz(4096, 64, 1, 1, 2) == 310
    assert tsa.tsa_schedule_max_nnz(8192, 64, 1, 2, 4) == 996
    assert tsa.tsa_schedule_max_nnz(32768, 64, 2, 4, 8) == 7575
    assert tsa.tsa_schedule_max_nnz(1024, 64, 0, 100, 0) == 136
    assert tsa.tsa_schedule_max_nnz(1000, 64, 1, 1, 2) == 70  # a partial last block counts: 16 blocks
    assert tsa.tsa_schedule_max_nnz(1024, 64, -1, 1, 2) == -1


def test_workspace_bytes():
    assert tsa.tsa_build_schedule_workspace_bytes(64, 32768, 128, 64) >= 64 * 512 * 128 * 8 + 512 * 512 * 8
    assert tsa.tsa_build_schedule_workspace_bytes(1, 64 * 4097, 64, 64) == 0  # beyond 4096 blocks
    assert tsa.tsa_build_schedule_workspace_bytes(1, 100, 64, 64) > 0  # 2 blocks, the last partial
    assert tsa.tsa_build_schedule_workspace_bytes(1, 100, 64, 0) == 0


def test_host_checks_before_any_device_call():
    L = tsa.lib()
    fake = ctypes.c_void_p(4096)
    # null pointers
    assert L.tsa_scheduled_attention(None, fake, fake, fake, fake, fake, 0, 1, 1, 64, 64, 64, 0.1, None) == 1
    assert L.tsa_build_schedule(None, 0, 1, 64, 64, 64, 1, 1, 2, fake, fake, 10, None, fake, 1 << 20, None) == 1
    assert L.tsa_dense_causal_csr(64, 64, None, fake, 1, None) == 1
    assert L.tsa_build_schedule_ex(fake, 0, 1, 64, 64, 64, 1, 1, 2, 7, fake, fake, 10, None, fake,
                                   1 << 20, None) == 1  # unknown tie rule
    assert L.tsa_fixed_segment_csr(4096, 64, 512, None, fake, 288, None) == 1
    assert L.tsa_fixed_segment_csr(4096, 64, 512, fake, fake, 287, None) == 5  # capacity
    assert L.tsa_fixed_segment_csr(4096, 64, 0, fake, fake, 288, None) == 1
    assert L.tsa_segment_csr(4096, 64, None, 3, fake, fake, 10, None) == 1  # starts missing
    assert L.tsa_segment_csr(4000, 64, None, 0, fake, fake, 10, None) == 1
    # unsupported block or head dimension
    assert L.tsa_scheduled_attention(fake, fake, fake, fake, fake, fake, 0, 1, 1, 64, 64, 16, 0.1, None) == 2
    assert L.tsa_scheduled_attention(fake, fake, fake, fake, fake, fake, 0, 1, 1, 64, 96, 64, 0.1, None) == 2
    # empty sequence, bad dtype, non-finite scale, misaligned pointer
    assert L.tsa_scheduled_attention(fake, fake, fake, fake, fake, fake, 0, 1, 1, 0, 64, 64, 0.1, None) == 1
    assert L.tsa_scheduled_attention(fake, fake, fake, fake, fake, fake, 5, 1, 1, 64, 64, 64, 0.1, None) == 1
    assert L.tsa_scheduled_attention(fake, fake, fake, fake, fake, fake, 0, 1, 1, 64, 64, 64,
                                     float("nan"), None) == 1
    odd = ctypes.c_void_p(4098)
    assert L.tsa_scheduled_attention(odd, fake, fake, fake, fake, fake, 0, 1, 1, 64, 64, 64, 0.1, None) == 1
    # output aliasing an input
    assert L.tsa_scheduled_attention(fake, fake, fake, fake, fake, fake, 0, 1, 1, 64, 64, 64, 0.1, None) == 1
    # capacity checks
    assert L.tsa_dense_causal_csr(1024, 64, fake, fake, 135, None) == 5
    assert L.tsa_build_schedule(fake, 0, 1, 1024, 64, 64, 1, 1, 2, fake, fake, 69, None, fake, 1 << 30,
                                None) == 5
    assert L.tsa_build_schedule(fake, 0, 1, 1024, 64, 64, 1, 1, 2, fake, fake, 70, None, fake, 16,
                                None) == 5
    # builder limits
    assert L.tsa_build_schedule(fake, 0, 1, 64 * 4097, 64, 64, 1, 1, 2, fake, fake, 1 << 30, None, fake,
                                1 << 40, None) == 2


def test_noalloc_host_checks_before_any_device_call():
    """The allocation-free builder refuses bad or oversized arguments on the host, before it
    looks up its device array: the callee's own size checks come first (so a size that wrapped
    around can never pass the capacity test), then the scratch capacity."""
    L = tsa.lib()
    fake = ctypes.c_void_p(4096)

    def call(K, lanes, S, D, block, row_ptr=fake, col_idx=fake):
        return L.tsa_build_schedule_noalloc(K, 0, lanes, S, D, block, 1, 1, 2, row_ptr, col_idx, 1 << 20,
                                            None, None)

    assert call(None, 1, 1024, 64, 64) == 1                    # null keys
    assert call(fake, 1, 1024, 64, 64, row_ptr=None) == 1     # null row_ptr
    assert call(fake, 1, 1024, 64, 64, col_idx=None) == 1     # null col_idx
    assert call(fake, 0, 1024, 64, 64) == 1                    # no lanes
    assert call(fake, 1, 0, 64, 64) == 1                       # empty sequence
    assert call(fake, 1, 1024, 0, 64) == 1                     # empty head dimension
    assert call(fake, 1, 1024, 64, 0) == 1                     # zero block
    assert call(fake, 1, 64 * 4097, 64, 64) == 2               # beyond 4096 blocks
    assert call(fake, 1, 1024, 4096, 64) == 2                  # head dimension beyond the builder's
    # lanes * S * D past int64: refused as invalid, never wrapped into a small scratch need
    assert call(fake, 1 << 50, 1 << 10, 1 << 10, 64) == 1
    assert tsa.tsa_build_schedule_workspace_bytes(1 << 50, 1 << 10, 1 << 10, 64) == 0
    # a valid workload larger than the 16 MiB array
    assert tsa.tsa_build_schedule_workspace_bytes(64, 32768, 128, 64) > 16 << 20
    assert call(fake, 64, 32768, 128, 64) == 5


def test_fixed_segment_nnz_closed_form():
    # the mirror page's counts at S 4096, block 64: 288 (512-token), 160 (256-token), 2080 dense
    assert tsa.tsa_fixed_segment_nnz(4096, 64, 512) == 288
    assert tsa.tsa_fixed_segment_nnz(4096, 64, 256) == 160
    assert tsa.tsa_fixed_segment_nnz(4096, 64, 4096) == 2080
    assert tsa.tsa_fixed_segment_nnz(4096, 64, 64) == 64
    assert tsa.tsa_fixed_segment_nnz(4096, 64, 1) == 64
    assert tsa.tsa_fixed_segment_nnz(4000, 64, 512) == -1
    assert tsa.tsa_fixed_segment_nnz(4096, 64, 0) == -1


def test_host_step_argument_errors_need_no_gpu():
    """tsa_topology_attention_host rejects bad arguments before touching the device."""
    L = tsa.lib()
    f = 4096  # any non-null, 256-byte aligned address: never dereferenced on these paths
    m = 1 << 20  # distinct device buffers (128 KB each here), so that they do not overlap
    args = [f, f, f, f, 1, 1, 1, 1024, 64, 64, 1, 1, 2, 0, 0.125, f, f + m, f + 2 * m, f + 3 * m, f, f, 1000, f,
            1 << 30, 0, None]
    a = list(args); a[0] = None
    assert L.tsa_topology_attention_host(*a) == 1          # null host pointer
    a = list(args); a[4] = 7
    assert L.tsa_topology_attention_host(*a) == 1          # unknown dtype
    a = list(args); a[13] = 9
    assert L.tsa_topology_attention_host(*a) == 1          # unknown tie rule
    a = list(args); a[9] = 16
    assert L.tsa_topology_attention_host(*a) == 2          # block 16
    a = list(args); a[8] = 96
    assert L.tsa_topology_attention_host(*a) == 2          # head dim 96
    a = list(args); a[24] = -1
    assert L.tsa_topology_attention_host(*a) == 1          # negative lane chunk
    a = list(args); a[16] = f + 8
    assert L.tsa_topology_attention_host(*a) == 1          # misaligned device buffer
    a = list(args); a[17] = f + (64 << 10)  # inside dQ
    assert L.tsa_topology_attention_host(*a) == 1          # overlapping device buffers
    a = list(args); a[21] = 5
    assert L.tsa_topology_attention_host(*a) == 5          # CSR capacity below the bound (70)
