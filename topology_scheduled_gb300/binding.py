"""Python binding of libtsa (include/tsa.h): argument marshalling only.

Every step of the schedule builder and of the attention runs in the CUDA kernels of
libtsa.so; PyTorch only provides device memory and the current stream.  There is no
fallback: if the library is missing or a call fails, the functions raise.
"""
from __future__ import annotations

import ctypes
import math
import os
import threading

import torch

from . import build as _build

TSA_OK = 0
STATUS_NAMES = {
    0: "TSA_OK", 1: "TSA_ERR_INVALID_ARGUMENT", 2: "TSA_ERR_UNSUPPORTED",
    3: "TSA_ERR_NOT_DEVICE_POINTER", 4: "TSA_ERR_DEVICE_MISMATCH", 5: "TSA_ERR_CAPACITY",
    6: "TSA_ERR_CUDA", 7: "TSA_ERR_TIMEOUT", 8: "TSA_ERR_BAD_SCHEDULE", 9: "TSA_ERR_DEVICE",
}
TSA_F16, TSA_BF16 = 0, 1
TIE_RULES = {"index": 0, "content": 1}

_LOCK = threading.Lock()
_LIB = None

_P = ctypes.c_void_p
_I64 = ctypes.c_int64
_SZ = ctypes.c_size_t

# name -> (restype, argtypes), mirroring include/tsa.h
SIGNATURES = {
    "tsa_status_string": (ctypes.c_char_p, [ctypes.c_int]),
    "tsa_schedule_max_nnz": (_I64, [_I64, _I64, _I64, _I64, _I64]),
    "tsa_build_schedule_workspace_bytes": (_SZ, [_I64, _I64, _I64, _I64]),
    "tsa_build_schedule": (ctypes.c_int, [_P, ctypes.c_int, _I64, _I64, _I64, _I64, _I64, _I64, _I64,
                                          _P, _P, _I64, _P, _P, _SZ, _P]),
    "tsa_build_schedule_ex": (ctypes.c_int, [_P, ctypes.c_int, _I64, _I64, _I64, _I64, _I64, _I64, _I64,
                                             ctypes.c_int, _P, _P, _I64, _P, _P, _SZ, _P]),
    "tsa_build_schedule_noalloc": (ctypes.c_int, [_P, ctypes.c_int, _I64, _I64, _I64, _I64, _I64, _I64,
                                                  _I64, _P, _P, _I64, _P, _P]),
    "tsa_block_sums": (ctypes.c_int, [_P, ctypes.c_int, _I64, _I64, _I64, _I64, _P, _P]),
    "tsa_build_schedule_from_sums": (ctypes.c_int, [_P, _I64, _I64, _I64, _I64, _I64, _I64, _I64,
                                                    ctypes.c_int, _P, _P, _I64, _P, _P, _SZ, _P]),
    "tsa_fixed_segment_nnz": (_I64, [_I64, _I64, _I64]),
    "tsa_fixed_segment_csr": (ctypes.c_int, [_I64, _I64, _I64, _P, _P, _I64, _P]),
    "tsa_segment_csr": (ctypes.c_int, [_I64, _I64, _P, _I64, _P, _P, _I64, _P]),
    "tsa_dense_causal_csr": (ctypes.c_int, [_I64, _I64, _P, _P, _I64, _P]),
    "tsa_scheduled_attention": (ctypes.c_int, [_P, _P, _P, _P, _P, _P, ctypes.c_int, _I64, _I64,
                                               _I64, _I64, _I64, ctypes.c_float, _P]),
    "tsa_last_device_status": (ctypes.c_int, [_P]),
    "tsa_debug_set_wait_injection": (ctypes.c_int, [ctypes.c_int]),
    "tsa_scheduled_attention_fwd": (ctypes.c_int, [_P, _P, _P, _P, _P, _P, _P, ctypes.c_int, _I64, _I64,
                                                   _I64, _I64, _I64, ctypes.c_float, _P]),
    "tsa_attention_backward_workspace_bytes": (_SZ, [_I64, _I64, _I64, _I64]),
    "tsa_scheduled_attention_backward": (ctypes.c_int, [_P, _P, _P, _P, _P, _P, _P, _P, _I64, _P, _P, _P,
                                                        ctypes.c_int, _I64, _I64, _I64, _I64, _I64,
                                                        ctypes.c_float, _P, _SZ, _P]),
    "tsa_topology_attention_host": (ctypes.c_int, [_P, _P, _P, _P, ctypes.c_int, _I64, _I64, _I64, _I64,
                                                   _I64, _I64, _I64, _I64, ctypes.c_int, ctypes.c_float,
                                                   _P, _P, _P, _P, _P, _P, _I64, _P, _SZ, _I64, _P]),
}


class TsaError(RuntimeError):
    def __init__(self, status: int, where: str):
        self.status = status
        super().__init__(f"{where}: {STATUS_NAMES.get(status, status)}")


def library_path() -> str:
    return _build.LIB


def lib(build_if_missing: bool = True) -> ctypes.CDLL:
    """The loaded libtsa.so (built on first use when nvcc is available)."""
    global _LIB
    with _LOCK:
        if _LIB is None:
            path = _build.LIB
            if build_if_missing:
                path = _build.build()
            if not os.path.exists(path):
                raise RuntimeError(f"libtsa.so is not built ({path}); run "
                                   "`python -m topology_scheduled_gb300.build`")
            L = ctypes.CDLL(path)
            for name, (res, args) in SIGNATURES.items():
                fn = getattr(L, name)
                fn.restype = res
                fn.argtypes = args
            _LIB = L
    return _LIB


def _check(status: int, where: str):
    if status != TSA_OK:
        raise TsaError(status, where)


def _dtype_code(t: torch.Tensor) -> int:
    if t.dtype == torch.float16:
        return TSA_F16
    if t.dtype == torch.bfloat16:
        return TSA_BF16
    raise TypeError(f"expected float16 or bfloat16, got {t.dtype}")


def _stream(stream) -> int | None:
    if stream is None:
        stream = torch.cuda.current_stream()
    return stream.cuda_stream if hasattr(stream, "cuda_stream") else int(stream)


def _lanes_S_D(x: torch.Tensor):
    if x.dim() == 2:
        return 1, 1, x.shape[0], x.shape[1]
    if x.dim() == 3:
        return 1, x.shape[0], x.shape[1], x.shape[2]
    if x.dim() == 4:
        return x.shape[0], x.shape[1], x.shape[2], x.shape[3]
    raise ValueError(f"expected [S, D], [L, S, D] or [B, H, S, D], got shape {tuple(x.shape)}")


def tsa_schedule_max_nnz(S: int, block: int, sink: int, local_radius: int, topk: int) -> int:
    return int(lib().tsa_schedule_max_nnz(S, block, sink, local_radius, topk))


def tsa_build_schedule_workspace_bytes(lanes: int, S: int, D: int, block: int) -> int:
    return int(lib().tsa_build_schedule_workspace_bytes(lanes, S, D, block))


def tsa_build_schedule(K: torch.Tensor, block: int = 64, sink: int = 1, local_radius: int = 1,
                       topk: int = 2, *, salience: bool = False, tie_break: str = "index",
                       workspace: torch.Tensor | None = None, row_ptr: torch.Tensor | None = None,
                       col_idx: torch.Tensor | None = None, stream=None):
    """Topology CSR from K ([S, D], [L, S, D] or [B, H, S, D]; lane-mean centroids).

    ``tie_break`` is "index" or "content" (the elder rule's tie rule).  Returns (row_ptr,
    col_idx) int32 device tensors -- col_idx has capacity length, its first row_ptr[-1] entries
    are the schedule -- plus the per-block squared merge distance (float64) when ``salience``
    is true.
    """
    if not K.is_cuda or not K.is_contiguous():
        raise ValueError("K must be a contiguous CUDA tensor")
    if tie_break not in TIE_RULES:
        raise ValueError(f"tie_break must be one of {sorted(TIE_RULES)}")
    B, H, S, D = _lanes_S_D(K)
    lanes = B * H
    L = lib()
    nb = -(-S // block) if block > 0 else 0  # a partial last block counts
    cap = int(L.tsa_schedule_max_nnz(S, block, sink, local_radius, topk))
    if cap < 0:
        raise TsaError(1, "tsa_schedule_max_nnz")
    ws_bytes = int(L.tsa_build_schedule_workspace_bytes(lanes, S, D, block))
    if ws_bytes == 0:
        raise TsaError(2, "tsa_build_schedule_workspace_bytes")
    dev = K.device
    if workspace is None:
        workspace = torch.empty(ws_bytes, dtype=torch.uint8, device=dev)
    if row_ptr is None:
        row_ptr = torch.empty(nb + 1, dtype=torch.int32, device=dev)
    if col_idx is None:
        col_idx = torch.empty(max(cap, 1), dtype=torch.int32, device=dev)
    sal = torch.empty(nb, dtype=torch.float64, device=dev) if salience else None
    _check(L.tsa_build_schedule_ex(K.data_ptr(), _dtype_code(K), lanes, S, D, block, sink,
                                   local_radius, topk, TIE_RULES[tie_break], row_ptr.data_ptr(),
                                   col_idx.data_ptr(), col_idx.numel(),
                                   sal.data_ptr() if sal is not None else None,
                                   workspace.data_ptr(), workspace.numel(), _stream(stream)),
           "tsa_build_schedule_ex")
    return (row_ptr, col_idx, sal) if salience else (row_ptr, col_idx)


def tsa_block_sums(K: torch.Tensor, block: int = 64, *, out: torch.Tensor | None = None, stream=None):
    """Per-lane block sums of K ([S, D], [L, S, D] or [B, H, S, D]): float64 [lanes, S/block, D]."""
    if not K.is_cuda or not K.is_contiguous():
        raise ValueError("K must be a contiguous CUDA tensor")
    B, H, S, D = _lanes_S_D(K)
    lanes = B * H
    nb = -(-S // block) if block > 0 else 0  # a partial last block counts
    if out is None:
        out = torch.empty((lanes, nb, D), dtype=torch.float64, device=K.device)
    elif out.dtype != torch.float64 or not out.is_contiguous() or out.numel() != lanes * nb * D:
        raise ValueError("out must be a contiguous float64 tensor of lanes * S/block * D elements")
    _check(lib().tsa_block_sums(K.data_ptr(), _dtype_code(K), lanes, S, D, block, out.data_ptr(),
                                _stream(stream)), "tsa_block_sums")
    return out


def tsa_build_schedule_from_sums(sums: torch.Tensor, block: int = 64, sink: int = 1, local_radius: int = 1,
                                 topk: int = 2, *, S: int | None = None, salience: bool = False,
                                 tie_break: str = "index", workspace: torch.Tensor | None = None,
                                 row_ptr: torch.Tensor | None = None, col_idx: torch.Tensor | None = None,
                                 stream=None):
    """tsa_build_schedule from the block sums of all lanes ([lanes, nb, D] float64, lanes in
    global order, e.g. gathered from the GPUs that hold them).  Same result as
    tsa_build_schedule on the full keys, bit for bit.  S is the sequence length (default
    nb * block; give it when the last block is partial).  row_ptr / col_idx, if given, receive
    the CSR (int32 CUDA tensors of nb + 1 and at least tsa_schedule_max_nnz entries)."""
    if not sums.is_cuda or not sums.is_contiguous() or sums.dtype != torch.float64 or sums.dim() != 3:
        raise ValueError("sums must be a contiguous CUDA float64 tensor [lanes, nb, D]")
    if tie_break not in TIE_RULES:
        raise ValueError(f"tie_break must be one of {sorted(TIE_RULES)}")
    lanes, nb, D = sums.shape
    if S is None:
        S = nb * block
    elif -(-S // block) != nb:
        raise ValueError("S does not give sums.shape[1] blocks")
    L = lib()
    cap = int(L.tsa_schedule_max_nnz(S, block, sink, local_radius, topk))
    if cap < 0:
        raise TsaError(1, "tsa_schedule_max_nnz")
    ws_bytes = int(L.tsa_build_schedule_workspace_bytes(lanes, S, D, block))
    if ws_bytes == 0:
        raise TsaError(2, "tsa_build_schedule_workspace_bytes")
    dev = sums.device
    if workspace is None:
        workspace = torch.empty(ws_bytes, dtype=torch.uint8, device=dev)
    if row_ptr is None:
        row_ptr = torch.empty(nb + 1, dtype=torch.int32, device=dev)
    if col_idx is None:
        col_idx = torch.empty(max(cap, 1), dtype=torch.int32, device=dev)
    for t in (row_ptr, col_idx):
        if t.dtype != torch.int32 or not t.is_contiguous() or t.device != dev:
            raise ValueError("row_ptr / col_idx must be contiguous int32 tensors on the sums' device")
    if row_ptr.numel() != nb + 1:
        raise ValueError("row_ptr must hold nb + 1 entries")
    sal = torch.empty(nb, dtype=torch.float64, device=dev) if salience else None
    _check(L.tsa_build_schedule_from_sums(sums.data_ptr(), lanes, S, D, block, sink, local_radius, topk,
                                          TIE_RULES[tie_break], row_ptr.data_ptr(), col_idx.data_ptr(),
                                          col_idx.numel(), sal.data_ptr() if sal is not None else None,
                                          workspace.data_ptr(), workspace.numel(), _stream(stream)),
           "tsa_build_schedule_from_sums")
    return (row_ptr, col_idx, sal) if salience else (row_ptr, col_idx)


def tsa_fixed_segment_nnz(S: int, block: int, segment_tokens: int) -> int:
    return int(lib().tsa_fixed_segment_nnz(S, block, segment_tokens))


def tsa_fixed_segment_csr(S: int, block: int, segment_tokens: int, device=None, stream=None):
    """CSR of fixed segments of ``segment_tokens`` tokens, as int32 device tensors."""
    nb = S // block if block > 0 else 0
    dev = torch.device(device) if device is not None else torch.device("cuda", torch.cuda.current_device())
    nnz = tsa_fixed_segment_nnz(S, block, segment_tokens)
    if nnz < 0:
        raise TsaError(1, "tsa_fixed_segment_nnz")
    row_ptr = torch.empty(nb + 1, dtype=torch.int32, device=dev)
    col_idx = torch.empty(max(nnz, 1), dtype=torch.int32, device=dev)
    _check(lib().tsa_fixed_segment_csr(S, block, segment_tokens, row_ptr.data_ptr(),
                                       col_idx.data_ptr(), col_idx.numel(), _stream(stream)),
           "tsa_fixed_segment_csr")
    return row_ptr, col_idx[:nnz]


def tsa_segment_csr(S: int, block: int, starts: torch.Tensor, *, col_cap: int | None = None,
                    stream=None):
    """CSR of the segment mask whose segments begin at the int32 device tokens ``starts``.

    col_idx has ``col_cap`` entries (default nb(nb+1)/2, always enough); the schedule is its
    first row_ptr[-1] entries.
    """
    if starts.dtype != torch.int32 or not starts.is_cuda or not starts.is_contiguous():
        raise TypeError("starts must be a contiguous int32 CUDA tensor")
    nb = S // block if block > 0 else 0
    if col_cap is None:
        col_cap = max(nb * (nb + 1) // 2, 1)
    row_ptr = torch.empty(nb + 1, dtype=torch.int32, device=starts.device)
    col_idx = torch.empty(col_cap, dtype=torch.int32, device=starts.device)
    _check(lib().tsa_segment_csr(S, block, starts.data_ptr() if starts.numel() else None,
                                 starts.numel(), row_ptr.data_ptr(), col_idx.data_ptr(), col_cap,
                                 _stream(stream)), "tsa_segment_csr")
    return row_ptr, col_idx


def tsa_dense_causal_csr(S: int, block: int = 64, device=None, stream=None):
    """Dense causal CSR (row i = blocks 0..i) as int32 device tensors."""
    nb = -(-S // block) if block > 0 else 0  # a partial last block counts
    dev = torch.device(device) if device is not None else torch.device("cuda", torch.cuda.current_device())
    row_ptr = torch.empty(nb + 1, dtype=torch.int32, device=dev)
    nnz = nb * (nb + 1) // 2
    col_idx = torch.empty(max(nnz, 1), dtype=torch.int32, device=dev)
    _check(lib().tsa_dense_causal_csr(S, block, row_ptr.data_ptr(), col_idx.data_ptr(),
                                      col_idx.numel(), _stream(stream)), "tsa_dense_causal_csr")
    return row_ptr, col_idx[:nnz] if nnz > 0 else col_idx[:0]


def _check_qkv(**tensors):
    ref = None
    for name, t in tensors.items():
        if not t.is_cuda or not t.is_contiguous():
            raise ValueError(f"{name} must be a contiguous CUDA tensor")
        if ref is not None and (t.shape != ref.shape or t.dtype != ref.dtype):
            raise ValueError(f"{', '.join(tensors)} must share shape and dtype")
        ref = t


def _check_csr(row_ptr, col_idx):
    if row_ptr.dtype != torch.int32 or col_idx.dtype != torch.int32:
        raise TypeError("row_ptr and col_idx must be int32 (the CSR schedule dtype)")


def tsa_scheduled_attention(Q: torch.Tensor, K: torch.Tensor, V: torch.Tensor,
                            row_ptr: torch.Tensor, col_idx: torch.Tensor, scale: float | None = None,
                            *, out: torch.Tensor | None = None, block: int = 64, stream=None):
    """CSR-scheduled causal attention forward; output in the input dtype and shape."""
    return tsa_scheduled_attention_fwd(Q, K, V, row_ptr, col_idx, scale, out=out, block=block,
                                       stream=stream, with_lse=False)


def tsa_scheduled_attention_fwd(Q: torch.Tensor, K: torch.Tensor, V: torch.Tensor,
                                row_ptr: torch.Tensor, col_idx: torch.Tensor, scale: float | None = None,
                                *, out: torch.Tensor | None = None, lse: torch.Tensor | None = None,
                                block: int = 64, stream=None, with_lse: bool = True):
    """Forward that also returns the per-row log-sum-exp ([B*H, S] float32) for the backward."""
    _check_qkv(Q=Q, K=K, V=V)
    _check_csr(row_ptr, col_idx)
    B, H, S, D = _lanes_S_D(Q)
    if scale is None:
        scale = 1.0 / math.sqrt(D)
    if out is None:
        out = torch.empty_like(Q)
    elif out.shape != Q.shape or out.dtype != Q.dtype or not out.is_contiguous():
        raise ValueError("out must be a contiguous tensor with Q's shape and dtype")
    if with_lse and lse is None:
        lse = torch.empty((B * H, S), dtype=torch.float32, device=Q.device)
    ci = col_idx if col_idx.numel() > 0 else torch.zeros(1, dtype=torch.int32, device=Q.device)
    _check(lib().tsa_scheduled_attention_fwd(Q.data_ptr(), K.data_ptr(), V.data_ptr(),
                                             row_ptr.data_ptr(), ci.data_ptr(), out.data_ptr(),
                                             lse.data_ptr() if with_lse else None,
                                             _dtype_code(Q), B, H, S, D, block, float(scale),
                                             _stream(stream)), "tsa_scheduled_attention_fwd")
    return (out, lse) if with_lse else out


def tsa_attention_backward_workspace_bytes(lanes: int, S: int, block: int, nnz_cap: int) -> int:
    return int(lib().tsa_attention_backward_workspace_bytes(lanes, S, block, nnz_cap))


def tsa_scheduled_attention_backward(Q, K, V, O, dO, lse, row_ptr, col_idx, scale: float | None = None,
                                     *, block: int = 64, dq=None, dk=None, dv=None, workspace=None,
                                     stream=None):
    """dQ, dK, dV of the scheduled attention for upstream gradient dO (input dtype and shape)."""
    _check_qkv(Q=Q, K=K, V=V, O=O, dO=dO)
    _check_csr(row_ptr, col_idx)
    B, H, S, D = _lanes_S_D(Q)
    if lse.dtype != torch.float32 or not lse.is_contiguous() or lse.numel() != B * H * S:
        raise ValueError("lse must be a contiguous float32 tensor of B*H*S elements")
    if scale is None:
        scale = 1.0 / math.sqrt(D)
    ci = col_idx if col_idx.numel() > 0 else torch.zeros(1, dtype=torch.int32, device=Q.device)
    nnz_cap = ci.numel()
    ws = tsa_attention_backward_workspace_bytes(B * H, S, block, nnz_cap)
    if ws == 0:
        raise TsaError(2, "tsa_attention_backward_workspace_bytes")
    if workspace is None:
        workspace = torch.empty(ws, dtype=torch.uint8, device=Q.device)
    dq = torch.empty_like(Q) if dq is None else dq
    dk = torch.empty_like(K) if dk is None else dk
    dv = torch.empty_like(V) if dv is None else dv
    _check(lib().tsa_scheduled_attention_backward(
        Q.data_ptr(), K.data_ptr(), V.data_ptr(), O.data_ptr(), dO.data_ptr(), lse.data_ptr(),
        row_ptr.data_ptr(), ci.data_ptr(), nnz_cap, dq.data_ptr(), dk.data_ptr(), dv.data_ptr(),
        _dtype_code(Q), B, H, S, D, block, float(scale), workspace.data_ptr(), workspace.numel(),
        _stream(stream)), "tsa_scheduled_attention_backward")
    return dq, dk, dv


def tsa_last_device_status(stream=None) -> int:
    """Synchronizes the stream; returns and clears the device status word (0 = TSA_OK)."""
    return int(lib().tsa_last_device_status(_stream(stream)))


def tsa_debug_set_wait_injection(on: bool) -> None:
    """Test hook for the failure path: while on, each scheduled-attention launch has its first
    CTA withhold its first scores, so a bounded wait runs out and the device status reports
    TSA_ERR_TIMEOUT (see include/tsa.h)."""
    _check(lib().tsa_debug_set_wait_injection(1 if on else 0), "tsa_debug_set_wait_injection")


def tsa_topology_attention_host(hQ: torch.Tensor, hK: torch.Tensor, hV: torch.Tensor, block: int = 64,
                                sink: int = 1, local_radius: int = 1, topk: int = 2, scale: float | None = None,
                                *, tie_break: str = "index", out: torch.Tensor | None = None,
                                device_buffers=None, row_ptr: torch.Tensor | None = None,
                                col_idx: torch.Tensor | None = None, workspace: torch.Tensor | None = None,
                                lane_chunk: int = 0, device=None, stream=None):
    """One forward step from host tensors ([S, D], [L, S, D] or [B, H, S, D]; page-locked for
    the copies to overlap): the topology CSR from K and the scheduled attention, O returned in
    host memory (``out``, page-locked if not given).  ``device_buffers`` = (dQ, dK, dV, dO) on
    the device; allocated when not given.  Returns (out, row_ptr, col_idx); the call is
    asynchronous on ``stream`` like the others."""
    for name, t in (("hQ", hQ), ("hK", hK), ("hV", hV)):
        if t.is_cuda or not t.is_contiguous():
            raise ValueError(f"{name} must be a contiguous host tensor")
    if not (hQ.shape == hK.shape == hV.shape and hQ.dtype == hK.dtype == hV.dtype):
        raise ValueError("hQ, hK, hV must share shape and dtype")
    if tie_break not in TIE_RULES:
        raise ValueError(f"tie_break must be one of {sorted(TIE_RULES)}")
    B, H, S, D = _lanes_S_D(hQ)
    lanes = B * H
    if scale is None:
        scale = 1.0 / math.sqrt(D)
    dev = torch.device("cuda", torch.cuda.current_device()) if device is None else torch.device(device)
    L = lib()
    nb = -(-S // block) if block > 0 else 0
    cap = int(L.tsa_schedule_max_nnz(S, block, sink, local_radius, topk))
    if cap < 0:
        raise TsaError(1, "tsa_schedule_max_nnz")
    ws_bytes = int(L.tsa_build_schedule_workspace_bytes(lanes, S, D, block))
    if ws_bytes == 0:
        raise TsaError(2, "tsa_build_schedule_workspace_bytes")
    if workspace is None:
        workspace = torch.empty(ws_bytes, dtype=torch.uint8, device=dev)
    if row_ptr is None:
        row_ptr = torch.empty(nb + 1, dtype=torch.int32, device=dev)
    if col_idx is None:
        col_idx = torch.empty(max(cap, 1), dtype=torch.int32, device=dev)
    if device_buffers is None:
        device_buffers = tuple(torch.empty(hQ.shape, dtype=hQ.dtype, device=dev) for _ in range(4))
    if out is None:
        out = torch.empty(hQ.shape, dtype=hQ.dtype, pin_memory=True)
    dq, dk, dv, do = device_buffers
    _check(L.tsa_topology_attention_host(hQ.data_ptr(), hK.data_ptr(), hV.data_ptr(), out.data_ptr(),
                                         _dtype_code(hQ), B, H, S, D, block, sink, local_radius, topk,
                                         TIE_RULES[tie_break], float(scale), dq.data_ptr(), dk.data_ptr(),
                                         dv.data_ptr(), do.data_ptr(), row_ptr.data_ptr(), col_idx.data_ptr(),
                                         col_idx.numel(), workspace.data_ptr(), workspace.numel(), int(lane_chunk),
                                         _stream(stream)), "tsa_topology_attention_host")
    return out, row_ptr, col_idx
