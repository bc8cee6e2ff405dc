"""Python access to the CPU oracle (oracle/tsa_oracle.c).

TEST INFRASTRUCTURE, NOT PRODUCT CODE.  Only the tests, ``__graft_entry__.smoke()``
and ``bench.py``'s CPU-baseline / reference leg may import this module.  The
oracle shares nothing with the CUDA library in ``topology_scheduled_gb300``;
this file only compiles the C source with gcc and marshals numpy / torch CPU
arrays into it.  Every function names the passage it follows in the C source.

Parity pins: every function below is pinned by a ``-m "not gpu"`` test in
tests/test_oracle_*.py (closed forms, printed counts, invariants, brute force
and library routines).
"""
from __future__ import annotations

import ctypes
import hashlib
import os
import subprocess
import threading

import numpy as np

_HERE = os.path.dirname(os.path.abspath(__file__))
_SRC = os.path.join(_HERE, "tsa_oracle.c")
_BUILD = os.path.join(_HERE, "_build")
_LOCK = threading.Lock()
_LIB = None

F16 = 0
BF16 = 1

_I64 = ctypes.c_int64
_PTR = ctypes.c_void_p


def _lib_path() -> str:
    with open(_SRC, "rb") as f:
        digest = hashlib.sha1(f.read()).hexdigest()[:12]
    return os.path.join(_BUILD, f"libtsa_oracle_{digest}.so")


def build() -> str:
    """Compile the oracle with gcc (no fused multiply-add unless written out)."""
    path = _lib_path()
    if not os.path.exists(path):
        os.makedirs(_BUILD, exist_ok=True)
        tmp = f"{path}.{os.getpid()}.tmp"
        subprocess.run(
            ["gcc", "-O2", "-std=c11", "-ffp-contract=off", "-fno-fast-math", "-fPIC",
             "-shared", "-pthread", _SRC, "-o", tmp, "-lm"],
            check=True,
        )
        os.replace(tmp, path)
    return path


def lib():
    global _LIB
    with _LOCK:
        if _LIB is None:
            L = ctypes.CDLL(build())
            for name in ("oracle_decode", "oracle_dense_causal_csr", "oracle_centroids",
                         "oracle_pairwise_d2", "oracle_salience", "oracle_salience_content",
                         "oracle_topology_csr", "oracle_build_schedule",
                         "oracle_build_schedule_tie", "oracle_segment_csr",
                         "oracle_fixed_segment_csr", "oracle_attention",
                         "oracle_attention_lse", "oracle_attention_backward"):
                getattr(L, name).restype = ctypes.c_int
            _LIB = L
    return _LIB


def _p(a: np.ndarray):
    return a.ctypes.data_as(_PTR)


def _bits(x, dtype: int | None = None):
    """16-bit payload of a torch f16/bf16 tensor (or a uint16 numpy array)."""
    try:
        import torch
    except ImportError:  # pragma: no cover
        torch = None
    if torch is not None and isinstance(x, torch.Tensor):
        if x.dtype == torch.float16:
            dt = F16
        elif x.dtype == torch.bfloat16:
            dt = BF16
        else:
            raise TypeError(f"oracle takes float16/bfloat16 tensors, got {x.dtype}")
        arr = x.detach().cpu().contiguous().view(torch.int16).numpy().view(np.uint16)
        return np.ascontiguousarray(arr), dt
    arr = np.ascontiguousarray(x, dtype=np.uint16)
    if dtype is None:
        raise TypeError("dtype is required for raw uint16 input")
    return arr, dtype


def _check(rc: int, what: str):
    if rc != 0:
        raise ValueError(f"{what} failed with code {rc}")


def decode(x, dtype: int | None = None) -> np.ndarray:
    """Exact binary64 value of each 16-bit element."""
    bits, dt = _bits(x, dtype)
    out = np.empty(bits.shape, dtype=np.float64)
    _check(lib().oracle_decode(_p(bits), _I64(bits.size), ctypes.c_int(dt), _p(out)), "decode")
    return out


def dense_causal_csr(nb: int):
    row_ptr = np.empty(nb + 1, dtype=np.int32)
    col_idx = np.empty(max(nb * (nb + 1) // 2, 1), dtype=np.int32)
    _check(lib().oracle_dense_causal_csr(_I64(nb), _p(row_ptr), _p(col_idx)), "dense_causal_csr")
    return row_ptr, col_idx[: nb * (nb + 1) // 2]


def centroids(K, block: int, dtype: int | None = None) -> np.ndarray:
    """Lane-mean key-block centroids, K shaped [L, S, D] (or [S, D]); ceil(S / block) blocks,
    a partial last block averaging the tokens it holds."""
    bits, dt = _bits(K, dtype)
    if bits.ndim == 2:
        bits = bits[None]
    bits = bits.reshape(-1, bits.shape[-2], bits.shape[-1])
    L, S, D = bits.shape
    C = np.empty((-(-S // block), D), dtype=np.float64)
    _check(lib().oracle_centroids(_p(bits), ctypes.c_int(dt), _I64(L), _I64(S), _I64(D),
                                  _I64(block), _p(C)), "centroids")
    return C


def pairwise_d2(C: np.ndarray) -> np.ndarray:
    C = np.ascontiguousarray(C, dtype=np.float64)
    nb, D = C.shape
    out = np.empty((nb, nb), dtype=np.float64)
    _check(lib().oracle_pairwise_d2(_p(C), _I64(nb), _I64(D), _p(out)), "pairwise_d2")
    return out


def salience(C: np.ndarray, tie: str = "index"):
    """Elder-rule squared merge distance per block, plus the MST edges in Kruskal order.

    ``tie`` is "index" (ties broken by block index) or "content" (by centroid content).
    """
    fn = {"index": "oracle_salience", "content": "oracle_salience_content"}[tie]
    C = np.ascontiguousarray(C, dtype=np.float64)
    nb, D = C.shape
    sal = np.empty(nb, dtype=np.float64)
    mu = np.empty(max(nb - 1, 1), dtype=np.int32)
    mv = np.empty(max(nb - 1, 1), dtype=np.int32)
    md = np.empty(max(nb - 1, 1), dtype=np.float64)
    _check(getattr(lib(), fn)(_p(C), _I64(nb), _I64(D), _p(sal), _p(mu), _p(mv), _p(md)),
           "salience")
    n = nb - 1
    return sal, (mu[:n], mv[:n], md[:n])


def max_nnz(nb: int, sink: int, local_radius: int, topk: int) -> int:
    """Upper bound on the topology CSR's nnz: sum_i min(i+1, sink + local_radius + 1 + topk)."""
    per = sink + local_radius + 1 + topk
    return int(sum(min(i + 1, per) for i in range(nb)))


def topology_csr(sal_sq: np.ndarray, sink: int, local_radius: int, topk: int):
    sal_sq = np.ascontiguousarray(sal_sq, dtype=np.float64)
    nb = sal_sq.shape[0]
    cap = max(max_nnz(nb, sink, local_radius, topk), 1)
    row_ptr = np.empty(nb + 1, dtype=np.int32)
    col_idx = np.empty(cap, dtype=np.int32)
    _check(lib().oracle_topology_csr(_p(sal_sq), _I64(nb), _I64(sink), _I64(local_radius),
                                     _I64(topk), _p(row_ptr), _p(col_idx), _I64(cap)),
           "topology_csr")
    return row_ptr, col_idx[: row_ptr[-1]].copy()


def build_schedule(K, block: int, sink: int, local_radius: int, topk: int,
                   dtype: int | None = None, tie: str = "index"):
    """Centroids -> elder-rule salience -> topology CSR. Returns (row_ptr, col_idx, sal_sq)."""
    content = {"index": 0, "content": 1}[tie]
    bits, dt = _bits(K, dtype)
    if bits.ndim == 2:
        bits = bits[None]
    bits = bits.reshape(-1, bits.shape[-2], bits.shape[-1])
    L, S, D = bits.shape
    nb = -(-S // block)  # a partial last block is a block too
    cap = max(max_nnz(nb, sink, local_radius, topk), 1)
    row_ptr = np.empty(nb + 1, dtype=np.int32)
    col_idx = np.empty(cap, dtype=np.int32)
    sal = np.empty(nb, dtype=np.float64)
    _check(lib().oracle_build_schedule_tie(_p(bits), ctypes.c_int(dt), _I64(L), _I64(S), _I64(D),
                                           _I64(block), _I64(sink), _I64(local_radius), _I64(topk),
                                           ctypes.c_int(content), _p(row_ptr), _p(col_idx),
                                           _I64(cap), _p(sal)),
           "build_schedule")
    return row_ptr, col_idx[: row_ptr[-1]].copy(), sal


def segment_csr(S: int, block: int, starts):
    """Block schedule of the segment mask whose segments begin at the tokens in ``starts``
    (strictly ascending in [0, S); token 0 always begins one)."""
    st = np.ascontiguousarray(np.asarray(starts, dtype=np.int64).reshape(-1))
    nb = S // block
    cap = max(nb * (nb + 1) // 2, 1)
    row_ptr = np.empty(nb + 1, dtype=np.int32)
    col_idx = np.empty(cap, dtype=np.int32)
    _check(lib().oracle_segment_csr(_I64(S), _I64(block), _p(st), _I64(st.size), _p(row_ptr),
                                    _p(col_idx), _I64(cap)), "segment_csr")
    return row_ptr, col_idx[: row_ptr[-1]].copy()


def fixed_segment_csr(S: int, block: int, seg_tokens: int):
    """Block schedule of fixed segments of ``seg_tokens`` tokens."""
    nb = S // block
    cap = max(nb * (nb + 1) // 2, 1)
    row_ptr = np.empty(nb + 1, dtype=np.int32)
    col_idx = np.empty(cap, dtype=np.int32)
    _check(lib().oracle_fixed_segment_csr(_I64(S), _I64(block), _I64(seg_tokens), _p(row_ptr),
                                          _p(col_idx), _I64(cap)), "fixed_segment_csr")
    return row_ptr, col_idx[: row_ptr[-1]].copy()


def _qkv_bits(tensors, dtype):
    bits = [_bits(t, dtype) for t in tensors]
    if len({b[1] for b in bits}) != 1:
        raise TypeError("inputs must share a dtype")
    S, D = bits[0][0].shape[-2], bits[0][0].shape[-1]
    return [b[0].reshape(-1, S, D) for b in bits], bits[0][1], S, D


def _csr(row_ptr, col_idx):
    row_ptr = np.ascontiguousarray(row_ptr, dtype=np.int32)
    col_idx = np.ascontiguousarray(col_idx, dtype=np.int32)
    if col_idx.size == 0:
        col_idx = np.zeros(1, dtype=np.int32)
    return row_ptr, col_idx


def attention(Q, K, V, row_ptr, col_idx, block: int, scale: float, lanes=None, tokens=None,
              online: bool = False, nthreads: int = 1, dtype: int | None = None,
              return_lse: bool = False):
    """fp64 masked attention for chosen (lane, token) rows; all rows when lanes/tokens are None.

    Q, K, V are [L, S, D] or [S, D] (or [B, H, S, D]); returns [n, D] float64 (or the full
    [L, S, D] array when no rows are given), and with ``return_lse`` also the log-sum-exp of
    the scaled scores per row ([n] or [L, S]; -inf for a row without keys).
    """
    (qb, kb, vb), dt, S, D = _qkv_bits((Q, K, V), dtype)
    L = qb.shape[0]
    full = lanes is None
    if full:
        lanes = np.repeat(np.arange(L, dtype=np.int64), S)
        tokens = np.tile(np.arange(S, dtype=np.int64), L)
    lanes = np.ascontiguousarray(lanes, dtype=np.int64)
    tokens = np.ascontiguousarray(tokens, dtype=np.int64)
    row_ptr, col_idx = _csr(row_ptr, col_idx)
    out = np.empty((lanes.shape[0], D), dtype=np.float64)
    lse = np.empty(lanes.shape[0], dtype=np.float64) if return_lse else None
    _check(lib().oracle_attention_lse(_p(qb), _p(kb), _p(vb), ctypes.c_int(dt), _I64(L), _I64(S),
                                      _I64(D), _I64(block), ctypes.c_double(scale), _p(row_ptr),
                                      _p(col_idx), _I64(lanes.shape[0]), _p(lanes), _p(tokens),
                                      _p(out), _p(lse) if lse is not None else None,
                                      ctypes.c_int(1 if online else 0),
                                      ctypes.c_int(int(nthreads))), "attention")
    if full:
        out = out.reshape(L, S, D)
        lse = lse.reshape(L, S) if lse is not None else None
    return (out, lse) if return_lse else out


def attention_backward(Q, K, V, dO, row_ptr, col_idx, block: int, scale: float,
                       nthreads: int = 1, dtype: int | None = None):
    """fp64 gradients (dQ, dK, dV), each [L, S, D], of the masked attention for upstream dO."""
    (qb, kb, vb, ob), dt, S, D = _qkv_bits((Q, K, V, dO), dtype)
    L = qb.shape[0]
    row_ptr, col_idx = _csr(row_ptr, col_idx)
    grads = [np.empty((L, S, D), dtype=np.float64) for _ in range(3)]
    _check(lib().oracle_attention_backward(_p(qb), _p(kb), _p(vb), _p(ob), ctypes.c_int(dt),
                                           _I64(L), _I64(S), _I64(D), _I64(block),
                                           ctypes.c_double(scale), _p(row_ptr), _p(col_idx),
                                           _p(grads[0]), _p(grads[1]), _p(grads[2]),
                                           ctypes.c_int(int(nthreads))), "attention_backward")
    return tuple(grads)
