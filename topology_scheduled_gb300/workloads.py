"""Seeded synthetic inputs for topology-scheduled sparse attention.

This module only draws random numbers; it holds none of the method's
arithmetic (no centroid, distance, salience, schedule rule or attention).  The
same tensors feed the CUDA library and the CPU oracle, so parity never depends
on the random number generator.

Shapes follow the pages' workloads ("Add topology-derived sparse attention
kernel" (triton-lang/kernels#22), Local benchmark: dim 64, block 64, seq
1024-4096, single lane) widened to the batched / headed shapes the same PR's
Summary supports ([batch, heads, seq, dim] with one CSR shared across lanes).

Recipes (one ``torch.Generator`` per call, seeded; draws in the order listed):

* ``iid``: Q, K, V ~ N(0, 1) in fp32, then cast to the dtype.
* ``clustered``: Q ~ N(0,1); ``n_means`` cluster means ~ N(0, 4 I) shared by all
  lanes; every token of a span takes its span's mean; K = mean + N(0, 1) noise
  per lane and token; V ~ N(0,1).  Spans are either fixed-length (each span's
  mean drawn uniformly from the means) or geometric-length (span k uses mean
  k mod n_means).  Span lengths and mean choices come from a CPU generator
  seeded with ``seed + 1`` so that they do not depend on the device.
* ``random_density_csr``: the diagonal plus round(p * nb(nb-1)/2) off-diagonal
  causal blocks chosen by a seeded permutation (a synthetic schedule, used to
  sweep density).
"""
from __future__ import annotations

import math
from dataclasses import dataclass, field

import numpy as np
import torch


@dataclass(frozen=True)
class Workload:
    name: str
    B: int
    H: int
    S: int
    D: int
    dtype: torch.dtype
    keys: str = "iid"                   # "iid" | "clustered_fixed" | "clustered_geometric"
    n_means: int = 0
    span: int = 0                       # fixed span length, or geometric mean length
    sink: int = 1
    local_radius: int = 1
    topk: int = 2
    block: int = 64
    densities: tuple = field(default=())

    @property
    def lanes(self) -> int:
        return self.B * self.H

    @property
    def nb(self) -> int:
        return self.S // self.block

    @property
    def scale(self) -> float:
        return 1.0 / math.sqrt(self.D)

    def describe(self) -> str:
        dt = "f16" if self.dtype == torch.float16 else "bf16"
        return (f"[B={self.B},H={self.H},S={self.S},D={self.D}] {dt} block {self.block}, "
                f"sink {self.sink}, local_radius {self.local_radius}, topk {self.topk}, "
                f"keys {self.keys}")


WORKLOADS = {
    # single lane, iid, topology (1,1,2) and dense causal CSR
    "s1024": Workload("s1024", 1, 1, 1024, 64, torch.float16),
    "s2048": Workload("s2048", 1, 1, 2048, 64, torch.float16),
    "s4096": Workload("s4096", 1, 1, 4096, 64, torch.float16),
    # 8 cluster means over contiguous 512-token spans, topology (1,2,4)
    "b4h16s8192": Workload("b4h16s8192", 4, 16, 8192, 64, torch.float16, "clustered_fixed",
                           n_means=8, span=512, sink=1, local_radius=2, topk=4),
    # 32 cluster means over geometric spans (mean 1024 tokens), topology (2,4,8)
    "b2h32s32768": Workload("b2h32s32768", 2, 32, 32768, 128, torch.bfloat16,
                            "clustered_geometric", n_means=32, span=1024, sink=2,
                            local_radius=4, topk=8),
    # density sweep, iid
    "b1h32s16384": Workload("b1h32s16384", 1, 32, 16384, 128, torch.bfloat16,
                            densities=(0.02, 0.05, 0.10, 0.25, 0.50, 1.00)),
}


def _gen(seed: int, device) -> torch.Generator:
    g = torch.Generator(device=device)
    g.manual_seed(int(seed))
    return g


def _span_means(S: int, keys: str, n_means: int, span: int, seed: int) -> torch.Tensor:
    """Mean index of every token (CPU, int64)."""
    g = _gen(seed + 1, "cpu")
    assign = torch.empty(S, dtype=torch.int64)
    if keys == "clustered_fixed":
        n_spans = (S + span - 1) // span
        choice = torch.randint(0, n_means, (n_spans,), generator=g)
        for s in range(n_spans):
            assign[s * span:(s + 1) * span] = choice[s]
    elif keys == "clustered_geometric":
        p = 1.0 / span
        pos, k = 0, 0
        while pos < S:
            u = float(torch.rand((), generator=g, dtype=torch.float64))
            length = max(1, int(math.ceil(math.log1p(-u) / math.log1p(-p))))
            assign[pos:pos + length] = k % n_means
            pos += length
            k += 1
    else:
        raise ValueError(keys)
    return assign


def make_qkv(w: Workload, seed: int = 0, device="cpu"):
    """Q, K, V shaped [B, H, S, D] in the workload's dtype, on ``device``."""
    g = _gen(seed, device)
    shape = (w.B, w.H, w.S, w.D)
    q = torch.randn(shape, generator=g, device=device, dtype=torch.float32).to(w.dtype)
    if w.keys == "iid":
        k = torch.randn(shape, generator=g, device=device, dtype=torch.float32).to(w.dtype)
    else:
        means = 2.0 * torch.randn((w.n_means, w.D), generator=g, device=device,
                                  dtype=torch.float32)
        assign = _span_means(w.S, w.keys, w.n_means, w.span, seed).to(device)
        k = torch.randn(shape, generator=g, device=device, dtype=torch.float32)
        k.add_(means[assign].view(1, 1, w.S, w.D))
        k = k.to(w.dtype)
    v = torch.randn(shape, generator=g, device=device, dtype=torch.float32).to(w.dtype)
    return q, k, v


def random_density_csr(nb: int, density: float, seed: int = 0):
    """Diagonal + round(density * nb(nb-1)/2) seeded off-diagonal causal blocks (int32 CSR)."""
    n_off = nb * (nb - 1) // 2
    keep = int(round(density * n_off))
    g = _gen(seed + 2, "cpu")
    perm = torch.randperm(n_off, generator=g)[:keep].numpy()
    # off-diagonal causal pair index e -> (i, j), j < i, enumerated row by row
    rows = np.floor((1 + np.sqrt(1 + 8 * perm.astype(np.float64))) / 2).astype(np.int64)
    # guard the float square root at row boundaries
    rows = np.where(rows * (rows - 1) // 2 > perm, rows - 1, rows)
    rows = np.where((rows + 1) * rows // 2 <= perm, rows + 1, rows)
    cols = perm - rows * (rows - 1) // 2
    mask = np.zeros((nb, nb), dtype=bool)
    mask[rows, cols] = True
    mask[np.arange(nb), np.arange(nb)] = True
    counts = mask.sum(axis=1)
    row_ptr = np.zeros(nb + 1, dtype=np.int32)
    row_ptr[1:] = np.cumsum(counts)
    col_idx = np.nonzero(mask)[1].astype(np.int32)
    return row_ptr, col_idx
