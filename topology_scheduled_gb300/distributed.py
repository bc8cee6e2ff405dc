"""Lane-sharded schedule build over a torch.distributed group (argument plumbing and the one
exchange; every computation runs in libtsa).

The topology schedule is one CSR shared by all lanes, built from the lane-mean key-block
centroids.  When the lanes are spread over ranks, each rank computes the block sums of its
own lanes (tsa_block_sums), the ranks all-gather them in global lane order, and every rank
builds the CSR from all of them (tsa_build_schedule_from_sums).  The centroid sums the lanes
in ascending order on every rank, exactly as the single-GPU build does, so every rank gets
the single-GPU CSR bit for bit.  The exchange is lanes * nb * D float64 values (33.5 MB for
64 lanes of [32768, 128] keys).  Rank r holds a contiguous run of lanes, ranks in order;
shards may differ in size.
"""
from __future__ import annotations

import torch
import torch.distributed as dist

from .binding import tsa_block_sums, tsa_build_schedule_from_sums


def gather_block_sums(local: torch.Tensor, group=None) -> torch.Tensor:
    """All-gather [lanes_r, nb, D] float64 block sums into [sum of lanes_r, nb, D], rank order."""
    world = dist.get_world_size(group)
    if world == 1:
        return local
    counts = torch.tensor([local.shape[0]], dtype=torch.int64, device=local.device)
    all_counts = [torch.empty_like(counts) for _ in range(world)]
    dist.all_gather(all_counts, counts, group=group)
    n = [int(c.item()) for c in all_counts]
    most = max(n)
    padded = local
    if local.shape[0] < most:  # all_gather moves equal-sized tensors
        padded = torch.zeros((most,) + tuple(local.shape[1:]), dtype=local.dtype, device=local.device)
        padded[: local.shape[0]] = local
    parts = [torch.empty_like(padded) for _ in range(world)]
    dist.all_gather(parts, padded.contiguous(), group=group)
    return torch.cat([p[:k] for p, k in zip(parts, n)], dim=0).contiguous()


def build_schedule_lane_sharded(K_local: torch.Tensor, block: int = 64, sink: int = 1, local_radius: int = 1,
                                topk: int = 2, *, tie_break: str = "index", group=None):
    """The topology CSR of the keys whose lanes are spread over the group's ranks (this rank:
    K_local, [lanes_r, S, D] or [B_r, H, S, D] on its GPU).  Every rank returns the same
    (row_ptr, col_idx)."""
    sums = tsa_block_sums(K_local, block)
    return tsa_build_schedule_from_sums(gather_block_sums(sums, group), block, sink, local_radius, topk,
                                        S=K_local.shape[-2], tie_break=tie_break)
