"""Lane-sharded schedule build over a torch.distributed group (argument plumbing and the one
exchange; every computation runs in libtsa).

The topology schedule is one CSR shared by all lanes, built from the lane-mean key-block
centroids.  When the lanes are spread over ranks, each rank computes the block sums of its
own lanes (tsa_block_sums), the ranks all-gather them in global lane order, and every rank
builds the CSR from all of them (tsa_build_schedule_from_sums).  The centroid sums the lanes
in ascending order on every rank, exactly as the single-GPU build does, so every rank gets
the single-GPU CSR bit for bit.  The exchange is lanes * nb * D float64 values (33.5 MB for
64 lanes of [32768, 128] keys).  Rank r holds a contiguous run of lanes, ranks in order;
shards may differ in size.  The attention itself needs no exchange: lanes are independent
and the CSR is shared.

With NCCL the block sums move between GPUs directly; with gloo (CPU collectives, e.g. several
processes sharing one GPU) they go through host memory and come back to the GPU.
"""
from __future__ import annotations

import torch
import torch.distributed as dist

from .binding import tsa_block_sums, tsa_build_schedule_from_sums


def _through_host(t: torch.Tensor, group) -> bool:
    return t.is_cuda and dist.get_backend(group) == "gloo"


def gather_block_sums(local: torch.Tensor, group=None, counts: list[int] | None = None) -> torch.Tensor:
    """All-gather [lanes_r, nb, D] float64 block sums into [sum of lanes_r, nb, D], rank order.
    `counts` (every rank's lanes_r, if the caller knows them) saves the exchange of the counts."""
    world = dist.get_world_size(group)
    if world == 1:
        return local
    device = local.device
    if _through_host(local, group):
        local = local.cpu()
    if counts is None:
        c = torch.tensor([local.shape[0]], dtype=torch.int64, device=local.device)
        all_counts = [torch.empty_like(c) for _ in range(world)]
        dist.all_gather(all_counts, c, group=group)
        counts = [int(x.item()) for x in all_counts]
    if len(counts) != world or counts[dist.get_rank(group)] != local.shape[0]:
        raise ValueError("counts must list every rank's number of lanes")
    most = max(counts)
    padded = local
    if local.shape[0] < most:  # all_gather moves equal-sized tensors
        padded = torch.zeros((most,) + tuple(local.shape[1:]), dtype=local.dtype, device=local.device)
        padded[: local.shape[0]] = local
    parts = [torch.empty_like(padded) for _ in range(world)]
    dist.all_gather(parts, padded.contiguous(), group=group)
    out = torch.cat([p[:k] for p, k in zip(parts, counts)], dim=0).contiguous()
    return out.to(device, non_blocking=False) if out.device != device else out


def build_schedule_lane_sharded(K_local: torch.Tensor, block: int = 64, sink: int = 1, local_radius: int = 1,
                                topk: int = 2, *, tie_break: str = "index", group=None,
                                counts: list[int] | None = None, salience: bool = False):
    """The topology CSR of the keys whose lanes are spread over the group's ranks (this rank:
    K_local, [lanes_r, S, D] or [B_r, H, S, D] on its GPU).  Every rank returns the same
    (row_ptr, col_idx) (and the squared merge distance per block with salience=True)."""
    if K_local.numel() == 0:  # a rank that holds no lanes still takes part in the exchange
        S, D = K_local.shape[-2], K_local.shape[-1]
        sums = torch.empty((0, -(-S // block), D), dtype=torch.float64, device=K_local.device)
    else:
        sums = tsa_block_sums(K_local, block)
    return tsa_build_schedule_from_sums(gather_block_sums(sums, group, counts), block, sink, local_radius,
                                        topk, S=K_local.shape[-2], tie_break=tie_break, salience=salience)
