"""torch.autograd wrapper over the scheduled-attention kernels (argument plumbing only).

``scheduled_attention(Q, K, V, row_ptr, col_idx, scale, block=64)`` runs
tsa_scheduled_attention_fwd and keeps its log-sum-exp; its backward runs
tsa_scheduled_attention_backward (blocks of 64 or 128 tokens).  The CSR is not differentiable.
"""
from __future__ import annotations

import torch

from .binding import tsa_scheduled_attention_backward, tsa_scheduled_attention_fwd


class ScheduledAttention(torch.autograd.Function):
    @staticmethod
    def forward(ctx, Q, K, V, row_ptr, col_idx, scale, block):
        Q, K, V = (t.contiguous() for t in (Q, K, V))
        O, lse = tsa_scheduled_attention_fwd(Q, K, V, row_ptr, col_idx, scale, block=block)
        ctx.save_for_backward(Q, K, V, O, lse, row_ptr, col_idx)
        ctx.scale = scale
        ctx.block = block
        return O

    @staticmethod
    def backward(ctx, dO):
        Q, K, V, O, lse, row_ptr, col_idx = ctx.saved_tensors
        dQ, dK, dV = tsa_scheduled_attention_backward(Q, K, V, O, dO.contiguous(), lse, row_ptr, col_idx,
                                                      ctx.scale, block=ctx.block)
        return dQ, dK, dV, None, None, None, None


def scheduled_attention(Q, K, V, row_ptr, col_idx, scale: float | None = None, block: int = 64):
    if scale is None:
        scale = Q.shape[-1] ** -0.5
    return ScheduledAttention.apply(Q, K, V, row_ptr, col_idx, float(scale), int(block))
