"""Splitting one KDA workload across ranks by heads (host-side bookkeeping).

Every (sequence, head) chain of the operator is independent ("Kimi K3：从三条
信息流到完整系统", §KDA 是带逐通道遗忘的 delta rule: the recurrence of eq. (1)
runs per head), so a workload partitions across GPUs with no exchange on the
data path: rank r runs the heads [h0, h1) of every token and sequence, and
the outputs of the ranks are disjoint slices of the unsplit outputs along the
head axis.  This module only computes the ranges and slices; the arithmetic
stays in the library's kernels on each rank.
"""
from __future__ import annotations


def head_range(rank: int, world: int, H: int):
    """Heads [h0, h1) of `rank` when H heads are split over `world` ranks as
    evenly as possible (the first H % world ranks take one extra head)."""
    if world < 1 or not 0 <= rank < world:
        raise ValueError(f"rank {rank} outside a world of {world}")
    if H < world:
        raise ValueError(f"{H} heads cannot be split over {world} ranks")
    base, extra = divmod(H, world)
    h0 = rank * base + min(rank, extra)
    return h0, h0 + base + (1 if rank < extra else 0)


def shard_heads(t, rank: int, world: int, axis: int):
    """The rank's contiguous head slice of tensor `t` along `axis` (a copy,
    contiguous, ready for the library's packed layouts)."""
    h0, h1 = head_range(rank, world, t.shape[axis])
    idx = [slice(None)] * t.dim()
    idx[axis] = slice(h0, h1)
    return t[tuple(idx)].contiguous()


def unshard_heads(parts, axis: int):
    """Reassemble the ranks' head slices (in rank order) along `axis`."""
    import torch
    return torch.cat(list(parts), dim=axis)
