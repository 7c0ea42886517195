"""Splitting one KDA workload across ranks.

By heads: every (sequence, head) chain of the operator is independent ("Kimi
K3：从三条信息流到完整系统", §KDA 是带逐通道遗忘的 delta rule: the recurrence of
eq. (1) runs per head), so a workload partitions across GPUs with no
exchange on the data path: rank r runs the heads [h0, h1) of every token and
sequence, and the outputs of the ranks are disjoint slices of the unsplit
outputs along the head axis.

By tokens (KCP, §FlashKDA 与 KCP, eq. (17)): rank r holds the r-th slice of
T tokens of the same sequences; the ranks exchange one (S0, Phi) pair per
sequence and head (kcp_prefill).

This module does the host-side bookkeeping and the exchange; the
arithmetic stays in the library's kernels on each rank.
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


def kcp_prefill(q, k, v, g_raw, beta, init_state=None, *, group=None, **params):
    """Sequence-parallel prefill: this rank's slice of T tokens of B
    sequences (q, k, g_raw [B, T, H, 128], v [B, T, H, 128], beta [B, T, H],
    bf16 on this rank's GPU; rank 0 holds the first slice).  init_state
    [B, H, 128, 128] (rank 0 only) or None.  One all-gather of the ranks'
    (S0, Phi) pairs ([B, 2, H, 128, 128] float32 each) over `group`; over a
    gloo group the pairs travel through host memory.  Returns (out [B, T, H,
    128] for this rank's tokens, the state after this rank's tokens: the
    sequences' final state on the last rank).  params: the gate and scale
    arguments of kda_chunk_fwd."""
    import torch
    import torch.distributed as dist

    from . import kda

    rank, world = dist.get_rank(group), dist.get_world_size(group)
    B, T, H, dk = q.shape
    dev = q.device
    if rank == 0:
        out, fin = kda.kda_chunk_fwd(q, k, v, g_raw, beta, init_state, **params)
        pair = torch.zeros((B, 2, H, dk, dk), dtype=torch.float32, device=dev)
        pair[:, 0] = fin
        ws = None
    else:
        ws = torch.empty(kda.kcp_workspace_bytes(B, T, H, dk, v.shape[-1]), dtype=torch.uint8, device=dev)
        pair = kda.kda_chunk_fwd_kcp_part(q, k, v, g_raw, beta, ws, **params)
    host = dist.get_backend(group) == "gloo"
    send = pair.cpu() if host else pair
    gathered = [torch.empty_like(send) for _ in range(world)]
    dist.all_gather(gathered, send, group=group)
    if rank == 0:
        return out, fin
    pairs = torch.stack([g.to(dev) for g in gathered[: rank + 1]]).contiguous()
    return kda.kda_chunk_fwd_kcp_finish(pairs, rank, ws, B, T, H, dk=dk, dv=v.shape[-1])
