"""Data-parallel sharding of the fused linear logp over tokens.

Rows are independent for logp, lse and grad_hidden, so ranks take
contiguous token shards and need no exchange for them.  grad_weight and
grad_bias are sums over tokens: the caller's gradient synchronisation adds
the ranks' partial tables.  `reduce_sum_fixed_order` does that sum in
ascending rank order on every rank (gather, then add rank 0, 1, ...), so the
result is bitwise identical on all ranks and from run to run, whatever the
transport.
"""
from __future__ import annotations


def shard_rows(N: int, world: int, rank: int) -> tuple[int, int]:
    """[begin, end) of rank's contiguous token shard (sizes differ by <= 1)."""
    if world < 1 or not (0 <= rank < world):
        raise ValueError("bad world/rank")
    base, rem = divmod(int(N), world)
    begin = rank * base + min(rank, rem)
    return begin, begin + base + (1 if rank < rem else 0)


def reduce_sum_fixed_order(t, group=None):
    """Sum of `t` over the ranks of `group`, added in ascending rank order.

    Returns a new tensor (same dtype and device); the input is unchanged.
    The accumulation happens in the tensor's dtype: ((t0 + t1) + t2) + ...
    """
    import torch
    import torch.distributed as dist

    world = dist.get_world_size(group)
    if world == 1:
        return t.clone()
    parts = [torch.empty_like(t) for _ in range(world)]
    dist.all_gather(parts, t.contiguous(), group=group)
    out = parts[0].clone()
    for p in parts[1:]:
        out.add_(p)
    return out
