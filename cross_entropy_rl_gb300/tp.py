"""Vocab-parallel (tensor-parallel) composition of the fused linear logp.

Each rank holds the rows [v0, v1) of W (and b) of one contiguous vocab
shard.  The shards start on LSE segment boundaries (multiples of
SEGMENT_COLS vocab entries), so a shard's per-segment (max, sum-exp)
partials are exactly those of the whole-vocab forward; gathered in rank
order and merged in ascending segment order they give the single-GPU logp
and lse bitwise, whatever the number of ranks (RL-Kernel PR #495: the
tensor-parallel shards start and end on a fixed vocab tile boundary, and
the coordinated cross entropy broke the cross-layout bitwise contract for
282 of 1200 rows).

Exchanges, all fixed-order or order-free:
  forward   all_gather of the [S_max, N] (m, s) partials (each rank padded
            to S_max segments with (-inf, 0), which the merge ignores
            bitwise) and a MAX all-reduce of zy (z at the target, -inf on
            every rank but its owner: an exact selection);
  backward  grad_hidden = sum of the ranks' parts in ascending rank order
            (gather, then add); grad_weight / grad_bias stay on their shard.

The per-shard calls go to `impl` (default: this package's C ABI binding);
a stand-in with the same three functions lets the host logic run on CPU
ranks.
"""
from __future__ import annotations

from . import dp

SEGMENT_COLS = 1024


def shard_bounds(V: int, world: int) -> list[tuple[int, int]]:
    """[(v0, v1)] per rank: whole segments, as even as possible, in order.
    Ranks beyond the number of segments get an empty shard (v0 == v1)."""
    if world < 1 or V < 1:
        raise ValueError("bad V / world")
    segs = -(-int(V) // SEGMENT_COLS)
    base, rem = divmod(segs, world)
    out, s0 = [], 0
    for r in range(world):
        s1 = s0 + base + (1 if r < rem else 0)
        out.append((min(s0 * SEGMENT_COLS, V), min(s1 * SEGMENT_COLS, V)))
        s0 = s1
    return out


def max_segments(V: int, world: int) -> int:
    """Segments of the largest shard of shard_bounds(V, world)."""
    return max(-(-(v1 - v0) // SEGMENT_COLS) for v0, v1 in shard_bounds(V, world))


def _impl(impl):
    if impl is not None:
        return impl
    import cross_entropy_rl_gb300 as binding
    return binding


def forward(hidden, weight, bias, targets, v0: int, V: int, group=None, impl=None,
            temperature=1.0):
    """(logp, lse) [N] of the whole vocab on every rank of `group`.

    weight / bias: this rank's shard rows (weight.shape[0] may be 0 for an
    empty shard); v0: the shard's first vocab id; targets: global ids."""
    import torch
    import torch.distributed as dist

    f = _impl(impl)
    world = dist.get_world_size(group)
    N = hidden.shape[0]
    Vs = weight.shape[0]
    S_max = max_segments(V, world)
    dev = hidden.device
    part_m = torch.full((S_max, N), -float("inf"), dtype=torch.float32, device=dev)
    part_s = torch.zeros((S_max, N), dtype=torch.float32, device=dev)
    zy = torch.full((N,), -float("inf"), dtype=torch.float32, device=dev)
    if Vs > 0 and N > 0:
        S = -(-Vs // SEGMENT_COLS)
        f.forward_shard(hidden, weight, bias, targets, v0, V, temperature=temperature,
                        out=(part_m[:S], part_s[:S], zy))
    gm = [torch.empty_like(part_m) for _ in range(world)]
    gs = [torch.empty_like(part_s) for _ in range(world)]
    dist.all_gather(gm, part_m, group=group)
    dist.all_gather(gs, part_s, group=group)
    dist.all_reduce(zy, op=dist.ReduceOp.MAX, group=group)
    all_m = torch.cat(gm, dim=0).contiguous()
    all_s = torch.cat(gs, dim=0).contiguous()
    return f.lse_merge(all_m, all_s, zy, targets, V)


def backward(grad_logp, hidden, weight, bias, targets, lse, v0: int, V: int, group=None,
             impl=None, need_db=None, token_chunks=0, temperature=1.0):
    """(grad_hidden [N, D] float32, equal on every rank; this shard's
    grad_weight rows; its grad_bias rows or None)."""
    import torch

    f = _impl(impl)
    N, D = hidden.shape
    Vs = weight.shape[0]
    if need_db is None:
        need_db = bias is not None
    if Vs > 0:
        dh, dW, db = f.backward_shard(grad_logp, hidden, weight, bias, targets, lse, v0, V,
                                      need_db=need_db, token_chunks=token_chunks,
                                      temperature=temperature)
    else:
        dh = torch.zeros(N, D, dtype=torch.float32, device=hidden.device)
        dW = torch.zeros(0, D, dtype=torch.float32, device=hidden.device)
        db = torch.zeros(0, dtype=torch.float32, device=hidden.device) if need_db else None
    # every rank reduces the same dtype (FP32), whatever produced its part
    return dp.reduce_sum_fixed_order(dh.float().contiguous(), group), dW, db
