"""Data-parallel sharding of the fused linear logp over tokens.

Rows are independent for logp, lse and grad_hidden, so ranks take
contiguous token shards and need no exchange for them.  grad_weight and
grad_bias are sums over tokens (issue #261, "Current accumulation": one FP32
table accumulated over token chunks; across ranks the chunks are the ranks'
shards), so the gradient synchronisation adds the ranks' partial tables.

`reduce_scatter_fixed_order` is that exchange: the table is cut into `world`
contiguous slices, rank r receives every rank's slice r (one all-to-all,
(world - 1) / world of the table sent and received per rank) and adds them in
ascending rank order with the library's `ll_sum_ordered` kernel.  Each slice
is summed once, by its owner, in a fixed order, so the result does not depend
on the transport or its timing.  `reduce_sum_fixed_order` follows it with an
all-gather of the slices, for an optimiser that needs the whole table: the
same bits on every rank.  Memory per rank is O(table), not O(world x table).

CUDA tensors are added by the library (which must be built); CPU tensors (the
gloo tests of this logic) by the same ascending FP32 additions in torch.
"""
from __future__ import annotations


def shard_rows(N: int, world: int, rank: int) -> tuple[int, int]:
    """[begin, end) of rank's contiguous token shard (sizes differ by <= 1)."""
    if world < 1 or not (0 <= rank < world):
        raise ValueError("bad world/rank")
    base, rem = divmod(int(N), world)
    begin = rank * base + min(rank, rem)
    return begin, begin + base + (1 if rank < rem else 0)


def slice_bytes(numel: int, elem_size: int, world: int) -> dict:
    """Bytes one rank sends and receives in reduce_scatter_fixed_order (and
    in the all-gather that completes reduce_sum_fixed_order) for a table of
    `numel` elements."""
    sizes = [e - b for b, e in (shard_rows(numel, world, r) for r in range(world))]
    worst = max(sizes) if sizes else 0
    moved = (numel - min(sizes)) * elem_size if world > 1 else 0
    return {"reduce_scatter_send": moved, "reduce_scatter_recv": (world - 1) * worst * elem_size,
            "all_gather": moved}


def _sum_parts(parts, out):
    """out = parts[0] + parts[1] + ... (ascending; FP32 accumulation, FP64
    for float64 tables on the host)."""
    if parts.is_cuda:
        import cross_entropy_rl_gb300 as ll

        return ll.sum_ordered(parts, out=out)
    import torch

    wide = torch.float64 if parts.dtype == torch.float64 else torch.float32
    acc = parts[0].to(wide).clone()
    for k in range(1, parts.shape[0]):
        acc += parts[k].to(wide)
    out.copy_(acc)
    return out


def reduce_scatter_fixed_order(t, group=None, recv=None):
    """This rank's slice of the sum of `t` over the ranks of `group`.

    t is flattened and cut into world contiguous slices (shard_rows over its
    elements); rank r returns slice r of sum_k t_k, added in ascending rank
    order k = 0, 1, ... (FP32 accumulation, one rounding to t's dtype).
    `recv` (optional): a buffer of world x (slice r's size) elements of t's
    dtype on t's device, reused between calls.
    """
    import torch
    import torch.distributed as dist

    world = dist.get_world_size(group)
    rank = dist.get_rank(group)
    flat = t.contiguous().view(-1)
    b, e = shard_rows(flat.numel(), world, rank)
    n = e - b
    if world == 1:
        return flat.clone()
    sizes = [hi - lo for lo, hi in (shard_rows(flat.numel(), world, r) for r in range(world))]
    if recv is None:
        recv = torch.empty(world * n, dtype=flat.dtype, device=flat.device)
    elif recv.numel() != world * n or recv.dtype != flat.dtype:
        raise ValueError("recv must hold world x slice elements of t's dtype")
    dist.all_to_all_single(recv, flat, output_split_sizes=[n] * world,
                           input_split_sizes=sizes, group=group)
    out = torch.empty(n, dtype=flat.dtype, device=flat.device)
    return _sum_parts(recv.view(world, n), out)


def reduce_sum_fixed_order(t, group=None):
    """Sum of `t` over the ranks of `group`, every slice added in ascending
    rank order by its owner (reduce_scatter_fixed_order), then all-gathered:
    a new tensor of t's shape, dtype and device, bitwise identical on every
    rank.  The input is unchanged."""
    import torch
    import torch.distributed as dist

    world = dist.get_world_size(group)
    if world == 1:
        return t.clone()
    flat = t.contiguous().view(-1)
    mine = reduce_scatter_fixed_order(flat, group)
    sizes = [e - b for b, e in (shard_rows(flat.numel(), world, r) for r in range(world))]
    if len(set(sizes)) == 1:
        out = torch.empty_like(flat)
        dist.all_gather_into_tensor(out, mine, group=group)
    else:  # slices differ by one element: gather padded slices, then cut
        m = max(sizes)
        pad = torch.zeros(m, dtype=flat.dtype, device=flat.device)
        pad[: mine.numel()] = mine
        gathered = torch.empty(world * m, dtype=flat.dtype, device=flat.device)
        dist.all_gather_into_tensor(gathered, pad, group=group)
        out = torch.cat([gathered[r * m: r * m + sizes[r]] for r in range(world)])
    return out.view(t.shape)
