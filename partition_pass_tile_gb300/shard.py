"""Scan, select-if and partition of an array split over the ranks of a process group.

Each rank holds one contiguous shard (``shard_bounds``) in its own device
memory.  A shard needs only what the shards before it contribute, which is
the exclusive scan of the P per-shard totals; so every operation is

    pre-pass (libgc: gc_reduce / gc_count_if)  ->  exchange (one all-gather
    of P 32-bit words)  ->  offsets (libgc: gc_shard_offsets, on the device)
    ->  placed pass (libgc: gc_exclusive_scan_carry / gc_select_if_at /
    gc_partition_at)

all on the current stream, with nothing read back to the host.  The only
collective is the all-gather of the totals: NCCL between GPUs, gloo on CPU
tensors.  No rank's kernels touch another rank's memory: each writes its
own output ranges into ``out``, the whole output as this rank holds it, and
assembling the ranks' ranges on one device (a copy of m elements) is left
to the caller.

This module does none of the method's arithmetic: the totals, the offsets
and every output element are computed by libgc's kernels; here there is only
the choice of shard bounds and the collective.
"""

from __future__ import annotations

import torch

from . import gc


def shard_bounds(n: int, parts: int, rank: int) -> tuple[int, int]:
    """[start, stop) of shard `rank` when n elements are cut into `parts`
    contiguous shards whose sizes differ by at most one (the first n % parts
    shards take one more)."""
    if parts <= 0 or not 0 <= rank < parts or n < 0:
        raise ValueError("need parts >= 1, 0 <= rank < parts and n >= 0")
    base, extra = divmod(n, parts)
    start = rank * base + min(rank, extra)
    return start, start + base + (1 if rank < extra else 0)


def shard_sizes(n: int, parts: int) -> list[int]:
    return [b - a for a, b in (shard_bounds(n, parts, r) for r in range(parts))]


def _group_info(group):
    import torch.distributed as dist
    return dist.get_rank(group), dist.get_world_size(group)


def gather_totals(local: torch.Tensor, group=None) -> torch.Tensor:
    """The exchange: every rank's 1-element total, gathered in rank order on
    every rank (an all-gather of P 32-bit words, moved as their bits)."""
    import torch.distributed as dist
    _, parts = _group_info(group)
    bits = local.view(torch.int32) if local.dtype == torch.uint32 else local
    out = torch.empty(parts, dtype=bits.dtype, device=bits.device)
    dist.all_gather_into_tensor(out, bits.contiguous(), group=group)
    return out.view(local.dtype)


def exclusive_scan(x: torch.Tensor, group=None, out: torch.Tensor | None = None,
                   ws: torch.Tensor | None = None):
    """This rank's part of the exclusive scan of the concatenated shards
    -> (out, total through this shard)."""
    rank, _ = _group_info(group)
    totals = gather_totals(gc.reduce(x, ws=ws), group)
    carry = gc.shard_offsets(gc.OP_EXCLUSIVE_SCAN, totals, rank)
    return gc.exclusive_scan_carry(x, carry, out=out, ws=ws)


def select_if(x: torch.Tensor, pred, out: torch.Tensor, group=None,
              ws: torch.Tensor | None = None):
    """This rank's survivors, written to out[base, base + count) of the whole
    output -> (out, count, base) with count and base device tensors."""
    rank, _ = _group_info(group)
    counts = gather_totals(gc.count_if(x, pred, ws=ws), group)
    base = gc.shard_offsets(gc.OP_SELECT_IF, counts, rank, dtype=gc.U32)
    out, count = gc.select_if_at(x, pred, out, base, ws=ws)
    return out, count, base


def partition(x: torch.Tensor, pred, out: torch.Tensor, sizes: list[int], group=None,
              ws: torch.Tensor | None = None):
    """This rank's kept and rejected elements, written to their places in the
    stable partition of the whole array (`sizes`: every shard's element
    count, in rank order) -> (out, kept count, offsets)."""
    rank, _ = _group_info(group)
    counts = gather_totals(gc.count_if(x, pred, ws=ws), group)
    offsets = gc.shard_offsets(gc.OP_PARTITION, counts, rank, sizes=sizes, dtype=gc.U32)
    out, kept = gc.partition_at(x, pred, out, offsets, ws=ws)
    return out, kept, offsets
