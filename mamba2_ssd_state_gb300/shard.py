"""Data-parallel sharding of the SSD ops across GPUs (one process per GPU).

The ops have no cross-sequence or cross-request data flow: every packed sequence of a
prefill batch and every decode row is independent.  So a multi-GPU job shards whole
sequences (prefill) or rows (decode) across ranks, each rank runs the unchanged kernels
on its shard, and no collective sits on the data path.  Only timing uses one
(``max_over_ranks``).
"""
from __future__ import annotations


def partition_sequences(seqlens, world_size):
    """Whole sequences to ranks, longest first, each to the rank with the fewest tokens
    so far (ties to the lower rank).  Returns, per rank, the sorted sequence indices."""
    if world_size < 1:
        raise ValueError("world_size must be >= 1")
    order = sorted(range(len(seqlens)), key=lambda i: (-int(seqlens[i]), i))
    load = [0] * world_size
    parts = [[] for _ in range(world_size)]
    for i in order:
        r = min(range(world_size), key=lambda k: (load[k], k))
        parts[r].append(i)
        load[r] += int(seqlens[i])
    return [sorted(p) for p in parts]


def partition_rows(batch, world_size):
    """Decode rows to ranks in contiguous, near-equal blocks."""
    base, extra = divmod(int(batch), world_size)
    out, start = [], 0
    for r in range(world_size):
        n = base + (1 if r < extra else 0)
        out.append(list(range(start, start + n)))
        start += n
    return out


def max_over_ranks(value, device=None):
    """Largest value over all ranks (the job's time is its slowest rank's)."""
    import torch
    import torch.distributed as dist

    if not (dist.is_available() and dist.is_initialized()) or dist.get_world_size() == 1:
        return float(value)
    t = torch.tensor([float(value)], dtype=torch.float64, device=device)
    dist.all_reduce(t, op=dist.ReduceOp.MAX)
    return float(t.item())
