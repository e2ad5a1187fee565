"""Host logic for running the hot path on several GPUs, one process each.

The path has no exchange step: rows of different sequences are independent
(each reads only its own sequence's keys, latent blocks and table), and the
rows of one K-token verify share a sequence.  So a batch is partitioned by
whole sequences -- a contiguous range of sequence groups per rank, never
splitting a verify group -- and every rank runs its share with no collective
on the data path.  The only cross-rank communication is timing: the step
time of a run is the maximum over ranks.
"""
from __future__ import annotations


def shard_groups(n_groups: int, rank: int, world: int) -> range:
    """Contiguous range of sequence groups handled by ``rank`` (sizes differ by
    at most one; lower ranks take the extra groups)."""
    if world < 1 or not 0 <= rank < world:
        raise ValueError("rank must lie in [0, world)")
    base, extra = divmod(n_groups, world)
    start = rank * base + min(rank, extra)
    return range(start, start + base + (1 if rank < extra else 0))


def shard_rows(rows: int, rows_per_seq: int, rank: int, world: int) -> range:
    """Rows of ``rank`` when consecutive groups of ``rows_per_seq`` rows share
    one sequence."""
    if rows_per_seq < 1 or rows % rows_per_seq:
        raise ValueError("rows must be a multiple of rows_per_seq")
    g = shard_groups(rows // rows_per_seq, rank, world)
    return range(g.start * rows_per_seq, g.stop * rows_per_seq)


def max_over_ranks(value: float, group=None) -> float:
    """Maximum of a per-rank float over the process group (identity when
    torch.distributed is not initialised)."""
    import torch
    import torch.distributed as dist
    if not (dist.is_available() and dist.is_initialized()):
        return float(value)
    backend = dist.get_backend(group)
    dev = torch.device("cuda", torch.cuda.current_device()) if backend == "nccl" else torch.device("cpu")
    t = torch.tensor([float(value)], dtype=torch.float64, device=dev)
    dist.all_reduce(t, op=dist.ReduceOp.MAX, group=group)
    return float(t.item())
