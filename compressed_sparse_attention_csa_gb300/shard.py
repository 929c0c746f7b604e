"""Batch sharding of the decode step across processes (one process per GPU).

Sequences of a decode batch are independent: each has its own compressed caches, queries,
window and output, and no stage of the step (compress, indexer, top-k, attention) reads
another sequence's data.  N processes therefore split a global batch into contiguous slices
and each runs the whole step on its slice with no exchange on the data path; the only
collectives are host-side (a barrier around the timed region and the reductions below).
"""
from typing import Tuple


def shard_rows(global_batch: int, world: int, rank: int) -> Tuple[int, int]:
    """(first sequence, count) of `rank`'s contiguous slice; the first global_batch % world
    ranks take one extra sequence, so every sequence belongs to exactly one rank."""
    if world < 1 or not 0 <= rank < world or global_batch < 0:
        raise ValueError(f"bad shard request: batch {global_batch}, world {world}, rank {rank}")
    base, extra = divmod(global_batch, world)
    count = base + (1 if rank < extra else 0)
    start = rank * base + min(rank, extra)
    return start, count


def _reduce(value: float, op) -> float:
    import torch
    import torch.distributed as dist
    if not (dist.is_available() and dist.is_initialized()) or dist.get_world_size() == 1:
        return float(value)
    dev = torch.device("cpu")
    if dist.get_backend() == "nccl":
        dev = torch.device("cuda", torch.cuda.current_device())
    t = torch.tensor([float(value)], dtype=torch.float64, device=dev)
    dist.all_reduce(t, op=op)
    return float(t.item())


def max_over_ranks(value: float) -> float:
    """Largest value over all ranks (the job's time is its slowest rank's time)."""
    import torch.distributed as dist
    return _reduce(value, dist.ReduceOp.MAX)


def sum_over_ranks(value: float) -> float:
    """Sum over all ranks (units processed by the whole job)."""
    import torch.distributed as dist
    return _reduce(value, dist.ReduceOp.SUM)


def job_throughput(units_per_rank: float, seconds_per_rank: float) -> float:
    """Whole-job units per second: units summed over ranks / the slowest rank's time."""
    units = sum_over_ranks(units_per_rank)
    seconds = max_over_ranks(seconds_per_rank)
    return units / seconds
