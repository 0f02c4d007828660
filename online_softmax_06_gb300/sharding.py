"""Host-side work partitioning for one process per GPU.

The attention forward has no exchange step between (sequence, head) pairs:
every pair is an independent problem (the grid of the kernel is exactly
these pairs times Q tiles).  A multi-GPU job therefore splits pairs across
ranks with no collective on the data path:

  * ``shard_range(n, rank, world)``: the contiguous block of n units a rank
    owns (sizes differ by at most one);
  * ``batch_shard`` / ``head_shard``: that rule applied to sequences or heads;
  * ``reduce_max_ms``: the job time is the slowest rank's time (the only
    collective, and it is for measurement, not for the data path);
  * ``job_throughput``: work summed over ranks divided by that time.

The benchmark runs weak scaling: each rank keeps a full replica of the
workload, so every rank owns all of its own units.
"""
from __future__ import annotations


def shard_range(n: int, rank: int, world: int) -> tuple[int, int]:
    """[begin, end) of the n units owned by `rank` out of `world`."""
    if world < 1 or not 0 <= rank < world or n < 0:
        raise ValueError("bad shard arguments")
    base, extra = divmod(n, world)
    begin = rank * base + min(rank, extra)
    return begin, begin + base + (1 if rank < extra else 0)


def batch_shard(B: int, rank: int, world: int) -> tuple[int, int]:
    """Sequences [b0, b1) of a dense [B, N, H, d] batch for this rank (a
    contiguous slice of the tensors)."""
    return shard_range(B, rank, world)


def head_shard(H: int, rank: int, world: int) -> tuple[int, int]:
    """Heads [h0, h1) for this rank."""
    return shard_range(H, rank, world)


def reduce_max_ms(ms: float, dist=None, device=None) -> float:
    """Maximum of `ms` over the ranks of the default process group."""
    if dist is None or not dist.is_initialized() or dist.get_world_size() == 1:
        return float(ms)
    import torch
    t = torch.tensor([float(ms)], dtype=torch.float64, device=device)
    dist.all_reduce(t, op=dist.ReduceOp.MAX)
    return float(t.item())


def job_throughput(units_per_rank: list[float], ms_max: float) -> float:
    """Units processed by all ranks per second, timed by the slowest rank."""
    if ms_max <= 0:
        raise ValueError("time must be positive")
    return sum(units_per_rank) / (ms_max / 1e3)
