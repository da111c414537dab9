"""Multi-rank plumbing: one process per GPU, launched by torchrun.

The (b, h) units of the attention are independent in the forward and the
backward, and R, u, v are per head, so the work shards with no collective on
the data path:
  * by head: every gradient of a rank's heads is complete on that rank;
  * by batch row: dR, du, dv are sums over b and need one sum over ranks.
The benchmark runs one independent replica per rank (weak scaling); the only
collectives are the barrier around the timed region and the max of the
ranks' times. Works with any torch.distributed backend (gloo on CPU, nccl
on GPUs).
"""
from __future__ import annotations

import os


def rank_world() -> tuple[int, int]:
    """(rank, world size) from the launcher's environment (1 process: (0, 1))."""
    return int(os.environ.get("RANK", "0")), int(os.environ.get("WORLD_SIZE", "1"))


def shard(n: int, rank: int, world: int) -> tuple[int, int]:
    """Contiguous [lo, hi) share of n units for `rank`; shares differ by at most one."""
    if world < 1 or not 0 <= rank < world or n < 0:
        raise ValueError(f"bad shard request n={n} rank={rank} world={world}")
    base, extra = divmod(n, world)
    lo = rank * base + min(rank, extra)
    return lo, lo + base + (1 if rank < extra else 0)


def replica_seed(base_seed: int, rank: int) -> int:
    """Seed of a rank's replica: distinct ranks draw distinct synthetic data."""
    return int(base_seed) + 1000003 * int(rank)


def max_over_ranks(x: float, world: int, device=None) -> float:
    """Maximum of a per-rank scalar over all ranks (the job's time is that of
    its slowest rank). No-op for one rank."""
    if world <= 1:
        return float(x)
    import torch
    import torch.distributed as dist
    t = torch.tensor([float(x)], dtype=torch.float64, device=device)
    dist.all_reduce(t, op=dist.ReduceOp.MAX)
    return float(t.item())


def whole_job_rate(units_per_rank: float, world: int, seconds: float) -> float:
    """Units all ranks processed per second, timed by the slowest rank."""
    if seconds <= 0:
        raise ValueError("time must be positive")
    return world * units_per_rank / seconds
