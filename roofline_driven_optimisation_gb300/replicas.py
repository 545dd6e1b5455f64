"""Host-side logic of multi-GPU runs.

A GEMM shards by columns with no exchange: rank r of G computes
C[:, n0:n1] = alpha * A * B[:, n0:n1] + beta * C[:, n0:n1] with A replicated,
and the full C is the concatenation of the shards.  The benchmark runs one
replica of the hot path per rank (weak scaling); its time is the maximum over
ranks and its throughput counts every rank's work.  Nothing here moves matrix
data between ranks; the only collective is on host-side scalars.
"""
from __future__ import annotations


def column_shard(n: int, world: int, rank: int) -> tuple[int, int]:
    """Contiguous columns [n0, n1) of rank `rank` among `world` ranks.

    Shard widths differ by at most one column; a shard may be empty when
    n < world.
    """
    if world < 1 or not 0 <= rank < world or n < 0:
        raise ValueError(f"bad shard request n={n} world={world} rank={rank}")
    return n * rank // world, n * (rank + 1) // world


def max_over_ranks(value: float, dist=None, device=None) -> float:
    """Maximum of a host scalar over all ranks (the scalar itself without a
    process group)."""
    if dist is None or not dist.is_available() or not dist.is_initialized():
        return float(value)
    import torch
    t = torch.tensor([float(value)], dtype=torch.float64,
                     device=device if device is not None else "cpu")
    dist.all_reduce(t, op=dist.ReduceOp.MAX)
    return float(t.item())


def whole_job_rate(units_per_rank: float, world: int, seconds: float) -> float:
    """Units per second of the whole job: every rank's units over the slowest
    rank's time."""
    if seconds <= 0:
        raise ValueError("time must be positive")
    return world * units_per_rank / seconds
