"""Host-side logic for running the path on several GPUs.

The rows of every operation are independent and the RMS statistic is per row,
so the path shards with no exchange step: each rank either runs its own
replica of a workload (weak scaling, what the benchmark does) or takes a
contiguous block of rows of one workload.  The only collective is the
benchmark's max-reduction of the timed region's length, which is measurement,
not data path.
"""
from __future__ import annotations


def row_block(rows: int, rank: int, world: int):
    """[start, end) of the rows rank `rank` of `world` owns: contiguous blocks
    whose sizes differ by at most one."""
    if world < 1 or not 0 <= rank < world or rows < 0:
        raise ValueError("bad rank/world/rows")
    base, extra = divmod(rows, world)
    start = rank * base + min(rank, extra)
    return start, start + base + (1 if rank < extra else 0)


def max_over_ranks(value: float, device=None) -> float:
    """The maximum of `value` over all ranks of the default process group (or
    `value` itself without one)."""
    import torch
    import torch.distributed as dist
    if not (dist.is_available() and dist.is_initialized()):
        return float(value)
    t = torch.tensor([float(value)], dtype=torch.float64,
                     device=device if device is not None else "cpu")
    dist.all_reduce(t, op=dist.ReduceOp.MAX)
    return float(t.item())


def aggregate_gbs(bytes_per_rank_step: int, steps: int, world: int, max_ms: float) -> float:
    """Whole-job GB/s: the bytes every rank moved over the slowest rank's time."""
    if max_ms <= 0:
        raise ValueError("non-positive time")
    return bytes_per_rank_step * steps * world / (max_ms * 1e-3) / 1e9
