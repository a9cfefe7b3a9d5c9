"""Host-side logic for running the path on several GPUs as independent replicas.

Every (batch, head) problem of attention forward + JVP is independent and the
method has no exchange step, so N GPUs run N replicas with no collective on
the data path.  Only the timing is combined: each rank's time is reduced with
MAX and the throughput is all ranks' work over the slowest rank's time.
``shard`` splits a batch*head range when a caller wants one problem spread
over ranks instead (each rank then calls the ABI on its own slice).
"""

from __future__ import annotations

from typing import Tuple

import torch
import torch.distributed as dist


def shard(n_units: int, rank: int, world: int) -> Tuple[int, int]:
    """Contiguous [start, stop) of n_units for this rank; sizes differ by at most one."""
    if world <= 0 or not 0 <= rank < world:
        raise ValueError("bad rank / world size")
    base, extra = divmod(n_units, world)
    start = rank * base + min(rank, extra)
    return start, start + base + (1 if rank < extra else 0)


def max_over_ranks(x: float, device=None) -> float:
    """MAX-reduce a scalar over the default process group (identity without one)."""
    if not (dist.is_available() and dist.is_initialized()) or dist.get_world_size() == 1:
        return float(x)
    t = torch.tensor([float(x)], dtype=torch.float64, device=device)
    dist.all_reduce(t, op=dist.ReduceOp.MAX)
    return float(t.item())


def aggregate_throughput(world: int, work_per_step: float, steps: int, max_total_s: float) -> float:
    """All ranks' work divided by the slowest rank's time."""
    return world * work_per_step * steps / max_total_s
