"""Host side of running the benchmark as N independent replicas (one process
per GPU): the slowest rank's times and the whole-job throughput.

The attention path itself has no exchange step (its units - (batch, head)
pairs, packed sequences, decode entries - are independent), so the only
collectives are these timing reductions.  They take any process group, so the
logic runs under gloo on the CPU as well as under NCCL.
"""
from __future__ import annotations

from typing import List, Optional, Sequence


def max_over_ranks(values: Sequence[float], device: str = "cpu", group=None) -> List[float]:
    """Element-wise maximum of ``values`` over the ranks of the default (or
    given) process group; the values themselves when not distributed."""
    import torch
    import torch.distributed as dist

    if not (dist.is_available() and dist.is_initialized()) or dist.get_world_size(group) == 1:
        return [float(v) for v in values]
    t = torch.tensor([float(v) for v in values], dtype=torch.float64, device=device)
    dist.all_reduce(t, op=dist.ReduceOp.MAX, group=group)
    return [float(v) for v in t.tolist()]


def whole_job_rate(world: int, units_per_rank_step: float, ms_per_step: float) -> float:
    """Units all ranks processed per second when each of ``world`` replicas
    processes ``units_per_rank_step`` units per step and the slowest takes
    ``ms_per_step``."""
    if world < 1 or ms_per_step <= 0:
        raise ValueError("world >= 1 and a positive step time are required")
    return world * units_per_rank_step / (ms_per_step * 1e-3)


def rescale_to_slowest(value: float, own_ms: float, slowest_ms: float, world: int) -> float:
    """A per-rank rate measured over own_ms, restated for the whole job at the
    slowest rank's time."""
    return world * value * own_ms / slowest_ms


def barrier(group: Optional[object] = None) -> None:
    import torch.distributed as dist

    if dist.is_available() and dist.is_initialized() and dist.get_world_size(group) > 1:
        dist.barrier(group=group)
