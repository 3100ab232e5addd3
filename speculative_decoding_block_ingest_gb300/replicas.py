"""Replicas across GPUs (one process per GPU).

Drafting rounds of different sequences are independent (no exchange between
them), so several GPUs run as replicas: every rank holds the whole drafter
and its own sequences, with no collective on the data path.  The job's time
over a timed region is the slowest rank's, and its throughput the ranks'
total work over that time.
"""
from __future__ import annotations


def slowest_ms(ms: float, dist=None, device: str = "cpu") -> float:
    """Maximum of each rank's elapsed milliseconds (identity on one rank).

    ``dist`` is ``torch.distributed`` with an initialised process group, or
    None; ``device`` is where the group's backend reduces (the rank's GPU for
    NCCL, "cpu" for gloo)."""
    if dist is None:
        return float(ms)
    import torch
    t = torch.tensor([float(ms)], dtype=torch.float64, device=device)
    dist.all_reduce(t, op=dist.ReduceOp.MAX)
    return float(t.item())


def job_throughput(world: int, units_per_rank: int, ms: float) -> float:
    """Units per second of the whole job: every rank did ``units_per_rank``
    in at most ``ms`` milliseconds (weak scaling)."""
    return world * units_per_rank / (ms / 1e3)
