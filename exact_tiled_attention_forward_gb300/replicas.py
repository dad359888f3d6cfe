"""Multi-GPU runs of the forward: independent replicas, one process per GPU.

The forward shards over (batch, head) with no exchange step ("Does the traffic
grow with the number of heads?": each head's K/V is read once, by the CTAs of
that head), so N GPUs run N independent replicas of the same workload and the
only cross-rank operations are host-side: a barrier around the timed region and
a max over ranks of the timed milliseconds. No collective touches the data path.
"""
from __future__ import annotations

import os


def replica_env() -> tuple[int, int, int]:
    """(rank, world size, local rank) as set by torch.distributed.run (1 process: 0, 1, 0)."""
    return (int(os.environ.get("RANK", "0")), int(os.environ.get("WORLD_SIZE", "1")),
            int(os.environ.get("LOCAL_RANK", "0")))


def slowest_rank_ms(ms: float, world: int, device=None) -> float:
    """The largest of every rank's timed milliseconds (all ranks call it; an
    initialised process group is required when world > 1, NCCL or gloo)."""
    if world <= 1:
        return ms
    import torch
    import torch.distributed as dist
    t = torch.tensor([ms], dtype=torch.float64, device=device)
    dist.all_reduce(t, op=dist.ReduceOp.MAX)
    return float(t.item())


def whole_job_rate(work_per_step: float, steps: int, slowest_ms: float, world: int) -> float:
    """Work per second of the whole job: every replica did `steps` steps of
    `work_per_step`, and the job took as long as its slowest rank."""
    return world * work_per_step * steps / (slowest_ms * 1e-3)
