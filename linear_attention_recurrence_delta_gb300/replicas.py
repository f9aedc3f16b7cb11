"""Data-parallel replicas of the gated delta rule across GPUs (one process per GPU).

Every (batch, head) recurrence is independent ("GDN & MLA Mechanism
Deep-Dive", Step 4: one state per head), so N GPUs run N replicas, each on a
batch of its own, with no collective on the data path (weak scaling).  The
only cross-rank steps are bookkeeping: each rank draws its own inputs, the
step time is the maximum over ranks, and the whole-job throughput counts the
tokens of every rank.  These helpers hold that bookkeeping so that it can be
exercised with any torch.distributed backend (gloo on CPU, nccl on GPUs).
"""
from __future__ import annotations

from . import inputs as I

RANK_SEED_STRIDE = 1000   # rank r draws its inputs with seed (workload seed + 1000 r)


def rank_workload(w: "I.Workload", rank: int, world: int) -> "I.Workload":
    """The workload replica `rank` runs: the same shapes with inputs of its own."""
    return w.with_(seed=w.seed + RANK_SEED_STRIDE * rank) if world > 1 else w


def max_over_ranks(value: float, dist=None, device: str = "cpu") -> float:
    """The maximum of `value` over all ranks of the default process group
    (identity without one)."""
    if dist is None or not dist.is_initialized() or dist.get_world_size() == 1:
        return float(value)
    import torch
    t = torch.tensor([float(value)], dtype=torch.float64, device=device)
    dist.all_reduce(t, op=dist.ReduceOp.MAX)
    return float(t.item())


def whole_job_tokens_per_s(tokens_per_rank: int, world: int, step_ms: float) -> float:
    """Tokens per second of the whole job: every rank's tokens over the slowest rank's step time."""
    return world * tokens_per_rank / (step_ms * 1e-3)
