"""Host-side multi-rank logic around the shard step.

One process per GPU.  The shards are independent partitions of the parameter
index set ("DeepSpeed ZeRO Stages", sec. 2.1 Fact 1: the Adam update is
elementwise), so ranks step their own shards with no exchange on the data
path.  Small pieces of host logic cross ranks:

  * the skip decision: an overflow on any rank must skip the step on every
    rank, so the per-rank flags are ORed (an all-reduce of one int);
  * with global gradient clipping, the squared gradient norm: each rank adds
    its shard's sum of squares and the ranks sum them (one double);
  * timing: the slowest rank's time bounds the job.

All use ``torch.distributed`` (NCCL on GPUs, gloo on CPU).
"""
from __future__ import annotations

import torch
import torch.distributed as dist


def replica_shard(base_rank: int, rank: int, n_d: int) -> int:
    """Shard stepped by process ``rank`` when every process runs a replica of
    a workload whose device plays ``base_rank``: consecutive ranks take
    consecutive shards."""
    return (int(base_rank) + int(rank)) % int(n_d)


def agree_overflow(flag: int, device=None) -> int:
    """OR of the overflow flags of all ranks (1 if any rank overflowed)."""
    if not (dist.is_available() and dist.is_initialized()) or dist.get_world_size() == 1:
        return int(bool(flag))
    t = torch.tensor([int(bool(flag))], dtype=torch.int32, device=device)
    dist.all_reduce(t, op=dist.ReduceOp.MAX)
    return int(t.item())


def allreduce_sqnorm(sqnorm: torch.Tensor) -> torch.Tensor:
    """Sum the ranks' squared-gradient-norm accumulators in place (the one
    scalar exchange global gradient clipping adds to the step)."""
    if dist.is_available() and dist.is_initialized() and dist.get_world_size() > 1:
        dist.all_reduce(sqnorm, op=dist.ReduceOp.SUM)
    return sqnorm


def max_over_ranks(value: float, device=None) -> float:
    """Largest value over all ranks (the job's time is the slowest rank's)."""
    if not (dist.is_available() and dist.is_initialized()) or dist.get_world_size() == 1:
        return float(value)
    t = torch.tensor([float(value)], dtype=torch.float64, device=device)
    dist.all_reduce(t, op=dist.ReduceOp.MAX)
    return float(t.item())
