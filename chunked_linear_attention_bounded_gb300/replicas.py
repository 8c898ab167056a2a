"""Host logic of the multi-GPU run: one process per GPU, each running its
own replica of the workload.

The (document, head) units of a step are independent (nothing in the forward
or the backward reads across documents or heads), so ranks share no data:
each rank draws its own batch (the workload's seed shifted by the rank),
runs it on its own GPU, and the only collectives are the ones that measure
(a barrier around the timed region and the maximum of the per-rank times).
Job throughput is the tokens of all ranks divided by the slowest rank's time.
"""
from __future__ import annotations

import dataclasses
import os

import torch
import torch.distributed as dist

from .inputs import Workload

# seeds of different ranks stay apart from the other workloads' seeds
RANK_SEED_STRIDE = 100


@dataclasses.dataclass(frozen=True)
class RankEnv:
    rank: int
    world: int
    local: int


def rank_env() -> RankEnv:
    """Rank, world size and local rank from the launcher's environment."""
    return RankEnv(int(os.environ.get("RANK", "0")), int(os.environ.get("WORLD_SIZE", "1")),
                   int(os.environ.get("LOCAL_RANK", "0")))


def rank_workload(w: Workload, rank: int) -> Workload:
    """The batch a rank processes: same shapes, its own seed."""
    return dataclasses.replace(w, seed=w.seed + RANK_SEED_STRIDE * rank) if rank else w


def barrier(world: int) -> None:
    if world > 1:
        dist.barrier()


def max_over_ranks(x: float, world: int, device=None) -> float:
    """Largest value of x over all ranks (x itself when world == 1)."""
    if world <= 1:
        return float(x)
    t = torch.tensor([float(x)], dtype=torch.float64, device=device)
    dist.all_reduce(t, op=dist.ReduceOp.MAX)
    return float(t.item())


def job_throughput(tokens_per_rank: int, world: int, ms_max: float) -> float:
    """Tokens per second of the whole job: every rank's tokens over the
    slowest rank's step time."""
    return world * tokens_per_rank / (ms_max / 1000.0)
