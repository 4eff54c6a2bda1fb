"""Data-parallel replicas of the attention path (one process per GPU).

Sequences are independent, so N GPUs run N independent replicas: each rank
processes its own batch of sequences (its own data shard, the same gamma,
omega, phi) and there is no exchange on the data path.  The only cross-rank
traffic is host-side bookkeeping: a barrier around the timed region and the
maximum of the per-rank step times, from which the whole-job throughput is
the tokens of all ranks divided by the slowest rank's time.

Host logic only (torch.distributed with NCCL on GPUs, gloo on CPU); no
computation of the method happens here.
"""
from __future__ import annotations

import os
from dataclasses import dataclass

import torch


@dataclass(frozen=True)
class Replica:
    world: int
    rank: int
    local: int


def setup(use_cuda: bool | None = None) -> Replica:
    """Read RANK / WORLD_SIZE / LOCAL_RANK and, for more than one rank, join
    the default process group (NCCL when CUDA is used, gloo otherwise)."""
    world = int(os.environ.get("WORLD_SIZE", "1"))
    rank = int(os.environ.get("RANK", "0"))
    local = int(os.environ.get("LOCAL_RANK", "0"))
    if use_cuda is None:
        use_cuda = torch.cuda.is_available()
    if world > 1:
        import torch.distributed as dist
        if not dist.is_initialized():
            if use_cuda:
                torch.cuda.set_device(local)
            dist.init_process_group("nccl" if use_cuda else "gloo")
    return Replica(world, rank, local)


def barrier(r: Replica) -> None:
    if r.world > 1:
        import torch.distributed as dist
        dist.barrier()


def max_over_ranks(x: float, r: Replica, device=None) -> float:
    """The largest value of x over all ranks (every rank gets it)."""
    if r.world == 1:
        return float(x)
    import torch.distributed as dist
    t = torch.tensor([float(x)], dtype=torch.float64, device=device)
    dist.all_reduce(t, op=dist.ReduceOp.MAX)
    return float(t.item())


def throughput(units_per_rank_step: float, r: Replica, ms_slowest: float) -> float:
    """Whole-job units per second: every rank's units over the slowest time."""
    return r.world * units_per_rank_step / (ms_slowest * 1e-3)


def shard_range(n: int, r: Replica) -> tuple[int, int]:
    """[start, stop) of rank r's share of n items split as evenly as possible
    (for callers that divide a fixed global batch instead of replicating)."""
    base, extra = divmod(int(n), r.world)
    start = r.rank * base + min(r.rank, extra)
    return start, start + base + (1 if r.rank < extra else 0)
