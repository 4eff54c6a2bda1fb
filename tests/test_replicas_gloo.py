"""The N > 1 (one process per GPU) host path, run as two gloo ranks on the CPU:
the process-group setup, the barrier, the max of per-rank step times, the
whole-job throughput, the even split of a global batch, and the per-replica
data shards (own sequences, shared gamma, omega, phi)."""
import os
import socket

import pytest
import torch
import torch.multiprocessing as mp


def _free_port():
    with socket.socket(socket.AF_INET, socket.SOCK_STREAM) as s:
        s.bind(("127.0.0.1", 0))
        return s.getsockname()[1]


def _rank_main(rank, world, port, out_dir):
    os.environ.update(MASTER_ADDR="127.0.0.1", MASTER_PORT=str(port), RANK=str(rank),
                      WORLD_SIZE=str(world), LOCAL_RANK=str(rank))
    import torch.distributed as dist

    from constant_state_recurrence_gb300 import replicas
    from constant_state_recurrence_gb300 import workloads as W

    r = replicas.setup(use_cuda=False)
    assert (r.world, r.rank) == (world, rank)
    replicas.barrier(r)
    # slowest rank's time and whole-job throughput
    ms = 2.0 + rank  # rank 1 is the slow one
    ms_max = replicas.max_over_ranks(ms, r)
    assert ms_max == 2.0 + (world - 1)
    assert replicas.throughput(1000.0, r, ms_max) == world * 1000.0 / (ms_max * 1e-3)
    # even split of a global batch: disjoint, covering, sizes differ by at most 1
    for n in (0, 1, 7, 96):
        lo, hi = replicas.shard_range(n, r)
        got = [None] * world
        dist.all_gather_object(got, (lo, hi))
        assert got[0][0] == 0 and got[-1][1] == n
        assert all(got[i][1] == got[i + 1][0] for i in range(world - 1))
        sizes = [b - a for a, b in got]
        assert max(sizes) - min(sizes) <= 1
    # replica data: own sequences, shared parameters
    x = W.make(W.TINY, B=1, H=2, T=16, shard=rank)
    qs = [torch.empty_like(x["q"]) for _ in range(world)]
    dist.all_gather(qs, x["q"].contiguous())
    gs = [torch.empty_like(x["omega"]) for _ in range(world)]
    dist.all_gather(gs, x["omega"].contiguous())
    assert not torch.equal(qs[0], qs[1])
    assert torch.equal(gs[0], gs[1])
    if rank == 0:
        assert torch.equal(x["q"], W.make(W.TINY, B=1, H=2, T=16)["q"])  # shard 0 = the workload
    replicas.barrier(r)
    dist.destroy_process_group()
    open(os.path.join(out_dir, f"ok{rank}"), "w").close()


def test_two_gloo_ranks(tmp_path):
    world = 2
    mp.start_processes(_rank_main, args=(world, _free_port(), str(tmp_path)), nprocs=world,
                       join=True, start_method="spawn")
    for rank in range(world):
        assert (tmp_path / f"ok{rank}").exists()


def test_single_process_needs_no_group():
    from constant_state_recurrence_gb300 import replicas
    r = replicas.Replica(1, 0, 0)
    replicas.barrier(r)
    assert replicas.max_over_ranks(3.5, r) == 3.5
    assert replicas.shard_range(10, r) == (0, 10)
    assert replicas.throughput(100.0, r, 1.0) == pytest.approx(1e5)
