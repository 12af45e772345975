"""The multi-GPU path of bench.py on CPU: two gloo ranks stand in for two GPUs.

The layer has no exchange step on one GPU, so N GPUs run N independent
replicas. The job's time is the slowest rank's (all ranks must finish), and its
throughput counts every rank's tokens.
"""
import os
import socket

import pytest
import torch.distributed as dist
import torch.multiprocessing as mp


def _free_port():
    with socket.socket() as s:
        s.bind(("127.0.0.1", 0))
        return s.getsockname()[1]


def _rank(rank, world, port, out):
    os.environ.update(MASTER_ADDR="127.0.0.1", MASTER_PORT=str(port), RANK=str(rank),
                      WORLD_SIZE=str(world))
    dist.init_process_group("gloo", rank=rank, world_size=world)
    import bench
    ms = [10.0, 12.5][rank]
    worst = bench.max_over_ranks(ms, world)
    out[rank] = (worst, bench.job_tokens_per_s(world, 64, 100, worst))
    dist.barrier()
    dist.destroy_process_group()


@pytest.mark.timeout(120)
def test_two_replicas_take_the_slowest_rank_and_count_all_tokens():
    world = 2
    with mp.Manager() as mgr:
        out = mgr.dict()
        mp.spawn(_rank, args=(world, _free_port(), out), nprocs=world, join=True)
        res = dict(out)
    for rank in range(world):
        worst, value = res[rank]
        assert worst == 12.5
        assert value == pytest.approx(2 * 64 * 100 / 12.5e-3)
