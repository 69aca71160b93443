"""The multi-replica path of bench.py on CPU (gloo, world size 2): the step
time reported is the slowest rank's, and the job throughput counts every
replica's work over that time."""
import os
import sys

import pytest
import torch
import torch.distributed as dist
import torch.multiprocessing as mp

ROOT = os.path.dirname(os.path.dirname(os.path.abspath(__file__)))


def _worker(rank, world, port, out):
    sys.path.insert(0, ROOT)
    os.environ.update(MASTER_ADDR="127.0.0.1", MASTER_PORT=str(port))
    dist.init_process_group("gloo", rank=rank, world_size=world)
    import bench
    times = [10.0 + 5.0 * rank, 20.0 - 3.0 * rank]        # rank 1 slower in the first, faster in the second
    got = bench.max_over_ranks(times, world)
    dist.barrier()
    out[rank] = got + [bench.job_throughput(3.0e12, got[0], world)]
    dist.destroy_process_group()


def test_max_over_ranks_and_job_throughput_gloo():
    world = 2
    mgr = mp.Manager()
    out = mgr.dict()
    port = 29500 + (os.getpid() % 1000)
    mp.spawn(_worker, args=(world, port, out), nprocs=world, join=True)
    for r in range(world):
        ms, e2e_ms, tflops = out[r]
        assert ms == 15.0 and e2e_ms == 20.0               # each entry's maximum over the ranks
        assert tflops == pytest.approx(2 * 3.0e12 / 15e-3 / 1e12)


def test_single_rank_is_identity():
    sys.path.insert(0, ROOT)
    import bench
    assert bench.max_over_ranks([1.5, 2.5], 1) == [1.5, 2.5]
    assert bench.job_throughput(1e12, 1.0, 1) == pytest.approx(1000.0)
