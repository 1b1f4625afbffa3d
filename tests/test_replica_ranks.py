"""bench.py's multi-rank arithmetic (replicas, one per GPU) on two CPU ranks
over gloo: the job time is the slowest rank's, the job rate world x the
slowest rank's rate, and the tokens/s value all ranks' tokens over the job
time."""

import os
import socket

import torch
import torch.distributed as dist
import torch.multiprocessing as mp

ROOT = os.path.dirname(os.path.dirname(os.path.abspath(__file__)))


def _free_port():
    with socket.socket() as s:
        s.bind(("127.0.0.1", 0))
        return s.getsockname()[1]


def _rank(rank, world, port, out):
    import sys
    sys.path.insert(0, ROOT)
    import bench
    os.environ.update(MASTER_ADDR="127.0.0.1", MASTER_PORT=str(port))
    dist.init_process_group("gloo", rank=rank, world_size=world)
    ms = [1.5, 2.0][rank]                 # rank 1 is the slower replica
    rate = [900.0, 700.0][rank]
    job_ms = bench.slowest_rank(dist, ms, "cpu")
    job = bench.job_rate(dist, rate, world, "cpu")
    dist.barrier()
    out[rank] = (job_ms, job)
    dist.destroy_process_group()


def test_two_replicas_slowest_rank_sets_the_job():
    world = 2
    with mp.Manager() as m:
        out = m.dict()
        mp.start_processes(_rank, args=(world, _free_port(), out), nprocs=world,
                           start_method="spawn")
        res = dict(out)
    for r in range(world):
        job_ms, job = res[r]
        assert job_ms == 2.0                  # every rank reports the slowest time
        assert job == 2 * 700.0               # world x the slowest rank's rate
    T = 64                                    # tokens per rank
    assert T * world / (res[0][0] * 1e-3) == 64000.0


def test_single_process_is_the_identity():
    import sys
    sys.path.insert(0, ROOT)
    import bench
    assert bench.slowest_rank(None, 1.25, "cpu") == 1.25
    assert bench.job_rate(None, 10.0, 1, "cpu") == 10.0
