"""The N > 1 host logic of bench.py on the CPU, with two gloo ranks.

The GPU arm runs one replica per GPU.  The job's step time is each timing's
maximum over ranks (max_over_ranks), and its throughput is the work of all
ranks over that time (job_tops, weak scaling).  Each rank here plays a
replica with its own timings; both ranks must agree on the slowest values."""
import os
import socket
import sys

import pytest
import torch
import torch.distributed as dist
import torch.multiprocessing as mp

ROOT = os.path.dirname(os.path.dirname(os.path.abspath(__file__)))


def free_port():
    with socket.socket() as s:
        s.bind(("127.0.0.1", 0))
        return s.getsockname()[1]


def worker(rank, world, port, out):
    sys.path.insert(0, ROOT)
    import bench
    dist.init_process_group("gloo", init_method=f"tcp://127.0.0.1:{port}", rank=rank, world_size=world)
    try:
        # rank r: step 10 + r ms, GEMM 8 - r ms, eager 9 ms
        mine = [10.0 + rank, 8.0 - rank, 9.0]
        got = bench.max_over_ranks(mine, world, "cpu")
        dist.barrier()
        out[rank] = got + [bench.job_tops(world, 2.0e12, got[0])]
    finally:
        dist.destroy_process_group()


def test_max_over_ranks_and_job_value_two_ranks():
    world = 2
    with mp.Manager() as m:
        out = m.dict()
        mp.start_processes(worker, args=(world, free_port(), out), nprocs=world, start_method="spawn")
        res = dict(out)
    assert set(res) == {0, 1}
    for r in (0, 1):
        step, gemm, eager, tops = res[r]
        assert (step, gemm, eager) == (11.0, 8.0, 9.0)        # the slowest rank, per timing
        assert tops == pytest.approx(2 * 2.0e12 / 11e-3 / 1e12)   # both ranks' work over the slowest time


def test_single_rank_is_the_identity():
    sys.path.insert(0, ROOT)
    import bench
    assert bench.max_over_ranks([1.5, 2], 1, "cpu") == [1.5, 2.0]
    assert bench.job_tops(1, 1.0e12, 1.0) == pytest.approx(1000.0)
