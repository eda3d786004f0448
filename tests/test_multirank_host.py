"""The N > 1 bench path on CPU: two gloo ranks (127.0.0.1) check the rank
reductions bench.py uses -- the whole-job work is the sum of every rank's own
work, the time is the slowest rank's -- and the barrier; and that the
reference arm runs on rank 0 only."""
import os
import socket

import pytest
import torch
import torch.distributed as dist
import torch.multiprocessing as mp


def _free_port() -> int:
    with socket.socket(socket.AF_INET, socket.SOCK_STREAM) as s:
        s.bind(("127.0.0.1", 0))
        return s.getsockname()[1]


def _worker(rank, world, port, results):
    os.environ["MASTER_ADDR"] = "127.0.0.1"
    os.environ["MASTER_PORT"] = str(port)
    dist.init_process_group("gloo", rank=rank, world_size=world)
    try:
        import bench
        cpu = torch.device("cpu")
        bench.barrier(world)
        mx = bench.max_over_ranks(world, cpu, [1.0 + rank, 10.0 - rank])
        sm = bench.sum_over_ranks(world, cpu, [100.0 * (rank + 1), 0.5])
        # a rank that finishes later than the other must set the job time
        results[rank] = (mx, sm)
    finally:
        dist.destroy_process_group()


def test_two_gloo_ranks_reduce_like_the_bench():
    world = 2
    port = _free_port()
    ctx = mp.get_context("spawn")     # no fork of a process that already runs threads
    with ctx.Manager() as m:
        results = m.dict()
        procs = [ctx.Process(target=_worker, args=(r, world, port, results)) for r in range(world)]
        for p in procs:
            p.start()
        for p in procs:
            p.join(timeout=120)
            assert p.exitcode == 0
        got = dict(results)
    for r in range(world):
        mx, sm = got[r]
        assert mx == [2.0, 10.0]           # element-wise maximum
        assert sm == [300.0, 1.0]          # element-wise sum


def test_single_rank_reductions_are_identity():
    import bench
    cpu = torch.device("cpu")
    assert bench.max_over_ranks(1, cpu, [3.0, 4.0]) == [3.0, 4.0]
    assert bench.sum_over_ranks(1, cpu, [3.0, 4.0]) == [3.0, 4.0]


def test_reference_arm_does_no_work_off_rank_zero(capsys):
    import argparse
    import bench
    args = argparse.Namespace(warmup=3, steps=2, ref_rows=16)
    bench.run_reference(args, rank=1, world=2)
    assert capsys.readouterr().out == ""
