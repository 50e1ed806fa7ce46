"""The N > 1 host path of bench.py on CPU: N independent replicas whose job
time is the slowest rank's (max over ranks through torch.distributed) and
whose throughput is the sum of the ranks' work over that time.  Two gloo
ranks on 127.0.0.1 stand in for the GPUs; nothing here needs one."""
import os
import socket
import sys

import pytest
import torch.multiprocessing as mp

ROOT = os.path.dirname(os.path.dirname(os.path.abspath(__file__)))


def free_port():
    with socket.socket(socket.AF_INET, socket.SOCK_STREAM) as s:
        s.bind(("127.0.0.1", 0))
        return s.getsockname()[1]


def rank_main(rank, world, port, out):
    import torch.distributed as dist
    sys.path.insert(0, ROOT)
    import bench
    dist.init_process_group("gloo", init_method=f"tcp://127.0.0.1:{port}", rank=rank, world_size=world)
    try:
        ms_local = 2.0 + rank            # rank 1 is the slow one
        ms = bench.max_over_ranks(ms_local)
        fl = bench.flops(8, 16384, 7168, 2048)
        out[rank] = (ms, bench.replica_tflops(world, fl, ms))
    finally:
        dist.destroy_process_group()


def test_two_gloo_ranks_agree_on_slowest_time_and_job_throughput():
    world = 2
    ctx = mp.get_context("spawn")
    with ctx.Manager() as mgr:
        out = mgr.dict()
        mp.start_processes(rank_main, args=(world, free_port(), out), nprocs=world, join=True,
                           start_method="spawn")
        res = dict(out)
    sys.path.insert(0, ROOT)
    import bench
    fl = bench.flops(8, 16384, 7168, 2048)
    for r in range(world):
        ms, tf = res[r]
        assert ms == 3.0                                   # the slowest rank's time on every rank
        assert tf == pytest.approx(world * fl / 3.0e-3 / 1e12)


def test_single_process_is_its_own_max():
    sys.path.insert(0, ROOT)
    import bench
    assert bench.max_over_ranks(1.25) == 1.25
    assert bench.replica_tflops(1, 2e12, 1000.0) == pytest.approx(2.0)


def test_reference_arm_runs_on_rank_zero_only():
    sys.path.insert(0, ROOT)
    import bench

    class Args:
        steps, warmup = 1, 0

    # a non-zero rank leaves at once, without touching the oracle or a GPU
    assert bench.run_reference(Args(), rank=1, world=2) == 0
