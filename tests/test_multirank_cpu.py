"""The N > 1 bench path on the host: two gloo ranks on CPU.

Each rank runs its own replica of the sublayer on its own batch (no data-path collective);
the only cross-rank steps are the barrier and the max of the step times, checked here."""
import os
import socket
import subprocess
import sys

import pytest
import torch.distributed as dist
import torch.multiprocessing as mp

ROOT = os.path.dirname(os.path.dirname(os.path.abspath(__file__)))


def _free_port():
    with socket.socket() as s:
        s.bind(("127.0.0.1", 0))
        return s.getsockname()[1]


def _rank_main(rank, world, port, times, out):
    sys.path.insert(0, ROOT)
    import bench

    dist.init_process_group("gloo", init_method=f"tcp://127.0.0.1:{port}", rank=rank,
                            world_size=world)
    try:
        dist.barrier()
        step_ms = bench.max_over_ranks(times[rank], dist)
        out[rank] = (step_ms, bench.whole_job_tflops(world, 2.0e12, step_ms))
    finally:
        dist.destroy_process_group()


def test_step_time_is_the_max_over_two_gloo_ranks():
    world, port = 2, _free_port()
    times = [1.25, 2.5]
    with mp.Manager() as m:
        out = m.dict()
        mp.spawn(_rank_main, args=(world, port, times, out), nprocs=world, join=True)
        res = dict(out)
    assert res[0][0] == res[1][0] == 2.5
    # two ranks, 2e12 FLOPs each per step, 2.5 ms per step -> 1600 TFLOP/s whole job
    assert res[0][1] == pytest.approx(1600.0)


def test_single_process_reduction_is_identity():
    sys.path.insert(0, ROOT)
    import bench

    assert bench.max_over_ranks(3.0, None) == 3.0
    assert bench.whole_job_tflops(1, 1e12, 1.0) == pytest.approx(1000.0)


def test_reference_arm_other_ranks_exit_without_output():
    env = dict(os.environ, RANK="1", WORLD_SIZE="2", LOCAL_RANK="1")
    r = subprocess.run([sys.executable, os.path.join(ROOT, "bench.py"), "--impl", "reference",
                        "--steps", "1", "--warmup", "3"], env=env, capture_output=True,
                       text=True, timeout=300)
    assert r.returncode == 0
    assert r.stdout.strip() == ""
