"""Host-side logic of bench.py's N > 1 run (replicas, one process per GPU):
the barrier, the max over ranks of the timed region and the whole-job rate,
checked with two `gloo` ranks on the CPU; and the reference arm's rule that
only rank 0 works."""
import os
import socket
import subprocess
import sys

import pytest
import torch.multiprocessing as mp

ROOT = os.path.dirname(os.path.dirname(os.path.abspath(__file__)))


def free_port():
    with socket.socket() as s:
        s.bind(("127.0.0.1", 0))
        return s.getsockname()[1]


def _rank(rank, world, port, out):
    import torch.distributed as dist
    sys.path.insert(0, ROOT)
    import bench
    os.environ.update(MASTER_ADDR="127.0.0.1", MASTER_PORT=str(port))
    dist.init_process_group("gloo", rank=rank, world_size=world)
    try:
        bench.rank_barrier(world)
        ms = 10.0 + 5.0 * rank  # rank 1 is the slower one
        m = bench.max_over_ranks_of(ms, world, "cpu")
        out.put((rank, m, bench.job_tflops(world, 1e12, m)))
        bench.rank_barrier(world)
    finally:
        dist.destroy_process_group()


def test_two_gloo_ranks_take_the_slowest_rank_and_sum_the_work():
    ctx = mp.get_context("spawn")
    q = ctx.Queue()
    port = free_port()
    procs = [ctx.Process(target=_rank, args=(r, 2, port, q)) for r in range(2)]
    for p in procs:
        p.start()
    for p in procs:
        p.join(120)
        assert p.exitcode == 0
    res = sorted(q.get(timeout=10) for _ in range(2))
    for rank, m, tflops in res:
        assert m == 15.0                      # both ranks see the slowest rank's time
        assert tflops == pytest.approx(2 * 1e12 / 0.015 / 1e12)  # the work of both ranks


def test_single_rank_needs_no_process_group():
    sys.path.insert(0, ROOT)
    import bench
    bench.rank_barrier(1)
    assert bench.max_over_ranks_of(3.5, 1, "cpu") == 3.5
    assert bench.job_tflops(1, 2e12, 1000.0) == pytest.approx(2.0)


def test_reference_arm_other_ranks_exit_without_work():
    env = dict(os.environ, RANK="1", WORLD_SIZE="2", LOCAL_RANK="1")
    r = subprocess.run([sys.executable, os.path.join(ROOT, "bench.py"), "--impl", "reference", "--gpus", "2",
                        "--steps", "1", "--warmup", "0"], env=env, capture_output=True, text=True, timeout=300)
    assert r.returncode == 0
    assert r.stdout.strip() == ""
