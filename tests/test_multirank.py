"""The benchmark's multi-rank logic on CPU: two gloo ranks (no GPU needed).

Sequences are independent, so N GPUs run N replicas with no data-path
collective; the only cross-rank steps are the barrier and the max over ranks of
the timed region.  Here two processes join a gloo group over 127.0.0.1 and
check the slowest-rank time and the whole-job rate, and the reference arm's
rank 1 exits without work.
"""
import os
import socket
import subprocess
import sys

import pytest
import torch.multiprocessing as mp

ROOT = os.path.dirname(os.path.dirname(os.path.abspath(__file__)))


def _free_port():
    with socket.socket() as s:
        s.bind(("127.0.0.1", 0))
        return s.getsockname()[1]


def _rank_main(rank, world, port, out):
    os.environ.update(MASTER_ADDR="127.0.0.1", MASTER_PORT=str(port), RANK=str(rank), WORLD_SIZE=str(world))
    sys.path.insert(0, ROOT)
    import torch.distributed as dist

    import bench

    dist.init_process_group("gloo", rank=rank, world_size=world)
    my_ms = 10.0 * (rank + 1)  # rank 1 is the slow one
    dist.barrier()
    worst = bench.max_over_ranks(my_ms, dist, "cpu")
    rate = bench.whole_job_rate(16, 100, world, worst)
    out.put((rank, worst, rate))
    dist.destroy_process_group()


def test_two_gloo_ranks_report_the_slowest_rank_and_the_whole_job_rate():
    ctx = mp.get_context("spawn")
    q = ctx.Queue()
    port = _free_port()
    procs = [ctx.Process(target=_rank_main, args=(r, 2, port, q)) for r in range(2)]
    for p in procs:
        p.start()
    for p in procs:
        p.join(120)
        assert p.exitcode == 0
    got = sorted(q.get(timeout=10) for _ in range(2))
    for rank, worst, rate in got:
        assert worst == pytest.approx(20.0)
        assert rate == pytest.approx(2 * 16 * 100 / 0.020)


def test_reference_arm_rank1_exits_without_work():
    env = dict(os.environ, RANK="1", WORLD_SIZE="2", LOCAL_RANK="1")
    res = subprocess.run([sys.executable, os.path.join(ROOT, "bench.py"), "--impl", "reference", "--gpus", "2",
                          "--steps", "3", "--warmup", "3"], env=env, capture_output=True, text=True, timeout=300)
    assert res.returncode == 0
    assert res.stdout.strip() == ""


def test_max_over_ranks_is_identity_without_a_group():
    sys.path.insert(0, ROOT)
    import bench

    assert bench.max_over_ranks(3.5, None, "cpu") == 3.5
    assert bench.whole_job_rate(16, 10, 1, 2.0) == pytest.approx(16 * 10 / 0.002)
