"""The multi-rank path of bench.py, on CPU.

Under torchrun each GPU runs one rank, a replica of the workload; the ranks only
meet at the barrier around the timed region and in the max of their times.  These
tests run that same code (bench.Ranks) as two gloo ranks on the CPU, check the
whole-job rate, and check that the reference arm's second rank exits without work.
"""

import os
import socket
import subprocess
import sys

import pytest

ROOT = os.path.dirname(os.path.dirname(os.path.abspath(__file__)))


def _free_port() -> int:
    with socket.socket(socket.AF_INET, socket.SOCK_STREAM) as s:
        s.bind(("127.0.0.1", 0))
        return s.getsockname()[1]


def _rank(rank: int, world: int, port: int, q) -> None:
    os.environ.update(MASTER_ADDR="127.0.0.1", MASTER_PORT=str(port), RANK=str(rank),
                      WORLD_SIZE=str(world), LOCAL_RANK=str(rank))
    import torch

    import bench

    r = bench.Ranks("gloo", torch.device("cpu"))
    r.barrier()
    # each rank "times" a different elapsed; every rank must see the slowest
    slowest = r.max_over_ranks(10.0 + 5.0 * rank)
    r.barrier()
    q.put((r.rank, r.world, slowest))
    r.close()


def test_two_gloo_ranks_share_the_slowest_time():
    import torch.multiprocessing as mp

    ctx = mp.get_context("spawn")
    q = ctx.Queue()
    port = _free_port()
    procs = [ctx.Process(target=_rank, args=(r, 2, port, q)) for r in range(2)]
    for p in procs:
        p.start()
    got = sorted(q.get(timeout=120) for _ in procs)
    for p in procs:
        p.join(timeout=60)
        assert p.exitcode == 0
    assert got == [(0, 2, 15.0), (1, 2, 15.0)]


def test_single_rank_needs_no_process_group(monkeypatch):
    for k in ("RANK", "WORLD_SIZE", "LOCAL_RANK"):
        monkeypatch.delenv(k, raising=False)
    import bench

    r = bench.Ranks("gloo")
    assert (r.rank, r.world) == (0, 1)
    r.barrier()
    assert r.max_over_ranks(3.5) == 3.5
    r.close()


def test_whole_job_rate_counts_every_rank():
    import bench

    # two replicas of 1e6 values each, the slower finishing in 2 ms: 1e9 values/s
    assert bench.whole_job_rate(2, 1e6, 2.0) == pytest.approx(1e9)
    assert bench.whole_job_rate(1, 1e6, 2.0) == pytest.approx(5e8)


def test_reference_arm_second_rank_exits_without_work():
    env = dict(os.environ, RANK="1", WORLD_SIZE="2", LOCAL_RANK="1",
               MASTER_ADDR="127.0.0.1", MASTER_PORT=str(_free_port()))
    res = subprocess.run([sys.executable, os.path.join(ROOT, "bench.py"), "--impl", "reference",
                          "--gpus", "2", "--steps", "1", "--warmup", "1"],
                         cwd=ROOT, env=env, capture_output=True, text=True, timeout=300)
    assert res.returncode == 0, res.stderr
    assert res.stdout.strip() == ""
