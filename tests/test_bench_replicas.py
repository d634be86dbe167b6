"""bench.py's replica aggregation on two CPU ranks over gloo: every rank sees the
slowest rank's time, the job rate counts all ranks' units over that time, the barrier
returns, and the reference arm does its work on rank 0 only."""
import os
import socket
import sys

import pytest
import torch.multiprocessing as mp

ROOT = os.path.dirname(os.path.dirname(os.path.abspath(__file__)))


def _free_port():
    with socket.socket() as s:
        s.bind(("127.0.0.1", 0))
        return s.getsockname()[1]


def _rank(rank, world, port, q):
    os.environ.update(RANK=str(rank), WORLD_SIZE=str(world), LOCAL_RANK=str(rank), MASTER_ADDR="127.0.0.1",
                      MASTER_PORT=str(port), MK_BENCH_BACKEND="gloo")
    sys.path.insert(0, ROOT)
    import bench
    import torch.distributed as dist
    r, w, local = bench.dist_setup(world)
    secs = [2.0, 5.0][r]                        # rank 1 is the slow one
    rate, t = bench.job_rate(100, secs, w)
    bench.barrier(w)
    q.put((r, w, local, rate, t))
    dist.destroy_process_group()


def test_two_rank_aggregation():
    ctx = mp.get_context("spawn")
    q = ctx.Queue()
    port = _free_port()
    procs = [ctx.Process(target=_rank, args=(r, 2, port, q)) for r in range(2)]
    for p in procs:
        p.start()
    out = sorted(q.get(timeout=120) for _ in procs)
    for p in procs:
        p.join(timeout=60)
        assert p.exitcode == 0
    for r, (rank, world, local, rate, t) in enumerate(out):
        assert (rank, world, local) == (r, 2, r)
        assert t == 5.0                          # the max over ranks
        assert rate == pytest.approx(2 * 100 / 5.0)


def test_single_rank_is_plain():
    sys.path.insert(0, ROOT)
    import bench
    assert bench.dist_setup(1) == (0, 1, 0)
    assert bench.job_rate(64, 2.0, 1) == (32.0, 2.0)


def test_reference_arm_rank1_exits_without_work(monkeypatch, capsys):
    sys.path.insert(0, ROOT)
    import bench
    monkeypatch.setenv("RANK", "1")
    monkeypatch.setenv("WORLD_SIZE", "2")

    class A:
        steps, warmup, gpus = 4, 3, 2
    assert bench.run_reference(A()) == 0
    assert capsys.readouterr().out == ""
