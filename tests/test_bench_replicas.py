"""The bench's multi-process (replicas) logic on CPU: two gloo ranks, no GPU.

bench.py runs N independent replicas under torchrun (the path has no collective of its own): the timing is
the maximum over ranks and the whole-job value counts every rank's work. The reference arm runs on rank 0
only."""
import os
import socket
import sys

import pytest

ROOT = os.path.dirname(os.path.dirname(os.path.abspath(__file__)))
sys.path.insert(0, ROOT)

torch = pytest.importorskip("torch")


def _free_port():
    s = socket.socket()
    s.bind(("127.0.0.1", 0))
    port = s.getsockname()[1]
    s.close()
    return port


def _rank_main(rank, world, port, q):
    os.environ.update({"RANK": str(rank), "WORLD_SIZE": str(world), "LOCAL_RANK": str(rank),
                       "MASTER_ADDR": "127.0.0.1", "MASTER_PORT": str(port)})
    import argparse
    import bench
    args = argparse.Namespace(impl="reference")
    w, r, local, pg = bench.dist_setup(args)
    seconds = [0.5, 2.0][rank]                       # rank 1 is the slow one
    value = bench.whole_job(pg, 100.0, seconds, w)    # 100 units per rank
    slowest = bench.max_over_ranks(pg, seconds)
    q.put((r, w, local, value, slowest))
    pg.destroy_process_group()


def test_two_gloo_replicas():
    import torch.multiprocessing as mp
    ctx = mp.get_context("spawn")
    q = ctx.Queue()
    port = _free_port()
    procs = [ctx.Process(target=_rank_main, args=(r, 2, port, q)) for r in range(2)]
    for p in procs:
        p.start()
    out = sorted(q.get(timeout=120) for _ in range(2))
    for p in procs:
        p.join(timeout=60)
        assert p.exitcode == 0
    assert [o[0] for o in out] == [0, 1]
    for r, w, local, value, slowest in out:
        assert w == 2 and local == r
        assert slowest == 2.0                         # max over ranks
        assert value == pytest.approx(200.0 / 2.0)    # both ranks' units over the slowest time


def test_reference_arm_other_ranks_exit(monkeypatch, capsys):
    import argparse
    import bench
    monkeypatch.setenv("RANK", "1")
    monkeypatch.setenv("WORLD_SIZE", "2")
    called = []
    monkeypatch.setattr(bench, "oracle_step_sample", lambda: called.append(1))
    bench.run_reference(argparse.Namespace(steps=1, warmup=3))
    assert not called and capsys.readouterr().out == ""


def test_single_process_whole_job():
    import bench
    assert bench.whole_job(None, 50.0, 0.25, 1) == pytest.approx(200.0)
