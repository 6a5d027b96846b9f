"""The multi-rank path of bench.py on CPU ranks (gloo, world size 2).

The benchmark runs one replica per GPU (no data-path collective): each rank
times its own steps, the ranks meet at barriers around the timed region, and
rank 0 reports the slowest rank's time.  These tests drive that logic with two
CPU processes over gloo; nothing here needs a GPU.
"""
import os
import socket
import sys

import pytest

torch = pytest.importorskip("torch")
import torch.multiprocessing as mp  # noqa: E402

ROOT = os.path.dirname(os.path.dirname(os.path.abspath(__file__)))


def _free_port():
    with socket.socket() as s:
        s.bind(("127.0.0.1", 0))
        return s.getsockname()[1]


def _rank_main(rank, world, port, out):
    os.environ.update({"WORLD_SIZE": str(world), "RANK": str(rank), "LOCAL_RANK": str(rank),
                       "MASTER_ADDR": "127.0.0.1", "MASTER_PORT": str(port)})
    sys.path.insert(0, ROOT)
    import bench
    d = bench.Dist(world)
    d.init("gloo")
    d.barrier()
    # each rank's "time": the maximum over ranks is what rank 0 reports
    got = d.max(10.0 + 5.0 * rank)
    d.barrier()
    d.close()
    out.put((rank, d.world, got))


def test_two_gloo_ranks_agree_on_the_slowest_time():
    ctx = mp.get_context("spawn")
    out = ctx.Queue()
    port = _free_port()
    procs = [ctx.Process(target=_rank_main, args=(r, 2, port, out)) for r in range(2)]
    for p in procs:
        p.start()
    for p in procs:
        p.join(timeout=120)
    assert all(p.exitcode == 0 for p in procs)
    res = sorted(out.get(timeout=5) for _ in range(2))
    assert res == [(0, 2, 15.0), (1, 2, 15.0)]


def test_reference_arm_other_ranks_exit_without_work(monkeypatch, capsys):
    """Under torchrun only rank 0 runs and prints the reference line."""
    sys.path.insert(0, ROOT)
    import bench
    monkeypatch.setenv("WORLD_SIZE", "2")
    monkeypatch.setenv("RANK", "1")

    class Args:
        gpus, steps, warmup = 2, 1, 0

    assert bench.run_reference(Args()) is None
    assert capsys.readouterr().out == ""


def test_single_rank_needs_no_process_group(monkeypatch):
    sys.path.insert(0, ROOT)
    import bench
    monkeypatch.delenv("WORLD_SIZE", raising=False)
    monkeypatch.delenv("RANK", raising=False)
    d = bench.Dist(1)
    d.init("gloo")
    d.barrier()
    assert d.max(3.5) == 3.5
    d.close()
