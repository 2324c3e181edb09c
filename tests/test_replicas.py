"""Several GPUs run independent replicas: nothing is exchanged but the
timing. bench.py reduces each rank's elapsed time with a max over ranks and
prints one line from rank 0; the reference arm runs on rank 0 alone. Two
CPU ranks over gloo (127.0.0.1) check the reduction and the barrier."""

import os
import socket
import sys

import torch.multiprocessing as mp

ROOT = os.path.dirname(os.path.dirname(os.path.abspath(__file__)))


def _free_port() -> int:
    s = socket.socket()
    s.bind(("127.0.0.1", 0))
    port = s.getsockname()[1]
    s.close()
    return port


def _rank_main(rank, world, port, q):
    os.environ.update(MASTER_ADDR="127.0.0.1", MASTER_PORT=str(port), RANK=str(rank), WORLD_SIZE=str(world),
                      LOCAL_RANK=str(rank))
    sys.path.insert(0, ROOT)
    import bench
    r, w, local, dist = bench._dist()
    slowest = bench._max_over_ranks(dist, 1.5 + rank)   # rank 1 took longer
    bench._barrier(dist)
    q.put((r, w, local, slowest))
    dist.destroy_process_group()


def test_max_over_two_gloo_ranks():
    ctx = mp.get_context("spawn")
    q = ctx.Queue()
    port = _free_port()
    procs = [ctx.Process(target=_rank_main, args=(r, 2, port, q)) for r in range(2)]
    for p in procs:
        p.start()
    got = sorted(q.get(timeout=120) for _ in procs)
    for p in procs:
        p.join(60)
        assert p.exitcode == 0
    assert got == [(0, 2, 0, 2.5), (1, 2, 1, 2.5)]


def test_single_process_needs_no_process_group(monkeypatch):
    monkeypatch.delenv("WORLD_SIZE", raising=False)
    sys.path.insert(0, ROOT)
    import bench
    assert bench._dist() == (0, 1, 0, None)
    assert bench._max_over_ranks(None, 3.25) == 3.25


def test_reference_arm_other_ranks_do_no_work(monkeypatch, capsys):
    """A rank other than 0 returns before building weights or running the oracle."""
    sys.path.insert(0, ROOT)
    import bench
    monkeypatch.setenv("RANK", "1")
    monkeypatch.setattr(bench, "_weights", lambda device: (_ for _ in ()).throw(AssertionError("work on rank 1")))

    class Args:
        steps, warmup = 1, 0
    bench.run_reference(Args())
    assert capsys.readouterr().out == ""
