"""The multi-rank host logic of bench.py (replicas: one process per GPU) on
CPU with the gloo backend, world size 2: rendezvous on 127.0.0.1, barrier,
and the max-over-ranks reduction the whole-job timing uses."""
import os
import socket
import sys

import pytest

ROOT = os.path.dirname(os.path.dirname(os.path.abspath(__file__)))


def _free_port():
    s = socket.socket()
    s.bind(("127.0.0.1", 0))
    port = s.getsockname()[1]
    s.close()
    return port


def _worker(rank, world, port, q):
    os.environ.update(RANK=str(rank), WORLD_SIZE=str(world), LOCAL_RANK=str(rank),
                      MASTER_ADDR="127.0.0.1", MASTER_PORT=str(port))
    sys.path.insert(0, ROOT)
    import bench
    import torch.distributed as dist
    r, w, local = bench.dist_setup("gloo")
    bench.barrier(w)
    mx = bench.max_over_ranks(10.0 + r, w, "cpu")
    q.put((r, w, local, mx))
    dist.destroy_process_group()


def test_two_rank_max_and_barrier():
    torch = pytest.importorskip("torch")
    import torch.multiprocessing as mp
    ctx = mp.get_context("spawn")
    q = ctx.Queue()
    port = _free_port()
    procs = [ctx.Process(target=_worker, args=(r, 2, port, q)) for r in range(2)]
    for p in procs:
        p.start()
    for p in procs:
        p.join(120)
        assert p.exitcode == 0
    got = sorted(q.get(timeout=5) for _ in range(2))
    assert [g[0] for g in got] == [0, 1]
    assert all(g[1] == 2 for g in got)
    assert all(g[3] == 11.0 for g in got)  # every rank sees the slowest rank's time


def test_reference_arm_other_ranks_exit_quietly(monkeypatch, capsys):
    """Under torchrun only rank 0 runs the oracle arm; the others print nothing."""
    sys.path.insert(0, ROOT)
    import bench
    monkeypatch.setattr(bench, "dist_setup", lambda backend: (1, 2, 1))

    class A:
        steps, warmup, gpus, ref_rows_total = 3, 3, 2, 100
    assert bench.run_reference(A()) == 0
    assert capsys.readouterr().out == ""
