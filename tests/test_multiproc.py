"""The N > 1 path of bench.py on the CPU: independent replicas, one process
per rank, whole-job time = the slowest rank's (max over ranks through
torch.distributed), value = units of all ranks / that time.  Run with two
gloo ranks on 127.0.0.1; the reference arm prints from rank 0 only."""

import contextlib
import io
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


def _worker(rank, world, port, q):
    import torch.distributed as dist
    sys.path.insert(0, ROOT)
    os.environ.update(MASTER_ADDR="127.0.0.1", MASTER_PORT=str(port))
    dist.init_process_group("gloo", rank=rank, world_size=world)
    import bench
    # rank r "measured" (r + 1) ms for the timed region and (10 - r) ms end to end
    got = bench.max_over_ranks([rank + 1.0, 10.0 - rank], world)
    dist.barrier()
    q.put((rank, got))
    dist.destroy_process_group()


def test_max_over_ranks_two_gloo_ranks():
    world, port = 2, _free_port()
    ctx = mp.get_context("spawn")
    q = ctx.Queue()
    procs = [ctx.Process(target=_worker, args=(r, world, port, q)) for r in range(world)]
    for p in procs:
        p.start()
    out = dict(q.get(timeout=120) for _ in range(world))
    for p in procs:
        p.join(timeout=60)
        assert p.exitcode == 0
    # every rank sees the slowest rank's times
    assert out[0] == out[1] == [2.0, 10.0]


def test_single_rank_is_identity():
    sys.path.insert(0, ROOT)
    import bench
    assert bench.max_over_ranks([3.5, 1.25], 1) == [3.5, 1.25]


def test_reference_arm_prints_on_rank0_only(monkeypatch):
    """Under torchrun the reference arm runs and prints on rank 0; the other
    ranks exit without work."""
    sys.path.insert(0, ROOT)
    import bench
    monkeypatch.setenv("WORLD_SIZE", "2")
    monkeypatch.setenv("RANK", "1")
    monkeypatch.setattr(sys, "argv", ["bench.py", "--impl", "reference", "--gpus", "2"])
    called = []
    monkeypatch.setattr(bench, "run_reference", lambda args: called.append(1) or {})
    buf = io.StringIO()
    with contextlib.redirect_stdout(buf):
        bench.main()
    assert buf.getvalue() == "" and not called
    monkeypatch.setenv("RANK", "0")
    with contextlib.redirect_stdout(buf):
        bench.main()
    assert called == [1] and buf.getvalue().strip() == "{}"
