"""Host logic of bench.py's multi-process path, on CPU with gloo.

With N replicas (one process per GPU, no collective on the data path) the
timed region is bracketed by barriers, the step time is the slowest rank's,
and the whole-job value is that time divided by the N layers the job
finished.  Two gloo ranks on 127.0.0.1 check the reduction and the
aggregation; the reference arm's non-zero ranks exit without work."""
import io
import multiprocessing as mp
import os
import socket
import sys
from contextlib import redirect_stdout

import pytest

ROOT = os.path.dirname(os.path.dirname(os.path.abspath(__file__)))


def _free_port():
    with socket.socket() as s:
        s.bind(("127.0.0.1", 0))
        return s.getsockname()[1]


def _worker(rank, ws, port, q):
    os.environ.update(MASTER_ADDR="127.0.0.1", MASTER_PORT=str(port), RANK=str(rank), WORLD_SIZE=str(ws),
                      LOCAL_RANK=str(rank))
    sys.path.insert(0, ROOT)
    import torch
    import torch.distributed as dist
    dist.init_process_group("gloo", rank=rank, world_size=ws)
    import bench
    step_ms = 1.5 + rank  # rank 1 is the slow one
    dist.barrier()
    got = bench.max_over_ranks(step_ms, torch.device("cpu"))
    q.put((rank, got, bench.job_us_per_layer(got * 1e3, ws)))
    dist.barrier()
    dist.destroy_process_group()


def test_two_gloo_ranks_take_the_slowest_step():
    ws, port = 2, _free_port()
    ctx = mp.get_context("spawn")
    q = ctx.Queue()
    procs = [ctx.Process(target=_worker, args=(r, ws, port, q)) for r in range(ws)]
    for p in procs:
        p.start()
    for p in procs:
        p.join(120)
    assert all(p.exitcode == 0 for p in procs)
    res = sorted(q.get(timeout=5) for _ in range(ws))
    assert [r[1] for r in res] == [2.5, 2.5]
    assert [r[2] for r in res] == [1250.0, 1250.0]


def test_single_process_needs_no_process_group():
    sys.path.insert(0, ROOT)
    import torch
    import bench
    assert bench.max_over_ranks(3.25, torch.device("cpu")) == 3.25
    assert bench.job_us_per_layer(170.0, 1) == 170.0


def test_reference_arm_other_ranks_exit_without_work(monkeypatch):
    sys.path.insert(0, ROOT)
    import bench
    monkeypatch.setenv("RANK", "1")
    monkeypatch.setenv("WORLD_SIZE", "2")
    monkeypatch.setattr(sys, "argv", ["bench.py", "--impl", "reference", "--gpus", "2", "--steps", "1",
                                      "--warmup", "0"])
    out = io.StringIO()
    with redirect_stdout(out):
        bench.main()
    assert out.getvalue() == ""
