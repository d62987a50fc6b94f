"""Host logic of the multi-rank benchmark run (replicas, one per GPU) on CPU
ranks with the gloo backend: the job's time is the slowest rank's, and the
reference arm runs on rank 0 only."""
import io
import os
import socket
import sys
import types
from contextlib import redirect_stdout

import pytest
import torch
import torch.distributed as dist
import torch.multiprocessing as mp

ROOT = os.path.dirname(os.path.dirname(os.path.abspath(__file__)))


def _free_port():
    with socket.socket() as s:
        s.bind(("127.0.0.1", 0))
        return s.getsockname()[1]


def _worker(rank, world, port, q):
    os.environ.update(MASTER_ADDR="127.0.0.1", MASTER_PORT=str(port), RANK=str(rank),
                      WORLD_SIZE=str(world), LOCAL_RANK=str(rank))
    sys.path.insert(0, ROOT)
    dist.init_process_group("gloo", rank=rank, world_size=world)
    try:
        import bench
        q.put((rank, bench.reduce_max(10.0 + 3.0 * rank, torch.device("cpu")),
               bench.dist_env()))
    finally:
        dist.destroy_process_group()


def test_slowest_rank_sets_the_time():
    world = 2
    ctx = mp.get_context("spawn")
    q = ctx.Queue()
    port = _free_port()
    procs = [ctx.Process(target=_worker, args=(r, world, port, q)) for r in range(world)]
    for p in procs:
        p.start()
    out = sorted(q.get(timeout=120) for _ in range(world))
    for p in procs:
        p.join(timeout=60)
        assert p.exitcode == 0
    assert [v for _, v, _ in out] == [13.0, 13.0]
    assert [e for _, _, e in out] == [(2, 0, 0), (2, 1, 1)]


def test_single_process_needs_no_process_group():
    sys.path.insert(0, ROOT)
    import bench
    assert bench.reduce_max(4.5, torch.device("cpu")) == 4.5


def test_reference_arm_prints_only_on_rank_zero(monkeypatch):
    sys.path.insert(0, ROOT)
    import bench
    monkeypatch.setenv("RANK", "1")
    monkeypatch.setenv("WORLD_SIZE", "2")
    args = types.SimpleNamespace(config="tiny", ref_tokens=8, steps=1, warmup=0)
    buf = io.StringIO()
    with redirect_stdout(buf):
        assert bench.run_reference(args) is None
    assert buf.getvalue() == ""
