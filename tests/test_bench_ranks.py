"""Multi-rank host logic of bench.py on CPU: two gloo ranks agree on the max
step time, and the reference arm does its work on rank 0 only."""
import io
import os
import socket
import sys
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


def _rank_main(rank, world, port, q):
    sys.path.insert(0, ROOT)
    import bench

    os.environ.update(MASTER_ADDR="127.0.0.1", MASTER_PORT=str(port))
    dist.init_process_group("gloo", rank=rank, world_size=world)
    try:
        got = bench.max_over_ranks(1.5 + rank * 2.25, dist, torch.device("cpu"))
        q.put((rank, got))
    finally:
        dist.destroy_process_group()


def test_max_over_ranks_gloo_world2():
    ctx = mp.get_context("spawn")
    q = ctx.Queue()
    port = _free_port()
    procs = [ctx.Process(target=_rank_main, args=(r, 2, port, q)) for r in range(2)]
    for p in procs:
        p.start()
    for p in procs:
        p.join(120)
        assert p.exitcode == 0
    res = dict(q.get(timeout=10) for _ in range(2))
    assert res == {0: 3.75, 1: 3.75}


def test_single_rank_max_is_identity():
    sys.path.insert(0, ROOT)
    import bench

    assert bench.max_over_ranks(2.5, None, torch.device("cpu")) == 2.5


def test_reference_arm_only_on_rank_zero(monkeypatch):
    sys.path.insert(0, ROOT)
    import bench

    monkeypatch.setenv("RANK", "1")
    args = type("A", (), {"workload": "int8_channel", "steps": 1, "warmup": 0, "gpus": 2})()
    buf = io.StringIO()
    with redirect_stdout(buf):
        bench.reference_arm(args)
    assert buf.getvalue() == ""


def test_reference_arm_line_on_rank_zero(monkeypatch):
    import json

    sys.path.insert(0, ROOT)
    import bench

    monkeypatch.setenv("RANK", "0")
    args = type("A", (), {"workload": "int8_channel", "steps": 2, "warmup": 1, "gpus": 1})()
    buf = io.StringIO()
    with redirect_stdout(buf):
        bench.reference_arm(args)
    line = json.loads(buf.getvalue())
    assert line["impl"] == "reference" and line["value"] > 0 and line["unit"] == "GB/s"
    assert line["cpu_baseline"]["kind"] == "oracle" and line["e2e"]["h2d_bytes_per_step"] == 0
