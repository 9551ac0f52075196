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


def test_gpus_flag_against_launcher_world_size():
    """--gpus N: one process runs N = 1 itself, starts N ranks when no launcher
    did, runs as one rank when the launcher's world size is N, and refuses a
    world size that disagrees with N."""
    sys.path.insert(0, ROOT)
    import bench

    assert bench.rank_plan(1, {}) == "run"
    assert bench.rank_plan(4, {}) == "spawn"
    assert bench.rank_plan(2, {"WORLD_SIZE": "2", "RANK": "1"}) == "run"
    assert bench.rank_plan(8, {"WORLD_SIZE": "8"}) == "run"
    assert bench.rank_plan(8, {"WORLD_SIZE": "1"}).startswith("error")
    assert bench.rank_plan(1, {"WORLD_SIZE": "2"}).startswith("error")
    assert bench.rank_plan(0, {}).startswith("error")


def test_gpus_flag_mismatch_exits_nonzero():
    import subprocess

    env = dict(os.environ, WORLD_SIZE="1", RANK="0", LOCAL_RANK="0")
    r = subprocess.run([sys.executable, os.path.join(ROOT, "bench.py"), "--gpus", "2", "--impl",
                        "reference"], env=env, capture_output=True, text=True, timeout=120)
    assert r.returncode != 0 and "WORLD_SIZE=1" in r.stderr


def test_gpus_flag_spawns_ranks_for_reference_arm(tmp_path):
    """Outside a launcher, --gpus 2 starts two ranks (torch.distributed.run on
    127.0.0.1); the reference arm then prints one line from rank 0."""
    import json
    import subprocess

    env = {k: v for k, v in os.environ.items() if k not in ("WORLD_SIZE", "RANK", "LOCAL_RANK")}
    r = subprocess.run([sys.executable, os.path.join(ROOT, "bench.py"), "--gpus", "2", "--impl",
                        "reference", "--workload", "int8_channel", "--steps", "1", "--warmup", "0"],
                       env=env, capture_output=True, text=True, timeout=600, cwd=str(tmp_path))
    assert r.returncode == 0, r.stderr[-2000:]
    lines = [json.loads(x) for x in r.stdout.splitlines() if x.startswith("{")]
    assert len(lines) == 1 and lines[0]["impl"] == "reference" and lines[0]["n_gpus"] == 2
