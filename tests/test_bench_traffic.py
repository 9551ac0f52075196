"""Stored DRAM traffic for the roofline line: an entry of profiles/traffic.json
counts only while the sources it names are unchanged (host logic, no GPU)."""
import json
import os

import bench


def _entry(tmp_path, text):
    src = tmp_path / "kernel.cu"
    src.write_text(text)
    rel = os.path.relpath(src, bench.ROOT)
    return src, {"dram_bytes_per_launch": 123456, "digest": bench.source_digest([rel]),
                 "sources": [rel], "capture": "test"}


def test_entry_counts_while_its_sources_are_unchanged(tmp_path, monkeypatch):
    src, row = _entry(tmp_path, "__global__ void k() {}\n")
    f = tmp_path / "traffic.json"
    f.write_text(json.dumps({"ops": {"op a": row}}))
    monkeypatch.setattr(bench, "TRAFFIC_FILE", str(f))
    assert bench.stored_traffic("op a") == 123456
    assert bench.stored_traffic("op b") is None  # no entry
    src.write_text("__global__ void k() { /* changed */ }\n")
    assert bench.stored_traffic("op a") is None  # sources changed since the capture


def test_entry_without_sources_or_with_a_bad_file_is_ignored(tmp_path, monkeypatch):
    _, row = _entry(tmp_path, "x\n")
    row["sources"] = []
    f = tmp_path / "traffic.json"
    f.write_text(json.dumps({"ops": {"op a": row}}))
    monkeypatch.setattr(bench, "TRAFFIC_FILE", str(f))
    assert bench.stored_traffic("op a") is None
    f.write_text("not json")
    assert bench.stored_traffic("op a") is None
    monkeypatch.setattr(bench, "TRAFFIC_FILE", str(tmp_path / "missing.json"))
    assert bench.stored_traffic("op a") is None


def test_committed_traffic_file_is_well_formed():
    with open(bench.TRAFFIC_FILE) as fh:
        t = json.load(fh)
    # every ncu capture leaves the clocks alone: directly or through $M
    defs = {c.split("=", 1)[0]: c.split("=", 1)[1] for c in t["commands"] if "=" in c.split(" ")[0]}
    ncu = [c for c in t["commands"] if "ncu " in c]
    assert ncu
    for c in ncu:
        assert "--clock-control none" in c.replace("$M", defs.get("M", "")), c
    for name, row in t["ops"].items():
        assert int(row["dram_bytes_per_launch"]) > 0, name
        assert len(row["digest"]) == 16 and row["sources"], name
        for s in row["sources"]:
            assert os.path.exists(os.path.join(bench.ROOT, s)), (name, s)
