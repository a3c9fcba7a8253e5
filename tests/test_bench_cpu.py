"""Host logic of bench.py that needs no GPU: the committed DRAM-traffic lookup
(used only while every source a stage depends on is unchanged since the
counters were taken) and the shape of profiles/traffic.json."""
import hashlib
import json
import os

import bench

ROOT = os.path.dirname(os.path.dirname(os.path.abspath(__file__)))


def _sha16(path):
    with open(os.path.join(ROOT, path), "rb") as f:
        return hashlib.sha256(f.read()).hexdigest()[:16]


def test_committed_traffic_entries_name_existing_sources():
    with open(os.path.join(ROOT, "profiles", "traffic.json")) as f:
        d = json.load(f)
    assert d, "no traffic entries"
    for key, e in d.items():
        stage, workload = key.split("@")
        assert e["bytes_per_launch"] > 0
        assert e["sources"], key
        for src in e["sources"]:
            assert os.path.exists(os.path.join(ROOT, src)), src
        assert os.path.exists(os.path.join(ROOT, e["from"])), e["from"]


def test_committed_traffic_follows_the_source_hashes(tmp_path, monkeypatch):
    src = tmp_path / "k.cu"
    src.write_text("kernel v1\n")
    prof = tmp_path / "profiles"
    prof.mkdir()
    h = hashlib.sha256(src.read_bytes()).hexdigest()[:16]
    (prof / "traffic.json").write_text(json.dumps(
        {"stage@wl": {"bytes_per_launch": 1234, "sources": {"k.cu": h}, "from": "x"}}))
    monkeypatch.setattr(bench, "ROOT", str(tmp_path))
    assert bench.committed_traffic("stage", "wl") == 1234
    assert bench.committed_traffic("stage", "other") is None
    src.write_text("kernel v2\n")  # the kernel changed since the counters were taken
    assert bench.committed_traffic("stage", "wl") is None
