"""The bench's recorded DRAM traffic: a figure taken from one ncu capture is
reported only while the kernel's sources are unchanged since the capture
(comments and blank space aside), and the committed records are well formed."""

import json
import os

import bench


def _tree(tmp_path, code):
    csrc = tmp_path / "query_aware_sparse_gb300" / "csrc"
    csrc.mkdir(parents=True)
    (csrc / "k.cuh").write_text(code)
    (tmp_path / "profiles").mkdir()
    return csrc / "k.cuh"


def test_source_hash_ignores_comments_not_code(tmp_path, monkeypatch):
    monkeypatch.setattr(bench, "ROOT", str(tmp_path))
    f = _tree(tmp_path, "int f(int x) {\n  return x + 1;  // one\n}\n")
    h0 = bench.source_hash("k.cuh")
    f.write_text("/* a new block\n comment */\nint f(int x) {\n\n    return x + 1;   // two\n}\n")
    assert bench.source_hash("k.cuh") == h0
    f.write_text("int f(int x) {\n  return x + 2;  // one\n}\n")
    assert bench.source_hash("k.cuh") != h0


def test_traffic_only_while_sources_match(tmp_path, monkeypatch):
    monkeypatch.setattr(bench, "ROOT", str(tmp_path))
    f = _tree(tmp_path, "int g() { return 3; }\n")
    rec = {"kern@wl": {"dram_bytes_per_launch": 1234, "sources": ["k.cuh"],
                       "source_hash": bench.source_hash("k.cuh")}}
    (tmp_path / "profiles" / "ncu_traffic.json").write_text(json.dumps(rec))
    assert bench.ncu_traffic("kern", "wl") == 1234
    assert bench.ncu_traffic("kern", "other") is None
    f.write_text("int g() { return 4; }\n")                 # the kernel changed
    assert bench.ncu_traffic("kern", "wl") is None
    os.remove(f)                                            # a recorded source is gone
    assert bench.ncu_traffic("kern", "wl") is None


def test_committed_records_are_well_formed():
    p = os.path.join(bench.ROOT, "profiles", "ncu_traffic.json")
    with open(p) as fh:
        rec = json.load(fh)
    assert rec
    for key, e in rec.items():
        kernel, workload = key.split("@")
        assert kernel and workload
        assert isinstance(e["dram_bytes_per_launch"], int) and e["dram_bytes_per_launch"] > 0
        assert e["sources"] and len(e["source_hash"]) == 16
        assert "--clock-control none" in e["capture"] and " -c 1" in e["capture"]
        for s in e["sources"]:
            assert os.path.exists(os.path.join(bench.ROOT, "query_aware_sparse_gb300", "csrc", s))
