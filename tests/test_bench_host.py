"""Host-side pieces of bench.py that need no GPU: the algorithmic work per
offset of each u8 method, and the rule that a stored DRAM-traffic figure is
reported only while the sources it was taken on are unchanged."""
import json
import os
import types

import numpy as np

import bench


def workload(ht, wt):
    return types.SimpleNamespace(tmpl=np.zeros((ht, wt), np.uint8))


def test_dp4a_per_offset_by_method():
    assert bench.dp4a_per_offset(workload(32, 32)) == 256             # box: N/4
    assert bench.dp4a_per_offset(workload(32, 32), "dp4a") == 768     # pages: 3N/4
    assert bench.dp4a_per_offset(workload(64, 64), "box") == 1024
    # a partial last word still costs one dp4a per row
    assert bench.dp4a_per_offset(workload(17, 31)) == 8 * 17
    assert bench.dp4a_per_offset(workload(5, 1), "dp4a") == 3 * 5


def test_traffic_reported_only_for_matching_sources(tmp_path, monkeypatch):
    src = tmp_path / "k.cu"
    src.write_text("kernel v1\n")
    prof = tmp_path / "profiles"
    prof.mkdir()
    table = {"k": {"source_sha256_16": bench.source_hash(str(src)),
                   "dram_bytes_per_launch": 1234}}
    (prof / "ncu_traffic.json").write_text(json.dumps(table))
    monkeypatch.setattr(bench, "ROOT", str(tmp_path))
    assert bench.traffic_for("k", [str(src)]) == 1234
    assert bench.traffic_for("other", [str(src)]) is None
    src.write_text("kernel v2\n")                  # the kernel changed since
    assert bench.traffic_for("k", [str(src)]) is None


def test_committed_traffic_record_names_its_sources():
    path = os.path.join(bench.ROOT, "profiles", "ncu_traffic.json")
    table = json.load(open(path))
    for key, e in table.items():
        assert e["dram_bytes_per_launch"] == e["dram_bytes_read"] + e["dram_bytes_write"]
        for s in e["sources"]:
            assert os.path.exists(os.path.join(bench.ROOT, s)), s
        assert "--clock-control none" in e["command"]
