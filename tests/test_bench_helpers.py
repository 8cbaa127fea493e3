"""bench.py's link between a committed ncu capture and a bench line: the DRAM traffic of a
capture is reported only for its own workload and only while the kernel sources are the
ones it was taken on."""
import json
import os
import sys

ROOT = os.path.dirname(os.path.dirname(os.path.abspath(__file__)))
sys.path.insert(0, ROOT)

import bench  # noqa: E402


def _write(tmp_path, captures):
    d = tmp_path / "profiles"
    d.mkdir()
    (d / "traffic.json").write_text(json.dumps({"captures": captures}))


def test_traffic_is_matched_by_workload_and_source(tmp_path, monkeypatch):
    monkeypatch.setattr(bench, "ROOT", str(tmp_path))
    monkeypatch.setattr(bench, "kernel_source_hash", lambda: "abc")
    _write(tmp_path, [
        {"workload": "penalties_bias", "kernel_source_sha": "abc", "dram_bytes_per_launch": 11},
        {"workload": "all_greedy", "kernel_source_sha": "abc", "dram_bytes_per_launch": 22},
        {"workload": "grammar", "kernel_source_sha": "old", "dram_bytes_per_launch": 33},
    ])
    assert bench.traffic_from_profile("penalties_bias") == 11
    assert bench.traffic_from_profile("all_greedy") == 22
    assert bench.traffic_from_profile("grammar") is None  # taken on other sources
    assert bench.traffic_from_profile("decode_mix") is None  # no capture


def test_single_capture_file_and_missing_file(tmp_path, monkeypatch):
    monkeypatch.setattr(bench, "ROOT", str(tmp_path))
    monkeypatch.setattr(bench, "kernel_source_hash", lambda: "abc")
    assert bench.traffic_from_profile("penalties_bias") is None
    d = tmp_path / "profiles"
    d.mkdir()
    (d / "traffic.json").write_text(json.dumps(
        {"workload": "penalties_bias", "kernel_source_sha": "abc", "dram_bytes_per_launch": 7}))
    assert bench.traffic_from_profile("penalties_bias") == 7


def test_committed_captures_name_their_kernels():
    with open(os.path.join(ROOT, "profiles", "traffic.json")) as f:
        d = json.load(f)
    for c in d["captures"]:
        assert c["dram_bytes_per_launch"] == c["dram_bytes_read_per_launch"] + c["dram_bytes_write_per_launch"]
        assert "--clock-control none" in c["source"] and c["kernel"]
