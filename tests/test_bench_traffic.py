"""bench.py's DRAM-traffic records (profiles/traffic.json), on CPU: a record
counts only while the hash of the kernel sources it was taken on matches the
current sources -- the GEMM's sources for a GEMM record (per launch), the
small-M LoRA kernels' for a LoRA-stage record (per forward) -- and the two
kinds are kept apart."""

import json
import os
import sys

ROOT = os.path.dirname(os.path.dirname(os.path.abspath(__file__)))
sys.path.insert(0, ROOT)

import bench  # noqa: E402


def _write(tmp_path, entries):
    path = tmp_path / "traffic.json"
    path.write_text(json.dumps({"entries": entries}))
    return str(path)


def test_records_follow_their_sources(tmp_path, monkeypatch):
    g = bench.source_hash(bench.GEMM_SOURCES)
    lo = bench.source_hash(bench.LORA_SOURCES)
    assert g == bench.gemm_source_hash() and g != lo
    monkeypatch.setattr(bench, "TRAFFIC_PATH", _write(tmp_path, [
        {"workload": "w", "dram_bytes_per_launch": 111, "source_hash": g},
        {"workload": "w", "stage": "lora", "dram_bytes_per_forward": 222, "source_hash": lo},
        {"workload": "stale", "dram_bytes_per_launch": 333, "source_hash": "0" * 16},
        {"workload": "crossed", "stage": "lora", "dram_bytes_per_forward": 444, "source_hash": g},
    ]))
    assert bench.ncu_traffic("w") == 111
    assert bench.ncu_traffic("w", "lora") == 222
    assert bench.ncu_traffic("stale") is None          # taken on other sources
    assert bench.ncu_traffic("crossed", "lora") is None  # a LoRA record keyed by the GEMM's sources
    assert bench.ncu_traffic("absent") is None


def test_missing_or_broken_file(tmp_path, monkeypatch):
    monkeypatch.setattr(bench, "TRAFFIC_PATH", str(tmp_path / "none.json"))
    assert bench.ncu_traffic("prefill_sgmv") is None
    bad = tmp_path / "bad.json"
    bad.write_text("{not json")
    monkeypatch.setattr(bench, "TRAFFIC_PATH", str(bad))
    assert bench.ncu_traffic("prefill_sgmv", "lora") is None
