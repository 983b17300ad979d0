"""Host-side bookkeeping of bench.py that needs no GPU: the roofline's DRAM traffic
comes from committed ncu counters only while the kernel's source is unchanged."""
import hashlib
import json
import os
import sys

ROOT = os.path.dirname(os.path.dirname(os.path.abspath(__file__)))
sys.path.insert(0, ROOT)

import bench  # noqa: E402


def _write(tmp_path, sha):
    rec = {"kernels": {"attend": {"dram_bytes_per_algorithmic_unit": 0.5, "source_sha256": sha}}}
    p = tmp_path / "traffic.json"
    p.write_text(json.dumps(rec))
    return str(p)


def test_traffic_scales_the_recorded_ratio_while_the_source_matches(tmp_path, monkeypatch):
    src = os.path.join(ROOT, "lsh_sampled_sparse_centered_gb300", "csrc", bench.KERNEL_SOURCE["attend"])
    sha = hashlib.sha256(open(src, "rb").read()).hexdigest()
    monkeypatch.setattr(bench, "TRAFFIC_FILE", _write(tmp_path, sha))
    assert bench.measured_traffic("attend", 1000.0) == 500.0


def test_traffic_is_null_once_the_source_changed_or_nothing_is_recorded(tmp_path, monkeypatch):
    monkeypatch.setattr(bench, "TRAFFIC_FILE", _write(tmp_path, "0" * 64))
    assert bench.measured_traffic("attend", 1000.0) is None
    assert bench.measured_traffic("match_csr", 1000.0) is None
    monkeypatch.setattr(bench, "TRAFFIC_FILE", str(tmp_path / "missing.json"))
    assert bench.measured_traffic("attend", 1000.0) is None


def test_committed_counters_cover_the_dominant_kernels():
    rec = json.load(open(bench.TRAFFIC_FILE))["kernels"]
    for k in ("attend", "match_csr", "hash_keys_tc", "csr_build"):
        assert k in rec and rec[k]["dram_bytes_per_algorithmic_unit"] > 0
