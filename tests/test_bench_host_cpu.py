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


def test_roofline_arithmetic_of_the_long_context_job():
    """summarize() against the per-unit algorithmic figures, worked by hand for the
    32-layer 96K job (256 units, 1024 query heads, K = 10, L = 150, d = 128, bf16):
    attention 2·d·2 + 4 = 516 B per list entry plus d·(2 + 4) B per query head and step;
    CSR build 4 B per (token, table) plus 2·(2^K + 1) B of offsets per 32768-token
    segment; hashing GEMM 2·d·K·L FLOP per key."""
    import workloads as WL
    wl = WL.WORKLOADS[2]
    pk = {"hbm_gbs": 6000.0, "bf16_tflops_sustained": 1500.0, "source": "test"}
    prof = {"attend": (64, 10.0), "csr_build": (1, 6.0), "hash_keys_tc": (1, 8.0), "match_csr": (64, 5.0)}
    entries, sampled, walked = 100_000_000, 95_000_000, 1_000_000_000
    out = bench.summarize(None, wl, prof, pk, entries, sampled, walked)
    k = out["kernels"]
    attend = entries * 516 + 64 * 1024 * 128 * 6
    assert k["attend"]["algorithmic_per_launch"] == attend / 64
    assert k["attend"]["achieved"] == attend / 10e-3 / 1e9
    assert k["csr_build"]["algorithmic_per_launch"] == 256 * 150 * (98300 * 4 + 3 * 1025 * 2) == 15_335_040_000
    assert k["hash_keys_tc"]["algorithmic_per_launch"] == 2 * 128 * 1500 * 256 * 98304
    assert k["hash_keys_tc"]["unit"] == "TFLOP/s"
    assert k["match_csr"]["algorithmic_per_launch"] == (walked * 2 + 64 * 1024 * 150 * (4 * 3 + 2) + entries * 4) / 64
    r = out["roofline"]
    assert r["kernel"] == "attend" and r["bound"] == "hbm" and r["peak"] == 6000.0
    assert r["frac"] == k["attend"]["achieved"] / 6000.0
    assert abs(sum(v["share"] for v in k.values()) - 1.0) < 1e-12
    assert out["build_ms"] == 14.0 and out["us_per_decode_step"] == 1e3 * 15.0 / 64


def test_end_to_end_groups_split_layers_then_sequences():
    """The end-to-end run issues the job in groups whose slices of K/V, W, queries and
    outputs are whole layers (or, with one layer, whole sequences)."""
    import workloads as WL
    assert bench.e2e_groups(WL.WORKLOADS[2]) == ("layers", 4)      # 32 layers: groups of 8
    assert bench.e2e_groups(WL.WORKLOADS[5]) == ("layers", 4)      # 4 layers: one each
    assert bench.e2e_groups(WL.WORKLOADS[3]) == ("batch", 4)       # one layer, 16 sequences
    assert bench.e2e_groups(WL.WORKLOADS[4]) == ("batch", 4)       # one layer, 4 sequences
    assert bench.e2e_groups(WL.WORKLOADS[1]) == (None, 1)          # one layer, one sequence
    assert bench.e2e_groups(WL.WORKLOADS[2].replace(layers=6)) == ("layers", 2)
