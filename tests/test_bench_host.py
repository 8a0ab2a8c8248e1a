"""Host logic of bench.py, no GPU: the stored DRAM traffic records are used
only while the sources they were measured on are unchanged, and the byte
accounting of the find-rho and gridding rooflines adds up as documented."""

import json
import os
import sys

ROOT = os.path.dirname(os.path.dirname(os.path.abspath(__file__)))
sys.path.insert(0, ROOT)

import bench  # noqa: E402


def test_traffic_records_follow_their_sources(tmp_path, monkeypatch):
    rec = {"grid_tc:w:fast": {"source_hash": bench.gather_source_hash("grid_tc"),
                              "dram_bytes_per_launch": 123},
           "toeplitz:w:product": {"source_hash": "0" * 16, "dram_bytes_per_launch": 456}}
    prof = tmp_path / "profiles"
    prof.mkdir()
    (prof / "traffic.json").write_text(json.dumps(rec))
    # the hashes come from the repository's sources, the records from the
    # temporary copy
    hashes = {k: bench.gather_source_hash(k) for k in ("grid_tc", "toeplitz")}
    monkeypatch.setattr(bench, "gather_source_hash", lambda kind="grid_tc": hashes[kind])
    monkeypatch.setattr(bench, "ROOT", str(tmp_path))
    assert bench.profiled_traffic("grid_tc", "fast", "w") == 123
    assert bench.profiled_traffic("toeplitz", "product", "w") is None   # stale hash
    assert bench.profiled_traffic("grid_tc", "accurate", "w") is None   # no record


def test_committed_traffic_records_are_well_formed():
    """Every record in profiles/traffic.json names a known kernel kind, a
    16-hex-digit source hash, its command and positive byte counts that add
    up (whether it is current is the bench's check: a stale record reports
    no traffic)."""
    with open(os.path.join(ROOT, "profiles", "traffic.json")) as fh:
        rec = json.load(fh)
    for key, entry in rec.items():
        if key.startswith("_"):
            continue
        kind, workload, variant = key.split(":")
        assert kind in bench.TRAFFIC_SOURCES, key
        assert len(entry["source_hash"]) == 16 and int(entry["source_hash"], 16) >= 0
        assert entry["dram_bytes_per_launch"] == (entry["dram_read_bytes"] +
                                                  entry["dram_write_bytes"]) > 0
        assert entry["command"].startswith("ncu ") and "--clock-control none" in entry["command"]


def test_find_rho_and_gridding_byte_accounting():
    # five stages: x forward 8 + 16, y forward 16 + 32, z 32 + 32 + 32,
    # y inverse 32 + 16, x inverse 16 + 8 + 8
    assert bench.TOEPLITZ_BYTES_PER_VOXEL == 248
    assert bench.TOEPLITZ_COMPULSORY_BYTES_PER_VOXEL == 48
    assert bench.CG_EXTRA_BYTES_PER_VOXEL == 64
    assert bench.GRIDDING_BYTES_PER_SAMPLE == 28
    assert bench.GRIDDING_BYTES_PER_VOXEL == 72


def test_general_gather_roofline_follows_the_kernel():
    """The SFU/FP32 bound of the general gather charges each unit what the
    kernel gives it: every sin/cos on the SFU (fast), every one as the 13-op
    polynomial on the FP32 pipe (accurate), or a share of them there."""
    ops = bench.algo_ops("fhd", "fast")
    assert (ops["mufu"], ops["fp32"]) == (2.0, 7.0)
    ops = bench.algo_ops("fhd", "accurate")
    assert (ops["mufu"], ops["fp32"]) == (0.0, 7.0 + 13.0)
    ops = bench.algo_ops("q", "fast", 0.25)
    assert ops["mufu"] == 1.5 and abs(ops["fp32"] - (5.0 + 14.0 * 0.25)) < 1e-12
    per, unit, _, _ = bench.peak_per_sm_clk("fhd", None, "fast")
    assert (per, unit) == (8.0, "mufu")                  # 16 sin/cos per SM per clock
    per, unit, _, _ = bench.peak_per_sm_clk("fhd", None, "accurate")
    assert (per, unit) == (128.0 / 20.0, "fp32")
    per, unit, _, _ = bench.peak_per_sm_clk("q", None, "fast", 0.25)
    assert abs(per - 16.0 / 1.5) < 1e-12 and unit == "mufu"
    # batched, 8 coils: FP32-bound, 3/8 + 4 operations per pair-coil
    per, unit, _, _ = bench.peak_per_sm_clk("fhd_batched", None, "fast")
    assert abs(per - 128.0 / 4.375) < 1e-12 and unit == "fp32"
    # batched on the tensor cores: the multiply-accumulate leaves the SM's
    # pipes; 2 sin/cos (fast) or 3 + 13 FP32 operations (accurate) per pair,
    # shared by 8 coils
    per, unit, _, _ = bench.peak_per_sm_clk("fhd_batched_tc", None, "fast")
    assert (per, unit) == (64.0, "mufu")
    per, unit, _, _ = bench.peak_per_sm_clk("fhd_batched_tc", None, "accurate")
    assert (per, unit) == (64.0, "fp32")
