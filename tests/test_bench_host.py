"""Host-side logic of bench.py (no GPU): which DRAM traffic figure a bench
line may carry, the clock-record rejection rule, and the roofline peak."""
import json
import os

import bench


def _profile():
    with open(os.path.join(bench.ROOT, "profiles", "split_pass2_traffic.json")) as f:
        return json.load(f)


def test_traffic_only_for_the_captured_workload_and_rows():
    d = _profile()
    current = d["source_sha256"] == bench.kernel_source_hash()
    got = bench._traffic_from_profile(d["workload_key"], d["rows"])
    assert got == (d["dram_bytes_per_launch"] if current else None)
    assert bench._traffic_from_profile("wide", d["rows"]) is None
    assert bench._traffic_from_profile(d["workload_key"], d["rows"] // 8) is None


def test_traffic_is_null_once_the_kernel_sources_change(monkeypatch):
    d = _profile()
    monkeypatch.setattr(bench, "kernel_source_hash", lambda: "0" * 64)
    assert bench._traffic_from_profile(d["workload_key"], d["rows"]) is None


def test_traffic_figure_is_a_full_launch_at_least_the_read():
    # the capture is scaled to a full launch: at least every logit of the
    # step batch read once
    d = _profile()
    assert d["dram_bytes_per_launch"] >= d["rows"] * 262144 * 4


def test_clock_records_rejected_for_slowdowns_or_a_stuck_clock():
    ok = {"sm_mhz": 2070.0, "sm_max_mhz": 2070.0, "reasons": []}
    assert not bench._clocks_rejected(ok)
    assert not bench._clocks_rejected(dict(ok, reasons=["sw_power_cap"]))
    for r in ("hw_slowdown", "hw_thermal_slowdown", "sw_thermal_slowdown"):
        assert bench._clocks_rejected(dict(ok, reasons=[r]))
    assert bench._clocks_rejected(dict(ok, sm_mhz=900.0))


def test_peak_is_the_measured_copy_bandwidth_when_present(monkeypatch, tmp_path):
    monkeypatch.setattr(bench, "ROOT", str(tmp_path))
    assert bench._peak_hbm() == (bench.FALLBACK_HBM_GBS, "fallback")
    (tmp_path / "MEASURED_PEAKS.json").write_text(json.dumps({"hbm_gbs": 6123.5}))
    assert bench._peak_hbm() == (6123.5, "measured")
