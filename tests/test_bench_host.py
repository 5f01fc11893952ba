"""Host-side logic of bench.py (no GPU): which DRAM traffic figure a bench
line may carry, the clock-record rejection rule, the roofline peak, and the
parity comparison of GPU rows with the oracle's."""
import json
import os

import numpy as np

import bench


def _write_profile(root, workload="step", rows=2048, sha="a" * 64, nbytes=3_300_000_000):
    os.makedirs(os.path.join(root, "profiles"), exist_ok=True)
    d = {"workload_key": workload, "rows": rows, "source_sha256": sha, "dram_bytes_per_call": nbytes}
    with open(os.path.join(root, bench.TRAFFIC_PROFILE), "w") as f:
        json.dump(d, f)
    return d


def test_traffic_only_for_the_captured_workload_and_rows(monkeypatch, tmp_path):
    d = _write_profile(str(tmp_path))
    monkeypatch.setattr(bench, "ROOT", str(tmp_path))
    monkeypatch.setattr(bench, "kernel_source_hash", lambda: d["source_sha256"])
    assert bench._traffic_from_profile("step", 2048) == d["dram_bytes_per_call"]
    assert bench._traffic_from_profile("wide", 2048) is None
    assert bench._traffic_from_profile("step", 256) is None


def test_traffic_is_null_once_the_kernel_sources_change(monkeypatch, tmp_path):
    _write_profile(str(tmp_path))
    monkeypatch.setattr(bench, "ROOT", str(tmp_path))
    monkeypatch.setattr(bench, "kernel_source_hash", lambda: "0" * 64)
    assert bench._traffic_from_profile("step", 2048) is None


def test_traffic_is_null_without_a_capture(monkeypatch, tmp_path):
    monkeypatch.setattr(bench, "ROOT", str(tmp_path))
    assert bench._traffic_from_profile("step", 2048) is None


def test_committed_traffic_figure_covers_the_algorithmic_bytes():
    # a committed capture of the whole call: at least every logit of the
    # batch read once and every probability written once
    path = os.path.join(bench.ROOT, bench.TRAFFIC_PROFILE)
    if not os.path.exists(path):
        return
    with open(path) as f:
        d = json.load(f)
    assert d["dram_bytes_per_call"] >= d["rows"] * 262144 * 6 * 0.99


def test_source_hash_covers_both_row_kernels():
    h1 = bench.kernel_source_hash()
    assert len(h1) == 64 and h1 == bench.kernel_source_hash()


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


def test_parity_counts_near_ties_apart_from_mismatches():
    # three rows: one exact, one sample mismatch inside the near-tie band,
    # one outside it; ids and logprobs of two top-k rows
    ref = {"argmax": np.array([1, 2, 3]), "sample": np.array([4, 5, 6]),
           "sample_gap": np.array([1.0, 1e-7, 0.5]), "sample_best": np.array([3.0, 3.0, 3.0]),
           "entropy": np.array([0.5, 0.25, 1.0]), "probs": np.array([[100, 200]], np.uint16)}
    gpu = {"argmax": np.array([1, 2, 3]), "sample": np.array([[4, 7, 8]]),
           "entropy": np.array([0.5, 0.25 + 2e-5, 1.0], np.float32),
           "probs": np.array([[101, 200]], np.uint16),
           "ids": np.array([[1, 2], [3, 4]], np.int32), "lps": np.array([[-0.5, -1.0], [-2.0, -3.0]], np.float32)}
    topk = (np.array([[1, 2], [3, 5]], np.int32), np.array([[-0.5, -1.0], [-2.0, -3.0]]))
    c = bench._compare(gpu, [ref], topk, 1)
    assert c["argmax_mismatch"] == 0
    assert c["sample_near_ties"] == 1 and c["sample_mismatch_outside_near_ties"] == 1
    assert c["probs_max_code_diff"] == 1
    assert c["topk_id_mismatch_rows"] == 1 and c["logprob_within_tolerance"]
    assert abs(c["entropy_max_abs_err"] - 2e-5) < 1e-6
