"""Host logic of bench.py on CPU: the peak file's parsing and fallback, the
clock samples kept and summarised (only those inside the timed region, with
the throttle reasons seen), and the committed traffic figures, reported only
while the kernel source still has the hash they were taken with."""

import hashlib
import json
import os

import pytest

import bench


def test_peaks_read_nested_keys_and_fall_back(tmp_path, monkeypatch):
    monkeypatch.setattr(bench, "ROOT", str(tmp_path))
    p = bench.peaks()
    assert p["source"] == "fallback" and p["bf16_tflops"] == 1900.0 and p["hbm_gbs"] == 6800.0
    (tmp_path / "MEASURED_PEAKS.json").write_text(json.dumps(
        {"gpu": "GB300", "copy": {"hbm_gbs": 6790.5}, "gemm": {"bf16_tflops": 1939.6, "bf16_tflops_sustained": 1734.7}}))
    p = bench.peaks()
    assert p == {"hbm_gbs": 6790.5, "bf16_tflops": 1939.6, "bf16_tflops_sustained": 1734.7, "source": "measured"}
    (tmp_path / "MEASURED_PEAKS.json").write_text(json.dumps({"hbm_gbs": 7000.0, "bf16_tflops": 2000.0}))
    p = bench.peaks()  # no sustained figure: the burst one stands in
    assert p["bf16_tflops_sustained"] == 2000.0 and p["source"] == "measured"
    (tmp_path / "MEASURED_PEAKS.json").write_text("{not json")
    assert bench.peaks()["source"] == "fallback"


def test_clock_summary_keeps_only_the_timed_region():
    c = bench.ClockSampler(0)
    c.lines = [
        (1.0, "0, 1000, 2070, 500.0, 0x0, Not Active, Not Active, Not Active, Not Active"),  # before
        (2.0, "0, 2070, 2070, 1300.0, 0x4, Not Active, Not Active, Not Active, Active"),
        (2.5, "0, 2055, 2070, 1350.0, 0x4, Not Active, Not Active, Not Active, Active"),
        (2.7, "[N/A] garbled line"),
        (3.0, "0, 2070, 2070, 1290.0, 0x0, Not Active, Not Active, Not Active, Not Active"),
        (4.0, "0, 800, 2070, 300.0, 0x0, Active, Not Active, Not Active, Not Active"),  # after
    ]
    c.t0, c.t1 = 1.5, 3.5
    s = c.summary()
    assert s == {"sm_mhz": 2070.0, "sm_max_mhz": 2070.0, "reasons": ["sw_power_cap"], "samples": 3}
    c.t0, c.t1 = 3.6, 4.5  # a region with a hardware slowdown
    assert c.summary()["reasons"] == ["hw_slowdown"]
    c.t0, c.t1 = 10.0, 11.0  # no samples inside
    assert c.summary() is None


def test_traffic_is_reported_only_for_the_captured_source(tmp_path, monkeypatch):
    monkeypatch.setattr(bench, "ROOT", str(tmp_path))
    src = tmp_path / "k.cu"
    src.write_text("// kernel v1\n")
    (tmp_path / "profiles").mkdir()
    entry = {"kernel": "k", "dram_read_bytes": 100, "dram_write_bytes": 23, "source": "k.cu",
             "sha256_16": hashlib.sha256(src.read_bytes()).hexdigest()[:16],
             "workload": "captured on a smaller case, scaled by blocks"}
    (tmp_path / "profiles" / "traffic.json").write_text(json.dumps({"kernels": {"k": entry}}))
    assert bench.measured_traffic("k") == 123
    assert bench.traffic_note("k") == "captured on a smaller case, scaled by blocks"
    assert bench.measured_traffic("other") is None
    src.write_text("// kernel v2\n")  # changed since the capture
    assert bench.measured_traffic("k") is None


def test_committed_traffic_entries_match_their_sources():
    """Every committed figure names a source that exists and a profile summary
    that exists; the hash states whether the figure is current."""
    root = os.path.dirname(os.path.dirname(os.path.abspath(__file__)))
    d = json.load(open(os.path.join(root, "profiles", "traffic.json")))
    for key, k in d["kernels"].items():
        assert os.path.exists(os.path.join(root, k["source"])), key
        assert os.path.exists(os.path.join(root, k["profile"])), key
        if "dram_read_bytes" in k:  # a figure for the bench's own launch
            assert k["dram_read_bytes"] > 0 and k["dram_write_bytes"] > 0, key
        else:  # a capture of a smaller case only, not scaled to the bench launch
            assert k["captured_dram_read_bytes"] > 0 and k["captured_dram_write_bytes"] > 0, key
            assert bench.measured_traffic(key) is None


@pytest.mark.parametrize("ws,ms,want", [(1, 8.0, 1e12 * 40 / 8e-3 / 1e12), (4, 10.0, 4 * 1e12 * 40 / 10e-3 / 1e12)])
def test_whole_job_rate(ws, ms, want):
    assert bench.whole_job_tflops(1e12, 40, ws, ms) == pytest.approx(want)
