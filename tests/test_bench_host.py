"""Host-side logic of bench.py that needs no GPU: the clock summary that
decides whether a run is throttled, the per-kernel DRAM traffic that is only
reported for the sources it was measured on, and the peak table."""

import json
import os
import sys

import pytest

ROOT = os.path.dirname(os.path.dirname(os.path.abspath(__file__)))
sys.path.insert(0, ROOT)

import bench  # noqa: E402


def _line(sm, smax, hw="Not Active", hwt="Not Active", swt="Not Active", pcap="Not Active"):
    return f"0, {sm}, {smax}, 900.00, 0x0000000000000000, {hw}, {hwt}, {swt}, {pcap}"


def test_clock_summary_uses_only_the_timed_region():
    lines = [
        (0.5, _line(1000, 2070, hw="Active")),   # before the timed region: ignored
        (1.0, _line(1800, 2070)),
        (1.1, _line(1900, 2070, pcap="Active")),
        (1.2, _line(2000, 2070)),
        (1.3, "0, [N/A], 2070, 900.00, 0x0, Not Active, Not Active, Not Active, Not Active"),  # unparsable clock
        (1.4, "0, 1950"),                          # truncated line
        (5.0, _line(500, 2070, hwt="Active")),   # after the region (beyond one sampling period): ignored
    ]
    s = bench.summarize_clocks(lines, 1.0, 1.25)
    assert s["samples"] == 3
    assert s["sm_mhz"] == 1900.0 and s["sm_max_mhz"] == 2070.0
    assert s["reasons"] == ["sw_power_cap"]


def test_clock_summary_reports_hardware_slowdown():
    lines = [(t, _line(1200, 2070, hw="Active", swt="Active")) for t in (2.0, 2.1)]
    s = bench.summarize_clocks(lines, 2.0, 2.1)
    assert s["reasons"] == ["hw_slowdown", "sw_thermal_slowdown"]
    assert bench.summarize_clocks([], 0.0, 1.0) == {"sm_mhz": None, "sm_max_mhz": None, "reasons": [], "samples": 0}


def test_traffic_only_for_the_measured_sources(monkeypatch):
    monkeypatch.setattr(bench, "TRAFFIC_SOURCE_HASH", bench.source_hash())
    assert bench.traffic_of("gemm2_partials") == bench.TRAFFIC_BYTES["gemm2_partials"]
    monkeypatch.setattr(bench, "TRAFFIC_SOURCE_HASH", "0" * 16)
    assert bench.traffic_of("gemm2_partials") is None


def test_source_hash_follows_the_step_sources(monkeypatch, tmp_path):
    h = bench.source_hash()
    csrc = tmp_path / "tensor_transformer_mlp_column_gb300" / "csrc"
    csrc.mkdir(parents=True)
    for f in bench.STEP_SOURCES:
        (csrc / f).write_bytes(open(os.path.join(ROOT, "tensor_transformer_mlp_column_gb300", "csrc", f), "rb").read())
    monkeypatch.setattr(bench, "ROOT", str(tmp_path))
    assert bench.source_hash() == h
    with open(csrc / bench.STEP_SOURCES[0], "ab") as fh:
        fh.write(b"\n// changed\n")
    assert bench.source_hash() != h


def test_peaks_measured_file_or_fallback(monkeypatch, tmp_path):
    monkeypatch.setattr(bench, "ROOT", str(tmp_path))
    p = bench.load_peaks()
    assert p["source"] == "fallback" and p["hbm_gbs"] == bench.FALLBACK_HBM_GBS
    (tmp_path / "MEASURED_PEAKS.json").write_text(json.dumps({"hbm_gbs": 7100.0, "bf16_tflops": 2000.0,
                                                               "bf16_tflops_sustained": 1800.0}))
    p = bench.load_peaks()
    assert p == {"hbm_gbs": 7100.0, "bf16_tflops": 2000.0, "bf16_tflops_sustained": 1800.0, "source": "measured"}
