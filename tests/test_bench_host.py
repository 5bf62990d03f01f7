"""CPU checks of the measurement plumbing in bench.py.

The source digest decides whether a committed ncu traffic figure still
applies to the code being measured; the clock summary decides whether a run
is rejected (throttling) or kept; the peak table supplies the roofline
denominators.
"""
import json

import pytest

import bench


def test_source_digest_ignores_comments_and_blank_lines(tmp_path, monkeypatch):
    monkeypatch.setattr(bench, "ROOT", str(tmp_path))
    src = tmp_path / "a.cu"
    src.write_text("int f() {\n  return 1;  // one\n}\n")
    d0 = bench.source_digest(["a.cu"])
    src.write_text("/* a header\n   comment */\nint f() {\n\n  return 1;  // uno\n}\n")
    assert bench.source_digest(["a.cu"]) == d0
    src.write_text("int f() {\n  return 2;\n}\n")
    assert bench.source_digest(["a.cu"]) != d0


def test_kernel_traffic_requires_the_recorded_digest(tmp_path, monkeypatch):
    monkeypatch.setattr(bench, "ROOT", str(tmp_path))
    (tmp_path / "k.cu").write_text("__global__ void k() {}\n")
    (tmp_path / "profiles").mkdir()
    digest = bench.source_digest(["k.cu"])
    (tmp_path / "profiles" / "k_T64.md").write_text(
        "# k\n\ntraffic_bytes_per_launch: 12345 source_sha256: %s\n" % digest)
    assert bench.kernel_traffic("k_T64", ["k.cu"]) == 12345.0
    # a change of code (not of comments) invalidates the recorded traffic
    (tmp_path / "k.cu").write_text("// note\n__global__ void k() {}\n")
    assert bench.kernel_traffic("k_T64", ["k.cu"]) == 12345.0
    (tmp_path / "k.cu").write_text("__global__ void k() { int x = 0; }\n")
    assert bench.kernel_traffic("k_T64", ["k.cu"]) is None
    assert bench.kernel_traffic("absent", ["k.cu"]) is None


def test_clock_summary_keeps_the_timed_window_and_its_reasons():
    cs = bench.ClockSampler("0")
    t = 1000.0
    idle = "Not Active"
    cs.samples = [
        (t - 1.0, "900, 2070, 500, 0x0, %s, %s, %s, %s" % (idle, idle, idle, idle)),
        (t + 0.1, "2070, 2070, 900, 0x4, %s, %s, %s, Active" % (idle, idle, idle)),
        (t + 0.2, "2065, 2070, 950, 0x0, %s, %s, %s, %s" % (idle, idle, idle, idle)),
        (t + 0.3, "garbled"),
        (t + 5.0, "300, 2070, 100, 0x8, Active, %s, %s, %s" % (idle, idle, idle)),
    ]
    cs.mark_start()
    cs.t0, cs.t1 = t, t + 1.0
    s = cs.summary()
    assert s["samples"] == 2
    assert s["sm_mhz"] == pytest.approx(2067.5)
    assert s["sm_max_mhz"] == 2070.0
    assert s["reasons"] == ["sw_power_cap"]      # the slowdown after the window is not counted


def test_clock_summary_without_samples():
    cs = bench.ClockSampler("0")
    cs.t0, cs.t1 = 0.0, 1.0
    assert cs.summary() == {"sm_mhz": None, "sm_max_mhz": None, "reasons": [], "samples": 0}


def test_peaks_measured_or_fallback(tmp_path, monkeypatch):
    monkeypatch.setattr(bench, "ROOT", str(tmp_path))
    peaks, kind = bench.load_peaks()
    assert kind == "fallback" and peaks == bench.FALLBACK_PEAKS
    (tmp_path / "MEASURED_PEAKS.json").write_text(json.dumps(
        {"hbm_gbs": 6657.0, "bf16_tflops": 1902.4, "bf16_tflops_sustained": 1700.5,
         "clocks": "recorded"}))
    peaks, kind = bench.load_peaks()
    assert kind == "measured"
    assert peaks == {"hbm_gbs": 6657.0, "bf16_tflops": 1902.4, "bf16_tflops_sustained": 1700.5}
