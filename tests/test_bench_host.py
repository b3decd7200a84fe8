"""Host logic of bench.py (no GPU): the clock record's summary, the peak
lookup and its fallback, and the DRAM-traffic record's staleness check."""
import json
import os

import pytest

import bench


def _sampler(lines):
    cs = bench.ClockSampler(0)
    cs.lines = lines
    return cs.summary()


def test_clock_summary_median_max_and_reasons():
    lines = [
        "0, 2032, 2032, 900.1, 0x0, Not Active, Not Active, Not Active, Not Active",
        "0, 1980, 2032, 1050.3, 0x4, Not Active, Not Active, Not Active, Active",
        "0, 2032, 2032, 990.0, 0x0, Not Active, Not Active, Not Active, Not Active",
        "garbage line",
        "0, [N/A], 2032, 0, 0x0, Not Active, Not Active, Not Active, Not Active",
    ]
    s = _sampler(lines)
    assert s["sm_mhz"] == 2032.0 and s["sm_max_mhz"] == 2032.0
    assert s["reasons"] == ["sw_power_cap"] and s["samples"] == 3


def test_clock_summary_flags_thermal_and_hardware_slowdown():
    lines = ["0, 1500, 2032, 1100, 0x8, Active, Not Active, Active, Not Active"]
    s = _sampler(lines)
    assert s["reasons"] == ["hw_slowdown", "sw_thermal_slowdown"]


def test_clock_summary_without_samples():
    assert _sampler([])["reasons"] == ["unsampled"]


def test_peaks_measured_and_fallback(tmp_path, monkeypatch):
    (tmp_path / "MEASURED_PEAKS.json").write_text(
        json.dumps({"hbm_gbs": 6000.5, "bf16_tflops": 1700.25}))
    monkeypatch.setattr(bench, "ROOT", str(tmp_path))
    hbm, hk, bf, bk = bench.peaks()
    assert (hbm, bf) == (6000.5, 1700.25) and hk == "measured" and bk.startswith("measured")
    os.remove(tmp_path / "MEASURED_PEAKS.json")
    hbm, hk, bf, bk = bench.peaks()
    assert (hbm, bf) == (6400.0, 1800.0) and hk == "fallback" and bk.startswith("fallback")


def test_traffic_record_is_used_only_for_its_source():
    here = os.path.dirname(os.path.abspath(bench.__file__))
    kv = {}
    for line in open(os.path.join(here, "profiles", "tl_mma_kernel_traffic.txt")):
        line = line.strip()
        if line and not line.startswith("#") and "=" in line:
            k, v = line.split("=", 1)
            kv[k] = v
    ratio = (int(kv["dram_bytes_read"]) + int(kv["dram_bytes_write"])) / int(kv["algorithmic_bytes"])
    assert bench.measured_traffic(1_000_000, record="no_such_record.txt") is None
    got = bench.measured_traffic(1_000_000)
    if got is None:
        pytest.skip("the traffic record predates the current kernel source")
    assert abs(got - ratio * 1_000_000) < 1e-6


def test_traffic_record_ignored_once_the_source_changes(tmp_path, monkeypatch):
    src = os.path.join(os.path.dirname(os.path.abspath(bench.__file__)),
                       "bit_matvec_ternary_b300", "csrc", "tl_kernels.cu")
    text = open(src).read()
    real_open = open

    def fake_open(path, *a, **k):
        if os.path.abspath(str(path)) == os.path.abspath(src):
            f = tmp_path / "changed.cu"
            f.write_text("// one more line\n" + text)
            return real_open(f, *a, **k)
        return real_open(path, *a, **k)

    monkeypatch.setattr("builtins.open", fake_open)
    assert bench.measured_traffic(1_000_000) is None
