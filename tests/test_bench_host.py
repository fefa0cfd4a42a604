"""Host logic of bench.py (no GPU): clock-sample parsing, the traffic record's
source gate, the peaks file and the work count of the headline workload."""
import json
import os
import sys

import pytest

ROOT = os.path.dirname(os.path.dirname(os.path.abspath(__file__)))
sys.path.insert(0, ROOT)
import bench  # noqa: E402


def _sampler(lines):
    s = bench.ClockSampler(0)
    s.lines = lines
    return s.summary()


def test_clock_summary_median_under_load_and_reasons():
    lines = ["0, 345, 2070, 150.0, 0x0, Not Active, Not Active, Not Active, Not Active",   # idle, dropped
             "0, 2070, 2070, 1100.0, 0x0, Not Active, Not Active, Not Active, Not Active",
             "0, 1965, 2070, 1390.0, 0x4, Not Active, Not Active, Not Active, Active",
             "0, 2025, 2070, 1200.0, 0x0, Not Active, Not Active, Not Active, Not Active",
             "garbage line",
             "0, [N/A], 2070, 1200.0, 0x0, Not Active, Not Active, Not Active, Not Active"]
    d = _sampler(lines)
    assert d["sm_mhz"] == 2025.0 and d["sm_max_mhz"] == 2070.0
    assert d["reasons"] == ["sw_power_cap"] and d["samples"] == 4


def test_clock_summary_flags_thermal_and_empty():
    d = _sampler(["0, 1500, 2070, 900.0, 0x40, Not Active, Active, Not Active, Not Active"])
    assert d["reasons"] == ["hw_thermal_slowdown"]
    d = _sampler([])
    assert d["sm_mhz"] is None and d["samples"] == 0


def test_headline_work_count():
    # 4 B H N^2 d for the Wan2.2 shape: 117.05 TFLOP per call
    assert bench.attn_flops(1, 40, 75600, 128) == pytest.approx(117.05e12, rel=1e-4)


def test_traffic_record_only_for_its_source(monkeypatch):
    with open(os.path.join(ROOT, "profiles", "traffic.json")) as f:
        rec = json.load(f)["attn_fwd_kernel"]
    monkeypatch.setattr(bench, "kernel_source_hash", lambda: rec["source_hash"])
    assert bench.ncu_traffic("attn_fwd_kernel") == rec["bytes_per_launch_full_size"]
    monkeypatch.setattr(bench, "kernel_source_hash", lambda: "0" * 16)
    assert bench.ncu_traffic("attn_fwd_kernel") is None
    assert bench.ncu_traffic("no_such_kernel") is None


def test_kernel_source_hash_is_stable():
    h = bench.kernel_source_hash()
    assert len(h) == 16 and h == bench.kernel_source_hash()


def test_measured_peaks_read_from_file():
    p = bench.measured_peaks()
    if os.path.exists(os.path.join(ROOT, "MEASURED_PEAKS.json")):
        with open(os.path.join(ROOT, "MEASURED_PEAKS.json")) as f:
            d = json.load(f)
        assert p["source"] == "measured" and p["hbm_gbs"] == d["hbm_gbs"] and p["bf16_tflops"] == d["bf16_tflops"]
    else:
        assert p["source"] == "fallback" and p["hbm_gbs"] == 6800.0


def test_fp8_peak_burst_only_at_full_clock_without_power_cap():
    peaks = {"bf16_tflops": 1900.0, "bf16_tflops_sustained": 1700.0, "sustained_sm_mhz": 1450.0}
    full = {"sm_mhz": 2070.0, "sm_max_mhz": 2070.0, "reasons": []}
    p = bench.fp8_peak_for(peaks, full)
    assert p["which"] == "burst" and p["peak"] == 3800.0 and p["sustained"] == 3400.0
    assert p["clock_matched"] == pytest.approx(3400.0 * 2070.0 / 1450.0)
    capped = dict(full, reasons=["sw_power_cap"])
    assert bench.fp8_peak_for(peaks, capped)["which"] == "sustained"
    slow = dict(full, sm_mhz=1800.0)
    assert bench.fp8_peak_for(peaks, slow)["peak"] == 3400.0
    none = {"sm_mhz": None, "sm_max_mhz": None, "reasons": []}
    p = bench.fp8_peak_for(dict(peaks, sustained_sm_mhz=None), none)
    assert p["which"] == "sustained" and p["clock_matched"] is None


def test_numa_helpers():
    """The e2e leg binds its pinned buffers to the GPU's NUMA node: the sysfs
    cpulist parser and the page-placement query it reports with."""
    import numpy as np
    assert bench._cpulist("0-3,8,10-11\n") == {0, 1, 2, 3, 8, 10, 11}
    assert bench._cpulist("") == set()
    buf = np.ones(1 << 22, np.uint8)          # 4 MB, touched: its pages are resident
    nodes = bench.pinned_pages_nodes(buf.ctypes.data)
    assert nodes is None or (sum(nodes.values()) > 0 and all(n >= 0 for n in nodes))
