"""Host-side arithmetic of bench.py (no GPU): the per-call roofline of the survey's measurement rule,
max((weight + activation bytes) / HBM, 2 M N K / bf16 peak), and its per-class sums."""
import os
import sys

import pytest

ROOT = os.path.dirname(os.path.dirname(os.path.abspath(__file__)))
sys.path.insert(0, ROOT)

import bench  # noqa: E402

PEAKS = {"hbm_gbs": 1000.0, "bf16_tflops": 100.0, "bf16_tflops_sustained": 90.0, "source": "test"}


def test_call_roofline_picks_the_larger_time():
    # 1e6 weight bytes + 1*1000*4 x bytes at 1000 GB/s = 1.004 us; 2*1*1000*1000 flops at 100 TF/s = 0.02 us
    t, b = bench.call_roofline(1, 1000, 1000, 1e6, 4, PEAKS)
    assert b == "hbm" and t == pytest.approx(1.004)
    # M = 4096: 2*4096*1e6 flops = 81.92 us at 100 TF/s > (1e6 + 4096*1000*4) / 1e9 s = 17.4 us
    t, b = bench.call_roofline(4096, 1000, 1000, 1e6, 4, PEAKS)
    assert b == "tensor" and t == pytest.approx(81.92)


def test_class_summary_sums_roofline_over_measured():
    calls = [("a", 1000, 1000, "Q4_K", 1, 0), ("b", 1000, 1000, "Q4_K", 4096, 0)]
    rf = [bench.call_roofline(c[4], c[1], c[2], bench.weight_bytes(c[1], c[2], c[3]), 4, PEAKS) for c in calls]
    call_ms = [0.002, 0.1]                     # 2 us and 100 us measured
    s = bench.class_summary([0, 1], calls, call_ms, rf, PEAKS)
    assert s["us_measured"] == pytest.approx(102.0)
    assert s["frac"] == pytest.approx(round((rf[0][0] + rf[1][0]) / 102.0, 4))
    assert s["bound"] == "tensor"


def test_reference_arm_reports_the_same_config():
    assert bench.bench_config(1) == bench.bench_config(1)
    c = bench.bench_config(1)
    assert c["calls_per_step"] == 105 and "workload" in c
