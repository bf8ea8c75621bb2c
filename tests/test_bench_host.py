"""Host-side arithmetic of bench.py (no GPU): the per-call roofline of the measurement rule,
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


def test_recorded_traffic_only_for_its_class_and_sources(monkeypatch):
    """The roofline's DRAM traffic is reported for the recorded class while the kernel and planner sources
    hash to the recorded digest, and is withheld once any of them differs."""
    rec = dict(bench.TRAFFIC)
    monkeypatch.setattr(bench, "TRAFFIC", dict(rec, sha256=bench.sources_digest(rec["sources"])))
    got = bench.recorded_traffic(rec["class"])
    assert got is not None and got["bytes_per_call"] == rec["bytes_per_call"]
    assert got["bytes_per_call"] >= got["algorithmic_bytes_per_call"] > 0
    assert bench.recorded_traffic("m_le_16" if rec["class"] != "m_le_16" else "m_ge_512") is None
    monkeypatch.setattr(bench, "TRAFFIC", dict(rec, sha256="0" * 64))
    assert bench.recorded_traffic(rec["class"]) is None

