"""Host-side pieces of bench.py: the roofline denominators and the recorded DRAM
traffic of the attention kernel (reported only while the kernel sources are the
ones it was captured with)."""
import json
import os

import pytest

import bench


def test_peaks_are_positive():
    peak, peak_sus, hbm, src = bench.peaks()
    assert peak > 0 and hbm > 0 and src in ("measured", "fallback")
    if src == "measured":
        with open(os.path.join(bench.ROOT, "MEASURED_PEAKS.json")) as f:
            p = json.load(f)
        assert peak == p["bf16_tflops"] and hbm == p["hbm_gbs"]


def test_attention_traffic_scales_with_pairs():
    t512 = bench.attention_traffic(512)
    if t512 is None:
        pytest.skip("kernel sources changed since the traffic capture (bench reports null)")
    assert t512 == pytest.approx(bench.ATTN_TRAFFIC_I512)
    assert bench.attention_traffic(2048) == pytest.approx(16 * t512)


def test_attention_traffic_null_for_other_sources(tmp_path, monkeypatch):
    # a copy of the kernel sources with one byte changed must not reuse the capture
    csrc = tmp_path / "protein_pair_representation_gate_b300" / "csrc"
    csrc.mkdir(parents=True)
    for f in ("sm103_kernels.cu", "sm103_ptx.cuh"):
        src = os.path.join(bench.ROOT, "protein_pair_representation_gate_b300", "csrc", f)
        with open(src, "rb") as fh:
            data = fh.read()
        (csrc / f).write_bytes(data + (b" " if f == "sm103_ptx.cuh" else b""))
    monkeypatch.setattr(bench, "ROOT", str(tmp_path))
    assert bench.attention_traffic(2048) is None


def test_clock_sampler_keeps_the_timed_region():
    import datetime
    c = bench.ClockSampler(0)
    na = "Not Active"
    c.lines = [f"2026/12/03 10:00:00.100, 0, 1200, 2032, 300.0, 0x0, {na}, {na}, {na}, {na}",
               f"2026/12/03 10:00:00.150, 0, 1950, 2032, 900.0, 0x4, {na}, {na}, {na}, Active",
               f"2026/12/03 10:00:00.200, 0, 1990, 2032, 950.0, 0x0, {na}, {na}, {na}, {na}",
               f"2026/12/03 10:00:00.400, 0, 1100, 2032, 200.0, 0x0, {na}, Active, {na}, {na}",
               "garbage line"]
    c.t0 = datetime.datetime(2026, 12, 3, 10, 0, 0, 120000)
    c.t1 = datetime.datetime(2026, 12, 3, 10, 0, 0, 300000)
    s = c.summary()
    assert s["samples"] == 2 and s["window"] == "timed region"
    assert s["sm_mhz"] == 1970.0 and s["sm_min_mhz"] == 1950.0 and s["sm_max_mhz"] == 2032.0
    assert s["reasons"] == ["sw_power_cap"]
    # no sample inside the region: every sample is reported, and the summary says so
    c.t0 = c.t1 = datetime.datetime(2026, 12, 3, 10, 0, 0, 310000)
    s = c.summary()
    assert s["samples"] == 4 and s["window"].startswith("whole run")
    assert s["reasons"] == ["hw_thermal_slowdown", "sw_power_cap"]
