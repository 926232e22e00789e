"""Host-side arithmetic of bench.py, without a GPU: the reported metric, the
roofline fraction, and when a stored ncu traffic figure may be reported."""
import os
import sys

import pytest

ROOT = os.path.dirname(os.path.dirname(os.path.abspath(__file__)))
sys.path.insert(0, ROOT)

import bench  # noqa: E402
import workloads  # noqa: E402

PEAKS = {"hbm_gbs": 6795.1, "bf16_tflops": 1936.3, "bf16_tflops_sustained": 1715.0,
         "source": "measured"}


def test_headline_metric_and_roofline():
    w = workloads.WORKLOADS["gemm_4096_bf16"]
    assert w.flops == 2.0 * 4096 ** 3
    ms = 0.08
    value, unit = bench.metric_of(w, ms)
    assert unit == "TFLOP/s"
    assert value == pytest.approx(2.0 * 4096 ** 3 / 80e-6 / 1e12)
    r = bench.roofline(w, ms, PEAKS, 123)
    assert r["bound"] == "tensor" and r["unit"] == "TFLOP/s" and r["traffic"] == 123
    assert r["achieved"] == pytest.approx(value, abs=0.05)
    assert r["frac"] == pytest.approx(value / 1936.3, abs=1e-4)
    assert r["frac_of_sustained"] == pytest.approx(value / 1715.0, abs=1e-4)


def test_decode_metric_is_bandwidth_of_the_compulsory_bytes():
    w = workloads.WORKLOADS["skinny_16x28672x8192"]
    assert bench.hbm_bound(w)
    # each input read once, the BF16 output written once
    assert w.algorithmic_bytes == 2 * (16 * 8192 + 28672 * 8192) + 2 * 16 * 28672
    value, unit = bench.metric_of(w, 0.0865)
    assert unit == "GB/s"
    assert value == pytest.approx(w.algorithmic_bytes / 86.5e-6 / 1e9)
    r = bench.roofline(w, 0.0865, PEAKS, None)
    assert r["bound"] == "hbm" and r["peak"] == 6795.1
    assert r["frac"] == pytest.approx(value / 6795.1, abs=1e-4)


@pytest.mark.parametrize("name", sorted(workloads.WORKLOADS))
def test_every_workload_reports_one_consistent_metric(name):
    w = workloads.WORKLOADS[name]
    value, unit = bench.metric_of(w, 1.0)
    r = bench.roofline(w, 1.0, PEAKS, None)
    assert value > 0
    assert unit == ("GB/s" if bench.hbm_bound(w) else "TFLOP/s") == r["unit"]
    assert r["bound"] == ("hbm" if unit == "GB/s" else "tensor")
    assert r["achieved"] == pytest.approx(value, abs=0.05)


def test_traffic_needs_the_same_sources_and_plan(monkeypatch):
    w = workloads.WORKLOADS["gemm_4096_bf16"]
    plan = {"kernel_name": "pair", "tile_n": 256, "split_k": 2, "tiles": 284, "stages": 6}
    entry = {"bytes": 1234, "sources": bench.PAIR_KERNEL_SOURCES,
             "src_sha": bench.kernel_source_hash(bench.PAIR_KERNEL_SOURCES), "plan": dict(plan)}
    monkeypatch.setattr(bench, "NCU_TRAFFIC", {w.name: entry})
    assert bench.traffic_of(w, dict(plan, grid=152)) == 1234
    assert bench.traffic_of(w, dict(plan, split_k=1)) is None        # another plan
    monkeypatch.setattr(bench, "NCU_TRAFFIC", {w.name: dict(entry, src_sha="0" * 16)})
    assert bench.traffic_of(w, plan) is None                          # other sources
    monkeypatch.setattr(bench, "NCU_TRAFFIC", {})
    assert bench.traffic_of(w, plan) is None                          # never measured


def test_source_hash_covers_the_named_files_only():
    pair = bench.kernel_source_hash(bench.PAIR_KERNEL_SOURCES)
    assert pair == bench.kernel_source_hash(tuple(reversed(bench.PAIR_KERNEL_SOURCES)))
    assert pair != bench.kernel_source_hash(bench.SMALLM_KERNEL_SOURCES)
    assert len(pair) == 16 and int(pair, 16) >= 0


class _FakeReader:
    """Stands in for NVML: a scripted SM clock per read, slowed down while
    `throttle` is set; counts reads and closes."""

    def __init__(self):
        self.reads = 0
        self.closed = False
        self.throttle = False

    def read(self):
        self.reads += 1
        if self.throttle:
            return 1400.0, 2070.0, 1350.0, ["sw_power_cap"]
        return 2070.0, 2070.0, 900.0, []

    def close(self):
        self.closed = True


def test_reason_bits_follow_nvml():
    # nvml.h: SwPowerCap 0x4, HwSlowdown 0x8, SwThermalSlowdown 0x20,
    # HwThermalSlowdown 0x40, HwPowerBrakeSlowdown 0x80; idle (0x1) and
    # application-clock (0x2) events are not slow-downs
    assert bench.reason_names(0x0) == []
    assert bench.reason_names(0x1 | 0x2) == []
    assert bench.reason_names(0x4) == ["sw_power_cap"]
    assert bench.reason_names(0x8 | 0x40) == ["hw_slowdown", "hw_thermal_slowdown"]
    assert bench.reason_names(0x20 | 0x80) == ["sw_thermal_slowdown", "hw_power_brake_slowdown"]


def test_smi_line_parses_clocks_power_and_reasons():
    line = "0, 1965, 2070, 1012.54, 0x0000000000000004, Not Active, Not Active, Not Active, Active"
    assert bench.parse_smi_line(line) == (1965.0, 2070.0, 1012.54, ["sw_power_cap"])
    assert bench.parse_smi_line("0, 2070") is None
    sm, smax, w, r = bench.parse_smi_line("0, [N/A], 2070, [N/A], 0x0, Active, Not Active, "
                                          "Not Active, Not Active")
    assert sm is None and w is None and smax == 2070.0 and r == ["hw_slowdown"]


def test_sampler_takes_several_samples_in_a_short_region():
    import time
    fake = _FakeReader()
    s = bench.ClockSampler(0, reader=fake, period=0.001)
    s.start()
    time.sleep(0.05)
    s.mark(True)
    fake.throttle = True
    time.sleep(0.02)          # a timed region of 20 ms
    fake.throttle = False
    s.mark(False)
    time.sleep(0.05)
    c = s.stop()
    assert fake.closed and c["source"] == "nvml"
    assert c["samples"] >= 3
    # the samples inside the region (and at most one period beyond it) decide
    assert c["sm_mhz"] == 1400.0 and c["sm_max_mhz"] == 2070.0
    assert c["reasons"] == ["sw_power_cap"] and c["power_w_max"] == 1350.0
    n = fake.reads
    time.sleep(0.01)
    assert fake.reads == n    # stopped


def test_sampler_without_any_clock_source(monkeypatch):
    def no_nvml(*a, **k):
        raise OSError("no NVML here")
    monkeypatch.setattr(bench, "NvmlReader", no_nvml)
    monkeypatch.setattr(bench.subprocess, "Popen",
                        lambda *a, **k: (_ for _ in ()).throw(FileNotFoundError("nvidia-smi")))
    s = bench.ClockSampler(0)
    s.start()
    s.mark(True)
    s.mark(False)
    c = s.stop()
    assert c["samples"] == 0 and c["sm_mhz"] is None and c["source"] is None
