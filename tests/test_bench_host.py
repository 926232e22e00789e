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
