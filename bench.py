#!/usr/bin/env python3
"""Benchmark of the GB300 BF16 GEMM library.

    python bench.py [--gpus N] [--steps K] [--warmup W] [--impl ours|reference]
                    [--workload NAME] [--shard] [--no-others] [--no-cpu-baseline]

One step is one library call on the headline workload (BF16 GEMM, M=N=K=4096,
BF16 output; other workloads with --workload).  Inputs are seeded synthetic
data already resident in HBM; the 96 MB working set fits in the 129 MB L2, so
between timed steps (outside the timed events) a 256 MiB buffer is written and
another 512 MiB buffer is read, which evicts the inputs and leaves only clean
lines in L2.  Each step is timed with CUDA events on the launching stream.
Prints ONE JSON line on rank 0.

``--impl reference`` times the CPU oracle (the reference arm of this
benchmark) on a bounded sample of the same workload on the host cores.

Under torchrun every rank runs its own copy of the workload (weak scaling),
or with ``--shard`` one copy of the workload is split over the ranks by
columns of the output (rank r computes C[:, n-slice r] from A and its rows of
B, with no collective: strong scaling).
"""
from __future__ import annotations

import argparse
import dataclasses
import hashlib
import json
import math
import os
import statistics
import subprocess
import sys
import threading
import time

ROOT = os.path.dirname(os.path.abspath(__file__))
sys.path.insert(0, ROOT)

import numpy as np  # noqa: E402
import torch  # noqa: E402

import workloads  # noqa: E402

FLUSH_BYTES = 256 << 20        # written
FLUSH_READ_BYTES = 512 << 20   # then read: four times the 129 MB L2

# DRAM traffic per launch from `ncu --metrics dram__bytes_read.sum,dram__bytes_write.sum`
# on the named workload, valid only for the sources the kernel is compiled from
# (`src_sha` over the kernel's source files) and for the plan it ran with.
PAIR_KERNEL_SOURCES = ("ptx.cuh", "gemm_kernels.cuh", "gemm_kernels_pair.cuh", "rms_norm.cuh")
SMALLM_KERNEL_SOURCES = ("ptx.cuh", "gemm_kernels.cuh", "gemm_smallm.cuh")
NCU_TRAFFIC: dict = {
    # the CTA-pair kernel on 4096^3 BF16: 75.94 MB read + 29.04 MB written per launch
    "gemm_4096_bf16": {"bytes": 104982528, "sources": PAIR_KERNEL_SOURCES,
                       "src_sha": "a5917f6edeffe008",
                       "plan": {"kernel_name": "pair", "tile_n": 256, "split_k": 2,
                                "tiles": 284, "stages": 6}},
    # the small-M kernel on 64 x 8192 x 8192: 135.48 MB read + 3.21 MB written per launch
    "smallm_64x8192x8192": {"bytes": 138696960, "sources": SMALLM_KERNEL_SOURCES,
                            "src_sha": "59d11cdda17c6d50",
                            "plan": {"kernel_name": "small_m", "tile_n": 64, "split_k": 4,
                                     "tiles": 64, "stages": 8}},
}


def kernel_source_hash(files=None) -> str:
    """sha256 prefix over the named csrc files (all .cu/.cuh files when None)."""
    h = hashlib.sha256()
    csrc = os.path.join(ROOT, "dense_bf16_gemm_gb300", "csrc")
    names = sorted(files) if files else sorted(f for f in os.listdir(csrc)
                                               if f.endswith((".cu", ".cuh")))
    for f in names:
        with open(os.path.join(csrc, f), "rb") as fh:
            h.update(f.encode())
            h.update(fh.read())
    return h.hexdigest()[:16]


def traffic_of(w, plan) -> int | None:
    """ncu DRAM bytes per launch of workload w, if taken with these kernel
    sources and this plan."""
    tr = NCU_TRAFFIC.get(w.name)
    if not tr or tr.get("src_sha") != kernel_source_hash(tr["sources"]):
        return None
    if any(plan.get(k) != v for k, v in tr["plan"].items()):
        return None
    return tr["bytes"]


def load_peaks() -> dict:
    path = os.path.join(ROOT, "MEASURED_PEAKS.json")
    if os.path.exists(path):
        with open(path) as f:
            d = json.load(f)
        return {"hbm_gbs": d["hbm_gbs"], "bf16_tflops": d["bf16_tflops"],
                "bf16_tflops_sustained": d.get("bf16_tflops_sustained"), "source": "measured"}
    return {"hbm_gbs": 6800.0, "bf16_tflops": 1900.0, "bf16_tflops_sustained": 1700.0,
            "source": "fallback"}


# ---------------------------------------------------------------------------
# clocks during the timed region
# ---------------------------------------------------------------------------
# Clock-event reason bits of NVML (nvml.h, nvmlClocksEventReason* /
# nvmlClocksThrottleReason*) that slow the SM clock, by the names nvidia-smi uses.
CLOCK_EVENT_REASONS = ((0x4, "sw_power_cap"), (0x8, "hw_slowdown"),
                       (0x20, "sw_thermal_slowdown"), (0x40, "hw_thermal_slowdown"),
                       (0x80, "hw_power_brake_slowdown"))


def reason_names(mask: int) -> list[str]:
    """The slow-down reasons set in an NVML clock-event reason mask."""
    return [name for bit, name in CLOCK_EVENT_REASONS if mask & bit]


class NvmlReader:
    """Reads one GPU's SM clock, maximum SM clock, power draw and active clock-event
    reasons through NVML's C library.  Queries only: nothing is set."""

    NVML_CLOCK_SM = 1

    def __init__(self, index: int, pci_bus_id: str | None = None):
        import ctypes
        self.ct = ctypes
        lib = ctypes.CDLL("libnvidia-ml.so.1")
        if lib.nvmlInit_v2() != 0:
            raise OSError("nvmlInit_v2 failed")
        self.lib = lib
        h = ctypes.c_void_p()
        rc = 1
        if pci_bus_id:
            rc = lib.nvmlDeviceGetHandleByPciBusId_v2(pci_bus_id.encode(), ctypes.byref(h))
        if rc != 0:
            rc = lib.nvmlDeviceGetHandleByIndex_v2(ctypes.c_uint(index), ctypes.byref(h))
        if rc != 0:
            lib.nvmlShutdown()
            raise OSError(f"no NVML handle for GPU {pci_bus_id or index}")
        self.h = h
        self.get_reasons = (getattr(lib, "nvmlDeviceGetCurrentClocksEventReasons", None)
                            or lib.nvmlDeviceGetCurrentClocksThrottleReasons)

    def read(self):
        """(SM MHz, max SM MHz, watts, [reasons]); None for a value NVML does not give.
        The power is the driver's averaged reading, so a region of a few
        milliseconds shows less than the draw under load."""
        ct = self.ct
        sm, smax, mw, mask = ct.c_uint(), ct.c_uint(), ct.c_uint(), ct.c_ulonglong()
        ok_sm = self.lib.nvmlDeviceGetClockInfo(self.h, self.NVML_CLOCK_SM, ct.byref(sm)) == 0
        ok_max = self.lib.nvmlDeviceGetMaxClockInfo(self.h, self.NVML_CLOCK_SM,
                                                    ct.byref(smax)) == 0
        ok_w = self.lib.nvmlDeviceGetPowerUsage(self.h, ct.byref(mw)) == 0
        ok_r = self.get_reasons(self.h, ct.byref(mask)) == 0
        return (float(sm.value) if ok_sm else None, float(smax.value) if ok_max else None,
                mw.value / 1000.0 if ok_w else None, reason_names(mask.value) if ok_r else [])

    def close(self):
        self.lib.nvmlShutdown()


def parse_smi_line(line: str):
    """One line of `nvidia-smi --query-gpu=<ClockSampler.FIELDS> --format=csv,noheader,
    nounits` as (SM MHz, max SM MHz, watts, [reasons]), or None."""
    parts = [p.strip() for p in line.split(",")]
    if len(parts) < 9:
        return None

    def num(x):
        try:
            return float(x)
        except ValueError:
            return None
    names = ["hw_slowdown", "hw_thermal_slowdown", "sw_thermal_slowdown", "sw_power_cap"]
    reasons = [n for n, v in zip(names, parts[5:9]) if v.lower() == "active"]
    return num(parts[1]), num(parts[2]), num(parts[3]), reasons


def pci_bus_id(dev) -> str | None:
    """The device's PCI address in NVML's form (domain:bus:device.0), or None."""
    try:
        p = torch.cuda.get_device_properties(dev)
        return f"{p.pci_domain_id:08X}:{p.pci_bus_id:02X}:{p.pci_device_id:02X}.0"
    except (AttributeError, RuntimeError, AssertionError):
        return None


class ClockSampler:
    """Samples the GPU's clocks while a timed region runs: through NVML every
    `period` seconds (so even a timed region of a few milliseconds gets several
    samples), else through `nvidia-smi -lms 100`.  `reader` replaces the NVML
    reader (tests)."""

    FIELDS = ("index,clocks.sm,clocks.max.sm,power.draw,clocks_event_reasons.active,"
              "clocks_event_reasons.hw_slowdown,clocks_event_reasons.hw_thermal_slowdown,"
              "clocks_event_reasons.sw_thermal_slowdown,clocks_event_reasons.sw_power_cap")

    def __init__(self, gpu_index: int, pci_bus_id: str | None = None, reader=None,
                 period: float = 0.002):
        self.gpu = gpu_index
        self.pci_bus_id = pci_bus_id
        self.reader = reader
        self.period = period
        self.source = None
        self.proc = None
        self._th = None
        self._stop = threading.Event()
        self.rows: list[tuple[float, tuple]] = []
        self.t0 = self.t1 = None

    def start(self):
        if self.reader is None:
            try:
                self.reader = NvmlReader(self.gpu, self.pci_bus_id)
            except (OSError, AttributeError):
                self.reader = None
        if self.reader is not None:
            self.source = "nvml"
            self._th = threading.Thread(target=self._poll, daemon=True)
            self._th.start()
            return
        try:
            self.proc = subprocess.Popen(
                ["nvidia-smi", f"--id={self.pci_bus_id or self.gpu}",
                 f"--query-gpu={self.FIELDS}", "--format=csv,noheader,nounits", "-lms", "100"],
                stdout=subprocess.PIPE, stderr=subprocess.DEVNULL, text=True)
        except (OSError, FileNotFoundError):
            self.proc = None
            return
        self.source = "nvidia-smi"
        self._th = threading.Thread(target=self._read_smi, daemon=True)
        self._th.start()

    def _poll(self):
        while not self._stop.is_set():
            t = time.time()
            try:
                r = self.reader.read()
            except Exception:  # a failing query ends the sampling, not the run
                return
            self.rows.append((t, r))
            self._stop.wait(self.period)

    def _read_smi(self):
        for line in self.proc.stdout:
            r = parse_smi_line(line)
            if r is not None:
                self.rows.append((time.time(), r))

    def mark(self, begin: bool):
        if begin:
            self.t0 = time.time()
        else:
            self.t1 = time.time()

    def stop(self) -> dict:
        if self.source is None:
            return {"sm_mhz": None, "sm_max_mhz": None, "reasons": ["clock source unavailable"],
                    "samples": 0, "source": None}
        if self.source == "nvml":
            time.sleep(2 * self.period)
            self._stop.set()
            self._th.join(timeout=5)
            try:
                self.reader.close()
            except Exception:
                pass
        else:
            time.sleep(0.25)
            self.proc.terminate()
            try:
                self.proc.wait(timeout=5)
            except subprocess.TimeoutExpired:
                self.proc.kill()
        return self.summary()

    def summary(self) -> dict:
        """Median SM clock, maximum SM clock, reasons seen and peak power over the
        samples inside the marked region, widened on each side by one sampling
        period (100 ms for nvidia-smi); all samples if none fell inside."""
        rows = list(self.rows)
        pad = self.period if self.source == "nvml" else 0.1
        inside = [r for t, r in rows
                  if self.t0 is not None and self.t1 is not None
                  and self.t0 - pad <= t <= self.t1 + pad]
        use = inside if inside else [r for _, r in rows]
        sm = [r[0] for r in use if r[0] is not None]
        smax = [r[1] for r in use if r[1] is not None]
        watts = [r[2] for r in use if r[2] is not None]
        reasons = sorted({name for r in use for name in r[3]})
        return {"sm_mhz": statistics.median(sm) if sm else None,
                "sm_max_mhz": max(smax) if smax else None,
                "reasons": reasons,
                "samples": len(inside),
                "power_w_max": max(watts) if watts else None,
                "source": self.source}


# ---------------------------------------------------------------------------
# distributed plumbing (one process per GPU, no data-path collective)
# ---------------------------------------------------------------------------
def dist_setup(n_gpus: int):
    world = int(os.environ.get("WORLD_SIZE", "1"))
    rank = int(os.environ.get("RANK", "0"))
    local = int(os.environ.get("LOCAL_RANK", "0"))
    pg = None
    if world > 1:
        import torch.distributed as dist
        backend = "nccl" if torch.cuda.is_available() else "gloo"
        if torch.cuda.is_available():
            torch.cuda.set_device(local)
        dist.init_process_group(backend=backend)
        pg = dist
    elif torch.cuda.is_available():
        torch.cuda.set_device(0)
    return world, rank, local, pg


def barrier(pg):
    if pg is not None:
        pg.barrier()


def max_over_ranks(pg, x: float) -> float:
    if pg is None:
        return x
    t = torch.tensor([x], dtype=torch.float64,
                     device="cuda" if torch.cuda.is_available() else "cpu")
    pg.all_reduce(t, op=pg.ReduceOp.MAX)
    return float(t.item())


def sum_over_ranks(pg, x: float) -> float:
    if pg is None:
        return x
    t = torch.tensor([x], dtype=torch.float64,
                     device="cuda" if torch.cuda.is_available() else "cpu")
    pg.all_reduce(t, op=pg.ReduceOp.SUM)
    return float(t.item())


SHARD_ALIGN = 256   # the widest tile: every slice but the last is whole tiles


def shard_bounds(N: int, world: int, rank: int, align: int = SHARD_ALIGN):
    """Columns [n0, n1) of rank `rank` when N output columns are split over
    `world` ranks: contiguous slices of whole `align`-column blocks, as equal
    as the blocks allow (the last slice takes the ragged end)."""
    blocks = -(-N // align)
    per, extra = divmod(blocks, world)
    b0 = rank * per + min(rank, extra)
    b1 = b0 + per + (1 if rank < extra else 0)
    return min(N, b0 * align), min(N, b1 * align)


def shardable(w) -> bool:
    """Workloads whose output columns are independent (split N, no exchange)."""
    return w.kind in ("gemm", "gate_up") and w.batch == 1


def shard_host_inputs(w, host, n0, n1):
    """The slice of the workload's inputs one rank needs for columns [n0, n1):
    all of A (or X), rows n0..n1-1 of B (or Wg, Wu), columns n0..n1-1 of C."""
    out = {}
    for k, v in host.items():
        if k in ("B", "Wg", "Wu"):
            out[k] = v[n0:n1].contiguous()
        elif k == "C":
            out[k] = v[:, n0:n1].contiguous()
        else:
            out[k] = v
    return out


def workload_config(w, world: int, shard: bool) -> dict:
    """The `config` object of the JSON line, the same for both arms."""
    return {"workload": w.name, "batch": w.batch, "M": w.M, "N": w.N, "K": w.K,
            "in_dtype": compute_dtype(w), "out_dtype": SHORT[w.out_dtype],
            "alpha": w.alpha, "beta": w.beta,
            "l2": "GPU arm: flushed between steps (256 MiB write + 512 MiB read, untimed)",
            "parallelism": (f"{world}-way split of the output columns, no collective" if shard
                            else f"{world} independent replica(s), no collective")}


# ---------------------------------------------------------------------------
# our arm
# ---------------------------------------------------------------------------
def host_inputs(w):
    """The workload's seeded CPU tensors, by name."""
    if w.kind == "gate_up":
        X, Wg, Wu = workloads.gate_up_inputs(w.M, w.N, w.K, w.seed, w.dist_a, w.dist_b)
        return {"X": X, "Wg": Wg, "Wu": Wu}
    if w.kind == "rms_norm":
        X, G = workloads.inputs_for(w)
        return {"X": X, "G": G}
    if w.kind == "rmsnorm_gate_up":
        X, G, Wg, Wu = workloads.inputs_for(w)
        return {"X": X, "G": G, "Wg": Wg, "Wu": Wu}
    if w.kind == "attention":
        Q, K, V = workloads.inputs_for(w)
        return {"Q": Q, "K": K, "V": V}
    A, B, C = workloads.inputs_for(w)
    d = {"A": A, "B": B}
    if C is not None:
        d["C"] = C.to(w.out_dtype)
    return d


def out_shape(w):
    """Shape of the workload's main result."""
    if w.kind == "rms_norm":
        return (w.M, w.K)
    if w.kind == "attention":
        return (w.batch, w.M, w.K)
    return (w.batch, w.M, w.N) if w.batch > 1 else (w.M, w.N)


def make_device_inputs(w, dev, host=None):
    t = {k: v.to(dev) for k, v in (host if host is not None else host_inputs(w)).items()}
    if "C" not in t:
        t["C"] = torch.empty(out_shape(w), dtype=w.out_dtype, device=dev)
    if w.kind == "rmsnorm_gate_up":
        t["Xn"] = torch.empty((w.M, w.K), dtype=torch.bfloat16, device=dev)
    if w.kind == "gemm_row_stats":
        lead = (w.batch, w.M) if w.batch > 1 else (w.M,)
        t["stats"] = [torch.empty(lead, dtype=torch.float32, device=dev) for _ in range(3)]
    return t


def call(lib, w, t, stream):
    """One step: the workload's library call on device-resident tensors.
    Returns the main result."""
    if w.kind == "gate_up":
        return lib.gate_up_silu(t["X"], t["Wg"], t["Wu"], t["C"], stream=stream)
    if w.kind == "rms_norm":
        return lib.rms_norm(t["X"], t["G"], w.eps, Y=t["C"], stream=stream)
    if w.kind == "rmsnorm_gate_up":
        return lib.rmsnorm_gate_up_silu(t["X"], t["G"], w.eps, t["Wg"], t["Wu"], Xn=t["Xn"],
                                        Y=t["C"], stream=stream)[0]
    if w.kind == "gemm_row_stats":
        return lib.gemm_row_stats(t["A"], t["B"], t["C"], alpha=w.alpha, beta=w.beta,
                                  stream=stream, stats=t["stats"])[0]
    if w.kind == "attention":
        return lib.attention(t["Q"], t["K"], t["V"], w.K ** -0.5, O=t["C"], stream=stream)
    return lib.gemm(t["A"], t["B"], t["C"], alpha=w.alpha, beta=w.beta, stream=stream)


def plan_of(lib, w):
    if w.kind == "gate_up":
        return lib.gate_up_plan(w.M, w.N, w.K)
    if w.kind == "rmsnorm_gate_up":
        pl = dict(lib.gate_up_plan(w.M, w.N, w.K))
        single = (pl["kernel_name"] == "pair_gate_up" and w.K % 8 == 0 and w.K * 10 <= 224 * 1024
                  and os.environ.get("GB3_NORM_ROW_WARPS") != "1"
                  and os.environ.get("GB3_RMSNORM_SINGLE_LAUNCH", "0") == "1")
        if single:
            pl["kernel_name"] = "pair_gate_up with the normalisation in the same launch"
        else:
            pl["launches"] += 1      # the normalisation, then the projection
            pl["kernel_name"] = "rms_norm+" + pl["kernel_name"]
        return pl
    if w.kind == "rms_norm":
        return {"kernel_name": "rms_norm", "tile_n": w.K, "split_k": 1, "grid": None,
                "launches": 1}
    if w.kind == "attention":
        return {"kernel_name": "attention", "tile_n": 128, "split_k": 1,
                "grid": w.batch * -(-w.M // 128), "launches": 1}
    in_dt = torch.float16 if w.in_f16 else torch.bfloat16
    if w.kind == "gemm_row_stats":
        return lib.row_stats_plan(w.batch, w.M, w.N, w.K, in_dt, w.out_dtype)
    return lib.batched_plan(w.batch, w.M, w.N, w.K, in_dt, w.out_dtype)


def flush_l2(flush):
    """Evict L2 without leaving dirty lines: write one 256 MiB buffer, then
    read a 512 MiB one, so the write-backs of the first happen here, untimed,
    and not during the next timed step.  Reading only 256 MiB left some of the
    written lines dirty in L2: on GB300 the next call then paid for their
    write-backs (the 64 x 8192 x 8192 small-M GEMM 40.8 us against 35.7 us
    after a 512 MiB read, the 16 x 28672 x 8192 decode GEMM 86.0 against 84.0;
    the 4096^3 GEMM unchanged)."""
    flush[0].add_(1)
    flush[1].sum()


def time_device(lib, w, t, steps, warmup, stream, flush, sampler=None):
    """Per-step CUDA-event times (ms) of one library call, L2 flushed between."""
    with torch.cuda.stream(stream):
        for _ in range(warmup):
            flush_l2(flush)
            call(lib, w, t, stream)
    torch.cuda.synchronize()
    ev = [(torch.cuda.Event(enable_timing=True), torch.cuda.Event(enable_timing=True))
          for _ in range(steps)]
    if sampler:
        sampler.mark(True)
    with torch.cuda.stream(stream):
        for i in range(steps):
            flush_l2(flush)
            ev[i][0].record(stream)
            call(lib, w, t, stream)
            ev[i][1].record(stream)
    torch.cuda.synchronize()
    if sampler:
        sampler.mark(False)
    return [a.elapsed_time(b) for a, b in ev]


def time_e2e(lib, w, steps, warmup, stream, dev, host=None):
    """Public API end to end, run as a serving loop runs it: every step copies
    its inputs from pinned host memory to the device, makes the library call and
    copies its result back to pinned host memory, all inside the timed region.
    Consecutive steps overlap: step i's inputs travel on a copy stream while
    step i-1 computes and step i-2's result travels back on a third stream
    (two device buffer sets, each reused once its previous step's result is
    back on the host)."""
    host = {k: v.pin_memory() for k, v in (host if host is not None else host_inputs(w)).items()}
    sets = [make_device_inputs(w, dev, host) for _ in range(2)]
    host_out = [torch.empty(out_shape(w), dtype=w.out_dtype).pin_memory() for _ in range(2)]
    h2d = sum(h.numel() * h.element_size() for h in host.values())
    d2h = host_out[0].numel() * host_out[0].element_size()
    s_in, s_out = torch.cuda.Stream(dev), torch.cuda.Stream(dev)
    ev = {name: [torch.cuda.Event() for _ in range(2)] for name in ("in", "comp", "out")}
    issued = [0, 0]

    def one(i):
        b = i % 2
        t = sets[b]
        if issued[b]:
            s_in.wait_event(ev["out"][b])      # buffer set b's previous result is home
        with torch.cuda.stream(s_in):
            for k, h in host.items():
                t[k].copy_(h, non_blocking=True)
            ev["in"][b].record(s_in)
        stream.wait_event(ev["in"][b])
        with torch.cuda.stream(stream):
            out = call(lib, w, t, stream)
            ev["comp"][b].record(stream)
        s_out.wait_event(ev["comp"][b])
        with torch.cuda.stream(s_out):
            host_out[b].copy_(out, non_blocking=True)
            ev["out"][b].record(s_out)
        issued[b] = 1

    for i in range(warmup):
        one(i)
    torch.cuda.synchronize()
    t0 = torch.cuda.Event(enable_timing=True)
    t1 = torch.cuda.Event(enable_timing=True)
    t0.record(stream)
    s_in.wait_event(t0)
    for i in range(steps):
        one(warmup + i)
    stream.wait_stream(s_out)
    t1.record(stream)
    torch.cuda.synchronize()
    return t0.elapsed_time(t1) / steps, h2d, d2h


def hbm_bound(w) -> bool:
    """Workloads whose metric is bandwidth: the decode-shaped GEMMs (M = 16
    and 64) and the row normalisation."""
    return w.name.startswith(("skinny", "smallm")) or w.kind == "rms_norm"


def metric_of(w, ms):
    """(value, unit) of the workload's metric for a step time in ms."""
    if hbm_bound(w):
        return w.algorithmic_bytes / (ms * 1e-3) / 1e9, "GB/s"
    return w.flops / (ms * 1e-3) / 1e12, "TFLOP/s"


def roofline(w, ms, peaks, traffic):
    if hbm_bound(w):
        achieved = w.algorithmic_bytes / (ms * 1e-3) / 1e9
        peak = peaks["hbm_gbs"]
        return {"bound": "hbm", "achieved": round(achieved, 1), "peak": peak, "unit": "GB/s",
                "frac": round(achieved / peak, 4), "traffic": traffic,
                "peak_source": peaks["source"] + " copy bandwidth"}
    achieved = w.flops / (ms * 1e-3) / 1e12
    peak = peaks["bf16_tflops"]
    out = {"bound": "tensor", "achieved": round(achieved, 1), "peak": peak, "unit": "TFLOP/s",
           "frac": round(achieved / peak, 4), "traffic": traffic,
           "peak_source": peaks["source"] + " bf16 burst"}
    if peaks.get("bf16_tflops_sustained"):
        out["frac_of_sustained"] = round(achieved / peaks["bf16_tflops_sustained"], 4)
    return out


def oracle_rows(w):
    """A function computing whole output rows 0 .. rows-1 of the workload
    (of its first matrix when batched) with the oracle, as it stands."""
    import oracle
    h = host_inputs(w)
    if w.kind == "gate_up":
        def run(rows):
            r = np.repeat(np.arange(rows), w.N)
            c = np.tile(np.arange(w.N), rows)
            oracle.gate_up_entries(h["X"], h["Wg"], h["Wu"], r, c)
    elif w.kind == "rmsnorm_gate_up":
        def run(rows):
            r = np.repeat(np.arange(rows), w.N)
            c = np.tile(np.arange(w.N), rows)
            oracle.rmsnorm_gate_up_entries(h["X"], h["G"], w.eps, h["Wg"], h["Wu"], r, c)
    elif w.kind == "rms_norm":
        def run(rows):
            oracle.rms_norm(h["X"], h["G"], w.eps, np.arange(rows))
    elif w.kind == "attention":
        def run(rows):
            oracle.attention_rows(h["Q"], h["K"], h["V"], w.K ** -0.5, np.zeros(rows, np.int64),
                                  np.arange(rows))
    else:
        A, B, C = first_matrix(h["A"], h["B"], h.get("C"))

        def run(rows):
            Cs = C[:rows].float() if C is not None else None
            v, _ = oracle.gemm_full(A[:rows], B, alpha=w.alpha, beta=w.beta, C=Cs)
            if w.kind == "gemm_row_stats":
                v.sum(axis=1), v.max(axis=1), v.min(axis=1)
    return run


def sample_text(w, rows):
    cols = f"all {w.K} columns" if w.kind == "rms_norm" else f"all {w.N} columns, K={w.K}"
    if w.kind == "attention":
        cols = f"all {w.K} columns over {w.N} keys, head 0 of {w.batch}"
        return (f"query rows 0..{rows - 1} of {w.M} ({cols}); metric scaled to the full "
                f"workload by the row fraction")
    return (f"output rows 0..{rows - 1} of {w.M}{sample_of(w)} ({cols}); "
            f"metric scaled to the full workload by the row fraction")


def cpu_baseline(w, target_s=12.0):
    """The oracle, as it stands, on a bounded sample of the workload: whole
    rows of the output, sized to take about target_s seconds."""
    import oracle
    run = oracle_rows(w)
    rows = 1
    run(rows)                       # threads up, pages touched
    rows = min(w.M, 32 if w.kind != "rms_norm" else 4096)
    t0 = time.perf_counter()
    run(rows)
    dt = time.perf_counter() - t0
    rows = int(max(1, min(w.M, rows * target_s / max(dt, 1e-3))))
    t0 = time.perf_counter()
    run(rows)
    dt = time.perf_counter() - t0
    frac = rows / (w.M * w.batch)
    ms_full = dt / frac * 1e3
    value, unit = metric_of(w, ms_full)
    return {"value": round(value, 6), "unit": unit, "cores": oracle.num_threads(),
            "kind": "oracle", "seconds": round(dt, 3), "sample": sample_text(w, rows)}


SHORT = {torch.float32: "f32", torch.bfloat16: "bf16", torch.float16: "f16"}
METRIC = "BF16 GEMM TFLOP/s & % of GB300 dense peak; GB/s & % of HBM for M=16 skinny"
API = {"gemm": "gemm (C ABI gemm_bf16 / gemm_batched)",
       "gate_up": "gate_up_silu (C ABI gemm_gate_up_silu)",
       "gemm_row_stats": "gemm_row_stats (C ABI gemm_row_stats)",
       "rms_norm": "rms_norm (C ABI gemm_rms_norm)",
       "rmsnorm_gate_up": "rmsnorm_gate_up_silu (C ABI gemm_rmsnorm_gate_up_silu)",
       "attention": "attention (C ABI gemm_attention)"}


def compute_dtype(w) -> str:
    """The arithmetic type of the operands the path computes on."""
    if w.kind == "rms_norm":
        return w.norm_in
    return "f16" if w.in_f16 else "bf16"


def first_matrix(A, B, C):
    """The first problem of a batched workload (the workload itself otherwise)."""
    if A.dim() == 3:
        return A[0], B[0], (C[0] if C is not None else None)
    return A, B, C


def sample_of(w):
    return f" of matrix 0 of {w.batch}" if w.batch > 1 else ""


def run_ours(args):
    world, rank, local, pg = dist_setup(args.gpus)
    dev = torch.device("cuda", local)
    from dense_bf16_gemm_gb300 import build as _b
    _b.build()
    import dense_bf16_gemm_gb300 as lib
    lib._native.lib()
    w_full = workloads.WORKLOADS[args.workload]
    shard = args.shard and world > 1
    if args.shard and not shardable(w_full):
        raise SystemExit(f"--shard splits the output columns of gemm or gate/up workloads, "
                         f"not {w_full.name}")
    w, host = w_full, None
    if shard:
        # this rank's columns of the one problem all ranks share
        n0, n1 = shard_bounds(w_full.N, world, rank)
        w = dataclasses.replace(w_full, N=n1 - n0)
        host = shard_host_inputs(w_full, host_inputs(w_full), n0, n1)
    peaks = load_peaks()
    stream = torch.cuda.Stream(device=dev)
    flush = (torch.zeros(FLUSH_BYTES // 4, dtype=torch.float32, device=dev),
             torch.zeros(FLUSH_READ_BYTES // 4, dtype=torch.float32, device=dev))
    t = make_device_inputs(w, dev, host)
    pl = plan_of(lib, w)

    sampler = ClockSampler(local, pci_bus_id(dev))
    sampler.start()
    barrier(pg)
    torch.cuda.synchronize()
    times = time_device(lib, w, t, args.steps, args.warmup, stream, flush, sampler)
    torch.cuda.synchronize()
    barrier(pg)
    clocks = sampler.stop()
    st, site = lib.device_status(stream)
    if st != 0:
        raise SystemExit(f"device status {st} at site {site}")
    ms_mean = sum(times) / len(times)
    ms_step = max_over_ranks(pg, ms_mean)
    # weak scaling: every rank runs its own problem; shards: the ranks share one
    value, unit = metric_of(w_full, ms_step)
    if not shard:
        value *= world
    src_hash = kernel_source_hash()
    traffic = traffic_of(w, plan_of(lib, w)) if not shard else None
    roof = roofline(w, ms_mean, peaks, traffic)

    e2e_steps = max(3, min(args.steps, 20))
    e2e_ms, h2d, d2h = time_e2e(lib, w, e2e_steps, 2, stream, dev, host)
    e2e_ms = max_over_ranks(pg, e2e_ms)
    e2e_value, _ = metric_of(w_full, e2e_ms)
    if not shard:
        e2e_value *= world
    h2d = int(sum_over_ranks(pg, h2d))
    d2h = int(sum_over_ranks(pg, d2h))

    others = {}
    if not args.no_others and rank == 0 and world == 1:
        for name, ow in workloads.WORKLOADS.items():
            if name == w.name:
                continue
            ot = make_device_inputs(ow, dev)
            otimes = time_device(lib, ow, ot, max(10, min(args.steps, 50)), 3, stream, flush)
            oms = statistics.median(otimes)
            ov, ou = metric_of(ow, oms)
            orf = roofline(ow, oms, peaks, None)
            others[name] = {"value": round(ov, 1), "unit": ou, "ms": round(oms, 4),
                            "frac": orf["frac"], "bound": orf["bound"],
                            "plan": {k: plan_of(lib, ow)[k] for k in ("kernel_name", "tile_n",
                                                                      "split_k", "grid")}}
            del ot
        st, site = lib.device_status(stream)
        if st != 0:
            raise SystemExit(f"device status {st} at site {site}")

    cpu = None
    if rank == 0 and world == 1 and not args.no_cpu_baseline:
        cpu = cpu_baseline(w)

    if rank == 0:
        line = {
            "metric": METRIC,
            "value": round(value, 2),
            "unit": unit,
            "n_gpus": world,
            "steps": args.steps,
            "warmup": args.warmup,
            "ms_per_step": round(ms_step, 5),
            "ms_per_step_median": round(statistics.median(times), 5),
            "higher_is_better": True,
            "scaling": "strong" if shard else "weak",
            "vs_baseline": None,
            "dtype": compute_dtype(w),
            "data": "synthetic (seeded torch.Generator, BF16-rounded)",
            "config": workload_config(w_full, world, shard),
            "plan": pl if not shard else dict(pl, shard_columns=[n0, n1]),
            "roofline": roof,
            "clocks": clocks,
            "e2e": {"value": round(e2e_value, 2), "unit": unit, "ms_per_step": round(e2e_ms, 4),
                    "h2d_bytes_per_step": h2d, "d2h_bytes_per_step": d2h,  # all ranks
                    "api": f"dense_bf16_gemm_gb300.{API[w.kind]} with pinned host copies, "
                           "consecutive steps overlapped on three streams"},
            "gpu_launches": world * args.steps * pl["launches"],   # every rank's launches
            "kernel_src_sha": src_hash,
            "cpu_baseline": cpu,
            "others": others,
        }
        print(json.dumps(line), flush=True)
    if pg is not None:
        pg.destroy_process_group()


# ---------------------------------------------------------------------------
# reference arm: the CPU oracle
# ---------------------------------------------------------------------------
def reference_rows(w, cores: int) -> int:
    """Output rows per reference step: a bounded sample of the workload that
    keeps every core of the oracle's thread pool busy (it splits rows over its
    threads): a whole multiple of the thread count, at least 8 rows (8192 for
    the row normalisation, whose rows are short)."""
    want = 8192 if w.kind == "rms_norm" else 8
    rows = max(want, cores)
    rows = -(-rows // cores) * cores
    return min(w.M, rows)


def run_reference(args):
    world = int(os.environ.get("WORLD_SIZE", "1"))
    rank = int(os.environ.get("RANK", "0"))
    if rank != 0:
        return
    import oracle
    w = workloads.WORKLOADS[args.workload]
    run = oracle_rows(w)
    rows = reference_rows(w, oracle.num_threads())
    for _ in range(args.warmup):
        run(rows)
    t0 = time.perf_counter()
    for _ in range(args.steps):
        run(rows)
    dt = (time.perf_counter() - t0) / args.steps
    ms_full = dt / (rows / (w.M * w.batch)) * 1e3
    value, unit = metric_of(w, ms_full)
    sample = sample_text(w, rows).replace("; metric", " per step; metric")
    line = {
        "impl": "reference",
        "metric": METRIC,
        "value": round(value, 6), "unit": unit, "n_gpus": world, "steps": args.steps,
        "warmup": args.warmup, "ms_per_step": round(dt * 1e3, 3),
        "higher_is_better": True, "scaling": "weak", "vs_baseline": None, "dtype": "f64",
        "data": "synthetic (seeded torch.Generator, BF16-rounded)",
        "config": workload_config(w, world, args.shard and world > 1),
        "cpu_baseline": {"value": round(value, 6), "unit": unit, "cores": oracle.num_threads(),
                         "kind": "oracle", "sample": sample},
        "e2e": {"value": round(value, 6), "unit": unit, "h2d_bytes_per_step": 0,
                "d2h_bytes_per_step": 0},
        "note": "the reference arm is the CPU oracle (plain FP64 loops, OpenMP over rows)",
    }
    print(json.dumps(line), flush=True)


def main():
    ap = argparse.ArgumentParser()
    ap.add_argument("--gpus", type=int, default=1)
    ap.add_argument("--steps", type=int, default=5000)
    ap.add_argument("--warmup", type=int, default=10)
    ap.add_argument("--impl", choices=["ours", "reference"], default="ours")
    ap.add_argument("--workload", default=workloads.HEADLINE, choices=list(workloads.WORKLOADS))
    ap.add_argument("--shard", action="store_true",
                    help="under torchrun: split one problem's output columns over the ranks")
    ap.add_argument("--no-others", action="store_true")
    ap.add_argument("--no-cpu-baseline", action="store_true")
    args = ap.parse_args()
    if args.warmup < 3:
        args.warmup = 3
    if args.impl == "reference":
        run_reference(args)
    else:
        run_ours(args)


if __name__ == "__main__":
    main()
