#!/usr/bin/env python3
"""Benchmark of the GB300 BF16 GEMM library.

    python bench.py [--gpus N] [--steps K] [--warmup W] [--impl ours|reference]
                    [--workload NAME] [--no-others] [--no-cpu-baseline]

One step is one library call on the headline workload (BF16 GEMM, M=N=K=4096,
BF16 output; other workloads with --workload).  Inputs are seeded synthetic
data already resident in HBM; the 96 MB working set fits in the 129 MB L2, so
between timed steps (outside the timed events) a 256 MiB buffer is written and
another 256 MiB buffer is read, which evicts the inputs and leaves only clean
lines in L2.  Each step is timed with CUDA events on the launching stream.
Prints ONE JSON line on rank 0.

``--impl reference`` times the CPU oracle (the reference arm of this
benchmark) on a bounded sample of the same workload on the host cores.
"""
from __future__ import annotations

import argparse
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

FLUSH_BYTES = 256 << 20

# DRAM traffic per launch from `ncu --metrics dram__bytes_read.sum,dram__bytes_write.sum`
# (summarised under profiles/), valid only for the kernel sources it was taken with.
NCU_TRAFFIC: dict = {
    # profiles/gemm_pair_bf16_4096.md: 75.23 MB read + 29.90 MB written per launch
    "gemm_4096_bf16": {"bytes": 105130240, "src_sha": "16beb2a2762d052b"},
}


def kernel_source_hash() -> str:
    h = hashlib.sha256()
    csrc = os.path.join(ROOT, "dense_bf16_gemm_gb300", "csrc")
    for f in sorted(os.listdir(csrc)):
        if f.endswith((".cu", ".cuh")):
            with open(os.path.join(csrc, f), "rb") as fh:
                h.update(f.encode())
                h.update(fh.read())
    return h.hexdigest()[:16]


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
class ClockSampler:
    FIELDS = ("index,clocks.sm,clocks.max.sm,power.draw,clocks_event_reasons.active,"
              "clocks_event_reasons.hw_slowdown,clocks_event_reasons.hw_thermal_slowdown,"
              "clocks_event_reasons.sw_thermal_slowdown,clocks_event_reasons.sw_power_cap")

    def __init__(self, gpu_index: int):
        self.gpu = gpu_index
        self.proc = None
        self.lines: list[tuple[float, str]] = []
        self.t0 = self.t1 = None

    def start(self):
        try:
            self.proc = subprocess.Popen(
                ["nvidia-smi", f"--id={self.gpu}", f"--query-gpu={self.FIELDS}",
                 "--format=csv,noheader,nounits", "-lms", "100"],
                stdout=subprocess.PIPE, stderr=subprocess.DEVNULL, text=True)
        except (OSError, FileNotFoundError):
            self.proc = None
            return
        self._th = threading.Thread(target=self._read, daemon=True)
        self._th.start()

    def _read(self):
        for line in self.proc.stdout:
            self.lines.append((time.time(), line.strip()))

    def mark(self, begin: bool):
        if begin:
            self.t0 = time.time()
        else:
            self.t1 = time.time()

    def stop(self) -> dict:
        if self.proc is None:
            return {"sm_mhz": None, "sm_max_mhz": None, "reasons": ["nvidia-smi unavailable"],
                    "samples": 0}
        time.sleep(0.25)
        self.proc.terminate()
        try:
            self.proc.wait(timeout=5)
        except subprocess.TimeoutExpired:
            self.proc.kill()
        rows = []
        for t, line in self.lines:
            parts = [p.strip() for p in line.split(",")]
            if len(parts) < 9:
                continue
            rows.append((t, parts))
        inside = [r for t, r in rows if self.t0 is not None and self.t0 - 0.05 <= t <= self.t1 + 0.05]
        use = inside if inside else rows
        def num(x):
            try:
                return float(x)
            except ValueError:
                return None
        sm = [num(r[1]) for r in use if num(r[1]) is not None]
        smax = [num(r[2]) for r in use if num(r[2]) is not None]
        reasons = set()
        names = ["hw_slowdown", "hw_thermal_slowdown", "sw_thermal_slowdown", "sw_power_cap"]
        for r in use:
            for name, v in zip(names, r[5:9]):
                if v.strip().lower() == "active":
                    reasons.add(name)
        return {"sm_mhz": statistics.median(sm) if sm else None,
                "sm_max_mhz": max(smax) if smax else None,
                "reasons": sorted(reasons),
                "samples": len(inside),
                "power_w_max": max((num(r[3]) or 0.0) for r in use) if use else None}


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


# ---------------------------------------------------------------------------
# our arm
# ---------------------------------------------------------------------------
def make_device_inputs(w, dev):
    if w.kind == "gate_up":
        X, Wg, Wu = workloads.gate_up_inputs(w.M, w.N, w.K, w.seed, w.dist_a, w.dist_b)
        return {"X": X.to(dev), "Wg": Wg.to(dev), "Wu": Wu.to(dev),
                "Y": torch.empty((w.M, w.N), dtype=torch.bfloat16, device=dev)}
    A, B, C = workloads.inputs_for(w)
    shape = (w.batch, w.M, w.N) if w.batch > 1 else (w.M, w.N)
    Cd = C.to(dev, w.out_dtype) if C is not None else torch.empty(shape, dtype=w.out_dtype,
                                                                  device=dev)
    return {"A": A.to(dev), "B": B.to(dev), "C": Cd}


def call(lib, w, t, stream):
    if w.kind == "gate_up":
        lib.gate_up_silu(t["X"], t["Wg"], t["Wu"], t["Y"], stream=stream)
    else:
        lib.gemm(t["A"], t["B"], t["C"], alpha=w.alpha, beta=w.beta, stream=stream)


def plan_of(lib, w):
    if w.kind == "gate_up":
        return lib.gate_up_plan(w.M, w.N, w.K)
    return lib.batched_plan(w.batch, w.M, w.N, w.K,
                            torch.float16 if w.in_f16 else torch.bfloat16, w.out_dtype)


def flush_l2(flush):
    """Evict L2 without leaving dirty lines: write one 256 MiB buffer, then
    read another, so the write-backs of the first happen here, untimed, and
    not during the next timed step."""
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


def time_e2e(lib, w, steps, warmup, stream, dev):
    """Public API end to end: pinned host inputs -> device, call, result -> host."""
    if w.kind == "gate_up":
        X, Wg, Wu = workloads.gate_up_inputs(w.M, w.N, w.K, w.seed, w.dist_a, w.dist_b)
        host_in = [X.pin_memory(), Wg.pin_memory(), Wu.pin_memory()]
        out_dtype = torch.bfloat16
    else:
        A, B, C = workloads.inputs_for(w)
        out_dtype = w.out_dtype
        host_in = [A.pin_memory(), B.pin_memory()]
        if C is not None:
            host_in.append(C.to(out_dtype).pin_memory())
    dev_in = [torch.empty_like(h, device=dev) for h in host_in]
    host_out = torch.empty((w.batch, w.M, w.N) if w.batch > 1 else (w.M, w.N),
                           dtype=out_dtype).pin_memory()
    h2d = sum(h.numel() * h.element_size() for h in host_in)
    d2h = host_out.numel() * host_out.element_size()

    def one():
        for h, d in zip(host_in, dev_in):
            d.copy_(h, non_blocking=True)
        if w.kind == "gate_up":
            out = lib.gate_up_silu(dev_in[0], dev_in[1], dev_in[2], stream=stream)
        else:
            Cd = dev_in[2] if len(dev_in) > 2 else None
            out = lib.gemm(dev_in[0], dev_in[1], Cd, alpha=w.alpha, beta=w.beta,
                           out_dtype=out_dtype, stream=stream)
        host_out.copy_(out, non_blocking=True)

    with torch.cuda.stream(stream):
        for _ in range(warmup):
            one()
        torch.cuda.synchronize()
        t0 = torch.cuda.Event(enable_timing=True)
        t1 = torch.cuda.Event(enable_timing=True)
        t0.record(stream)
        for _ in range(steps):
            one()
        t1.record(stream)
    torch.cuda.synchronize()
    return t0.elapsed_time(t1) / steps, h2d, d2h


def metric_of(w, ms):
    """(value, unit) of the workload's metric for a step time in ms."""
    if w.name.startswith("skinny"):
        return w.algorithmic_bytes / (ms * 1e-3) / 1e9, "GB/s"
    return w.flops / (ms * 1e-3) / 1e12, "TFLOP/s"


def roofline(w, ms, peaks, traffic):
    if w.name.startswith("skinny"):
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


def cpu_baseline(w, target_s=12.0):
    """The oracle, as it stands, on a bounded sample of the workload: whole
    rows of the output, sized to take about target_s seconds."""
    import oracle
    if w.kind == "gate_up":
        X, Wg, Wu = workloads.gate_up_inputs(w.M, w.N, w.K, w.seed, w.dist_a, w.dist_b)

        def run(rows):
            r = np.repeat(np.arange(rows), w.N)
            c = np.tile(np.arange(w.N), rows)
            oracle.gate_up_entries(X, Wg, Wu, r, c)
    else:
        A, B, C = first_matrix(*workloads.inputs_for(w))

        def run(rows):
            Cs = C[:rows] if C is not None else None
            oracle.gemm_full(A[:rows], B, alpha=w.alpha, beta=w.beta, C=Cs)
    rows = 1
    run(rows)                       # threads up, pages touched
    rows = min(w.M, 32)
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
            "kind": "oracle", "seconds": round(dt, 3),
            "sample": f"output rows 0..{rows - 1} of {w.M}{sample_of(w)} (all {w.N} columns, "
                      f"K={w.K}); metric scaled to the full workload by the row fraction"}


SHORT = {torch.float32: "f32", torch.bfloat16: "bf16", torch.float16: "f16"}


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
    w = workloads.WORKLOADS[args.workload]
    peaks = load_peaks()
    stream = torch.cuda.Stream(device=dev)
    flush = (torch.zeros(FLUSH_BYTES // 4, dtype=torch.float32, device=dev),
             torch.zeros(FLUSH_BYTES // 4, dtype=torch.float32, device=dev))
    t = make_device_inputs(w, dev)
    pl = plan_of(lib, w)

    sampler = ClockSampler(local)
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
    value, unit = metric_of(w, ms_step)
    value *= world          # weak scaling: every rank runs its own problem
    src_hash = kernel_source_hash()
    traffic = None
    tr = NCU_TRAFFIC.get(w.name)
    if tr and tr.get("src_sha") == src_hash:
        traffic = tr["bytes"]
    roof = roofline(w, ms_mean, peaks, traffic)

    e2e_steps = max(3, min(args.steps, 20))
    e2e_ms, h2d, d2h = time_e2e(lib, w, e2e_steps, 2, stream, dev)
    e2e_ms = max_over_ranks(pg, e2e_ms)
    e2e_value, _ = metric_of(w, e2e_ms)
    e2e_value *= world

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
            "metric": "BF16 GEMM TFLOP/s & % of GB300 dense peak; GB/s & % of HBM for M=16 skinny",
            "value": round(value, 2),
            "unit": unit,
            "n_gpus": world,
            "steps": args.steps,
            "warmup": args.warmup,
            "ms_per_step": round(ms_step, 5),
            "ms_per_step_median": round(statistics.median(times), 5),
            "higher_is_better": True,
            "scaling": "weak",
            "vs_baseline": None,
            "dtype": "f16" if w.in_f16 else "bf16",
            "data": "synthetic (seeded torch.Generator, BF16-rounded)",
            "config": {"workload": w.name, "batch": w.batch, "M": w.M, "N": w.N, "K": w.K,
                       "in_dtype": "f16" if w.in_f16 else "bf16",
                       "out_dtype": SHORT[w.out_dtype], "alpha": w.alpha,
                       "beta": w.beta, "l2": "flushed between steps (256 MiB write + 256 MiB read, untimed)",
                       "parallelism": f"{world} independent replica(s), no collective",
                       "plan": pl},
            "roofline": roof,
            "clocks": clocks,
            "e2e": {"value": round(e2e_value, 2), "unit": unit, "ms_per_step": round(e2e_ms, 4),
                    "h2d_bytes_per_step": h2d, "d2h_bytes_per_step": d2h,
                    "api": "dense_bf16_gemm_gb300.gemm (C ABI gemm_bf16) with pinned host copies"},
            "gpu_launches": args.steps * pl["launches"],
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
def run_reference(args):
    world = int(os.environ.get("WORLD_SIZE", "1"))
    rank = int(os.environ.get("RANK", "0"))
    if rank != 0:
        return
    import oracle
    w = workloads.WORKLOADS[args.workload]
    A, B, C = first_matrix(*workloads.inputs_for(w)) if w.kind == "gemm" else (None,) * 3
    if w.kind == "gate_up":
        X, Wg, Wu = workloads.gate_up_inputs(w.M, w.N, w.K, w.seed, w.dist_a, w.dist_b)
    rows = 8   # output rows per step: a bounded sample of the workload

    def step():
        if w.kind == "gate_up":
            r = np.repeat(np.arange(rows), w.N)
            c = np.tile(np.arange(w.N), rows)
            oracle.gate_up_entries(X, Wg, Wu, r, c)
        else:
            oracle.gemm_full(A[:rows], B, alpha=w.alpha, beta=w.beta,
                             C=C[:rows] if C is not None else None)

    for _ in range(args.warmup):
        step()
    t0 = time.perf_counter()
    for _ in range(args.steps):
        step()
    dt = (time.perf_counter() - t0) / args.steps
    ms_full = dt / (rows / (w.M * w.batch)) * 1e3
    value, unit = metric_of(w, ms_full)
    sample = (f"output rows 0..{rows - 1} of {w.M}{sample_of(w)} per step (all {w.N} "
              f"columns, K={w.K}); metric scaled to the full workload by the row fraction")
    line = {
        "impl": "reference",
        "metric": "BF16 GEMM TFLOP/s & % of GB300 dense peak; GB/s & % of HBM for M=16 skinny",
        "value": round(value, 6), "unit": unit, "n_gpus": world, "steps": args.steps,
        "warmup": args.warmup, "ms_per_step": round(dt * 1e3, 3),
        "higher_is_better": True, "scaling": "weak", "vs_baseline": None, "dtype": "f64",
        "data": "synthetic (seeded torch.Generator, BF16-rounded)",
        "config": {"workload": w.name, "batch": w.batch, "M": w.M, "N": w.N, "K": w.K},
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
