"""The multi-process path of bench.py on CPU with the gloo backend, world
size 2: one process per rank, no collective on the data path, timing reduced by
max over ranks, a single JSON line from rank 0."""
import json
import os
import socket
import subprocess
import sys

import pytest
import torch
import torch.distributed as dist
import torch.multiprocessing as mp

ROOT = os.path.dirname(os.path.dirname(os.path.abspath(__file__)))


def free_port() -> int:
    with socket.socket() as s:
        s.bind(("127.0.0.1", 0))
        return s.getsockname()[1]


def _rank_main(rank, world, port, out):
    os.environ.update(MASTER_ADDR="127.0.0.1", MASTER_PORT=str(port), RANK=str(rank),
                      WORLD_SIZE=str(world), LOCAL_RANK=str(rank))
    sys.path.insert(0, ROOT)
    import bench
    dist.init_process_group("gloo", rank=rank, world_size=world)
    try:
        bench.barrier(dist)
        # each rank reports its own step time; the job's time is the slowest rank's
        t = bench.max_over_ranks(dist, 1.0 + rank * 0.25)
        out.put((rank, t))
    finally:
        dist.destroy_process_group()


def test_max_over_ranks_gloo_world2():
    ctx = mp.get_context("spawn")
    q = ctx.Queue()
    port = free_port()
    procs = [ctx.Process(target=_rank_main, args=(r, 2, port, q)) for r in range(2)]
    for p in procs:
        p.start()
    res = dict(q.get(timeout=120) for _ in range(2))
    for p in procs:
        p.join(timeout=60)
        assert p.exitcode == 0
    assert res == {0: 1.25, 1: 1.25}


def test_reference_arm_under_torchrun_world2():
    port = free_port()
    cmd = [sys.executable, "-m", "torch.distributed.run", "--nnodes=1", "--nproc-per-node=2",
           "--master-addr", "127.0.0.1", "--master-port", str(port),
           os.path.join(ROOT, "bench.py"), "--impl", "reference", "--gpus", "2",
           "--steps", "1", "--warmup", "3", "--workload", "gemm_256_f32"]
    env = dict(os.environ, OMP_NUM_THREADS="2")
    r = subprocess.run(cmd, capture_output=True, text=True, timeout=300, env=env, cwd=ROOT)
    assert r.returncode == 0, r.stderr[-2000:]
    lines = [l for l in r.stdout.splitlines() if l.startswith("{")]
    assert len(lines) == 1                      # rank 0 alone prints
    d = json.loads(lines[0])
    assert d["impl"] == "reference" and d["n_gpus"] == 2
    assert d["value"] > 0 and d["e2e"]["h2d_bytes_per_step"] == 0
    assert d["cpu_baseline"]["kind"] == "oracle"


def test_shard_bounds_tile_the_columns():
    sys.path.insert(0, ROOT)
    import bench
    for N in (1, 255, 256, 5000, 14336, 28672):
        for world in (1, 2, 3, 4, 8):
            bounds = [bench.shard_bounds(N, world, r) for r in range(world)]
            assert bounds[0][0] == 0 and bounds[-1][1] == N
            for (a0, a1), (b0, b1) in zip(bounds, bounds[1:]):
                assert a1 == b0 and a0 <= a1
            # slices start and end on 256-column blocks unless they reach N
            for n0, n1 in bounds:
                assert n0 % 256 == 0 or n0 == N
                assert n1 % 256 == 0 or n1 == N
            blocks = [-(-(n1 - n0) // 256) for n0, n1 in bounds]   # 256-column tiles each
            assert max(blocks) - min(blocks) <= 1


def _shard_rank_main(rank, world, port, out):
    os.environ.update(MASTER_ADDR="127.0.0.1", MASTER_PORT=str(port), RANK=str(rank),
                      WORLD_SIZE=str(world), LOCAL_RANK=str(rank))
    sys.path.insert(0, ROOT)
    import bench
    import workloads
    dist.init_process_group("gloo", rank=rank, world_size=world)
    try:
        w = workloads.Workload("t", "gemm", 40, 600, 64, 9, ("uniform",), ("uniform",),
                               alpha=0.5, beta=2.0, dist_c=("normal", 1.0))
        host = bench.host_inputs(w)
        n0, n1 = bench.shard_bounds(w.N, world, rank)
        mine = bench.shard_host_inputs(w, host, n0, n1)
        # the rank's slice of C, computed here in float64 as a stand-in for
        # the library call a GPU rank makes on exactly these tensors
        part = 0.5 * mine["A"].double() @ mine["B"].double().T + 2.0 * mine["C"].double()
        t = bench.max_over_ranks(dist, 1.0 + 0.5 * rank)
        nbytes = bench.sum_over_ranks(dist, float(sum(v.numel() * v.element_size()
                                                      for v in mine.values())))
        out.put((rank, n0, n1, part.numpy(), t, nbytes))
    finally:
        dist.destroy_process_group()


def test_shard_mode_slices_recombine_gloo_world2():
    """--shard on two ranks: the column slices tile the output, each rank's
    inputs are exactly its rows of B and columns of C, the step time is the
    slowest rank's and the copied bytes are the sum over ranks."""
    sys.path.insert(0, ROOT)
    import numpy as np
    import bench
    import workloads
    ctx = mp.get_context("spawn")
    q = ctx.Queue()
    port = free_port()
    procs = [ctx.Process(target=_shard_rank_main, args=(r, 2, port, q)) for r in range(2)]
    for p in procs:
        p.start()
    res = sorted((q.get(timeout=120) for _ in range(2)), key=lambda x: x[0])
    for p in procs:
        p.join(timeout=60)
        assert p.exitcode == 0
    w = workloads.Workload("t", "gemm", 40, 600, 64, 9, ("uniform",), ("uniform",),
                           alpha=0.5, beta=2.0, dist_c=("normal", 1.0))
    h = bench.host_inputs(w)
    full = 0.5 * h["A"].double() @ h["B"].double().T + 2.0 * h["C"].double()
    assert [(r[1], r[2]) for r in res] == [(0, 512), (512, 600)]
    assert np.array_equal(np.concatenate([r[3] for r in res], axis=1), full.numpy())
    assert all(r[4] == 1.5 for r in res)
    per_rank = [2 * 40 * 64 + 2 * (n1 - n0) * 64 + 4 * 40 * (n1 - n0) for _, n0, n1, *_ in res]
    assert all(r[5] == sum(per_rank) for r in res)


def test_shard_mode_is_refused_for_workloads_that_do_not_split_by_columns():
    sys.path.insert(0, ROOT)
    import bench
    import workloads
    assert bench.shardable(workloads.WORKLOADS["gemm_4096_bf16"])
    assert bench.shardable(workloads.WORKLOADS["gate_up_4096x14336x4096"])
    for name, w in workloads.WORKLOADS.items():
        if w.kind in ("attention", "rms_norm", "gemm_row_stats") or w.batch > 1:
            assert not bench.shardable(w), name


def test_reference_arm_config_matches_ours():
    sys.path.insert(0, ROOT)
    import bench
    import workloads
    w = workloads.WORKLOADS["gemm_4096_bf16"]
    cfg = bench.workload_config(w, 1, False)
    assert {"workload", "M", "N", "K", "in_dtype", "out_dtype", "alpha", "beta", "l2"} <= set(cfg)
    # one row per oracle thread at least, a whole multiple of the threads
    for cores in (1, 8, 16, 72):
        rows = bench.reference_rows(w, cores)
        assert rows >= min(cores, w.M) and rows % cores == 0 and rows >= 8
