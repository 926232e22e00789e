"""Parity of the CUDA library with the CPU oracle, element by element, on the
same seeded inputs.  All calls go through the C ABI (via the thin torch
binding, which only marshals pointers)."""
import numpy as np
import pytest
import torch

import oracle
import workloads

pytestmark = pytest.mark.gpu


@pytest.fixture(scope="module")
def g():
    from dense_bf16_gemm_gb300 import build
    build.build()
    import dense_bf16_gemm_gb300 as lib
    # the product path must be the native library
    lib._native.lib()
    return lib


def bits(t):
    return t.contiguous().view(torch.int16).numpy().view(np.uint16)


def to_f64(t):
    return t.detach().to("cpu").to(torch.float64).numpy()


def assert_within(got, ref, tol, what):
    err = np.abs(got - ref)
    bad = ~(err <= tol)
    if bad.any():
        idx = np.argwhere(bad)
        i = tuple(idx[0])
        worst = np.unravel_index(np.nanargmax(np.where(bad, err / np.maximum(tol, 1e-300), 0)),
                                 err.shape)
        raise AssertionError(
            f"{what}: {bad.sum()} of {bad.size} entries out of tolerance; first {i}: "
            f"got {got[i]!r} ref {ref[i]!r} tol {tol[i]!r}; worst {worst}: got {got[worst]!r} "
            f"ref {ref[worst]!r} tol {tol[worst]!r}")


def run_gemm(g, A, B, C=None, alpha=1.0, beta=0.0, out_dtype=torch.bfloat16, fill=float("nan")):
    M, N = A.shape[0], B.shape[0]
    Ad, Bd = A.cuda(), B.cuda()
    if C is not None:
        Cd = C.to(out_dtype).cuda()
    else:
        Cd = torch.full((M, N), fill, dtype=out_dtype, device="cuda")
    g.gemm(Ad, Bd, Cd, alpha=alpha, beta=beta)
    torch.cuda.synchronize()
    return Cd


def int_inputs(M, N, K, seed):
    return workloads.gemm_inputs(M, N, K, seed, ("int", -2, 2), ("int", -2, 2), ("int", -3, 3))


def assert_status_ok(g):
    st, site = g.device_status()
    assert st == 0, f"device status {st} at wait site {site}"


# ---------------------------------------------------------------------------
# bit-exact: integer-valued inputs make every FP32 partial sum exact, so any
# layout, swizzle, descriptor or indexing error shows as a wrong integer.
# ---------------------------------------------------------------------------
EXACT_SHAPES = [
    (128, 256, 64),      # one tile, one k-block
    (300, 520, 200),     # ragged in M, N and K
    (1000, 712, 1000),   # many tiles, slot reuse
    (17, 296, 64),       # just above the skinny threshold
    (256, 256, 8),       # K smaller than one k-block
    (200, 264, 72),      # K tail of 8
    (16, 1000, 4096),    # M <= 16: small-M kernel, or the split-K kernel when forced
    (3, 520, 1000),      # M < 16, ragged N
]


@pytest.mark.parametrize("M,N,K", EXACT_SHAPES)
@pytest.mark.parametrize("out_dtype", [torch.float32, torch.bfloat16])
@pytest.mark.parametrize("route", ["planned", "no_small_m"])
def test_integer_inputs_bit_exact(g, M, N, K, out_dtype, route, monkeypatch):
    if route == "no_small_m":
        if M > 16:
            pytest.skip("the route only changes for M <= 16")
        monkeypatch.setenv("GB3_GEMM_SMALL_M", "0")   # the split-K kernel
        assert g.plan(M, N, K, out_dtype)["kernel_name"] == "skinny_splitk"
    A, B, _ = int_inputs(M, N, K, seed=M + N + K)
    ref, _ = oracle.gemm_full(A, B)
    out = run_gemm(g, A, B, out_dtype=out_dtype)
    if out_dtype == torch.float32:
        assert np.array_equal(to_f64(out), ref)
    else:
        want = oracle.round_to_bf16_bits(ref)
        assert np.array_equal(bits(out.cpu()), want)
    assert_status_ok(g)


@pytest.mark.parametrize("M,N,K", [(300, 520, 200), (16, 1000, 4096), (5, 136, 640)])
@pytest.mark.parametrize("out_dtype", [torch.float32, torch.bfloat16])
def test_integer_inputs_alpha_beta_exact(g, M, N, K, out_dtype):
    A, B, C = int_inputs(M, N, K, seed=7 * M + K)
    alpha, beta = 2.0, -0.5   # powers of two keep the result exact
    Cq = C.to(out_dtype)      # the output storage type is also the input type of C
    ref, _ = oracle.gemm_full(A, B, alpha=alpha, beta=beta, C=Cq.to(torch.float32))
    out = run_gemm(g, A, B, C=Cq, alpha=alpha, beta=beta, out_dtype=out_dtype)
    if out_dtype == torch.float32:
        assert np.array_equal(to_f64(out), ref)
    else:
        assert np.array_equal(bits(out.cpu()), oracle.round_to_bf16_bits(ref))


# ---------------------------------------------------------------------------
# The five workloads
# ---------------------------------------------------------------------------
def check_gemm_workload(g, w, rows=None, cols=None):
    A, B, C = workloads.inputs_for(w)
    out_dtype = torch.bfloat16 if w.out_bf16 else torch.float32
    out = run_gemm(g, A, B, C=C, alpha=w.alpha, beta=w.beta, out_dtype=out_dtype)
    got = to_f64(out)
    if rows is None:
        ref, ab = oracle.gemm_full(A, B, alpha=w.alpha, beta=w.beta, C=C)
        cm = C.numpy() if C is not None else None
    else:
        ref, ab = oracle.gemm_entries(A, B, rows, cols, alpha=w.alpha, beta=w.beta, C=C)
        got = got[rows, cols]
        cm = C.numpy()[rows, cols] if C is not None else None
    tol = oracle.gemm_tolerance(ref, ab, w.alpha, w.beta, cm, out_bf16=w.out_bf16)
    assert_within(got, ref, tol, w.name)
    assert_status_ok(g)


def test_workload_gemm_256_f32(g):
    check_gemm_workload(g, workloads.WORKLOADS["gemm_256_f32"])


@pytest.mark.slow
def test_workload_gemm_4096_bf16(g):
    check_gemm_workload(g, workloads.WORKLOADS["gemm_4096_bf16"])


@pytest.mark.slow
def test_workload_gemm_ragged(g):
    check_gemm_workload(g, workloads.WORKLOADS["gemm_ragged_3000x5000x2000"])


@pytest.mark.slow
def test_workload_skinny(g):
    w = workloads.WORKLOADS["skinny_16x28672x8192"]
    rows, cols = workloads.sample_entries(w.M, w.N, w.seed)
    assert rows.size == w.M * w.N  # the edge region covers every entry
    check_gemm_workload(g, w, rows, cols)


@pytest.mark.slow
def test_workload_gemm_4096_f16(g):
    """FP16 operands and output at full size: sampled entries plus every edge band."""
    w = workloads.WORKLOADS["gemm_4096_f16"]
    A, B, _ = workloads.inputs_for(w)
    C = torch.full((w.M, w.N), float("nan"), dtype=torch.float16, device="cuda")
    g.gemm(A.cuda(), B.cuda(), C)
    torch.cuda.synchronize()
    rows, cols = workloads.sample_entries(w.M, w.N, w.seed)
    ref, ab = oracle.gemm_entries(A, B, rows, cols)
    tol = oracle.gemm_tolerance(ref, ab, 1.0, 0.0, out_f16=True)
    assert_within(to_f64(C)[rows, cols], ref, tol, w.name)
    assert_status_ok(g)


@pytest.mark.slow
def test_workload_gemm_batched(g):
    """Eight 2048^3 problems in one call: sampled entries plus edge bands of
    every matrix, each against the oracle on its own operands."""
    w = workloads.WORKLOADS["gemm_batched_8x2048"]
    A, B, _ = workloads.inputs_for(w)
    C = torch.full((w.batch, w.M, w.N), float("nan"), dtype=torch.bfloat16, device="cuda")
    g.gemm(A.cuda(), B.cuda(), C)
    torch.cuda.synchronize()
    got = to_f64(C)
    for b in range(w.batch):
        rows, cols = workloads.sample_entries(w.M, w.N, w.seed + b, count=16384, edge=128)
        ref, ab = oracle.gemm_entries(A[b], B[b], rows, cols)
        tol = oracle.gemm_tolerance(ref, ab, 1.0, 0.0, out_bf16=True)
        assert_within(got[b][rows, cols], ref, tol, f"{w.name}[{b}]")
    assert_status_ok(g)


def check_gate_up(g, M, N, K, seed, dist_w, rows=None, cols=None):
    X, Wg, Wu = workloads.gate_up_inputs(M, N, K, seed, ("normal", 1.0), dist_w)
    Y = torch.full((M, N), float("nan"), dtype=torch.bfloat16, device="cuda")
    g.gate_up_silu(X.cuda(), Wg.cuda(), Wu.cuda(), Y)
    torch.cuda.synchronize()
    if rows is None:
        rr, cc = np.meshgrid(np.arange(M), np.arange(N), indexing="ij")
        rows, cols = rr.ravel(), cc.ravel()
    res = oracle.gate_up_entries(X, Wg, Wu, rows, cols)
    got = to_f64(Y)[rows, cols]
    assert_within(got, res["y"], oracle.gate_up_tolerance(res), f"gate_up {M}x{N}x{K}")
    assert_status_ok(g)


@pytest.mark.parametrize("M,N,K", [(128, 128, 64), (200, 296, 104), (513, 1000, 640)])
def test_gate_up_ragged(g, M, N, K):
    check_gate_up(g, M, N, K, seed=M + N, dist_w=("normal", 1.0 / np.sqrt(K)))


@pytest.mark.parametrize("M,N,K", [(1, 296, 640), (7, 1000, 2048), (16, 1160, 4160), (16, 128, 64)])
@pytest.mark.parametrize("splits", ["planned", "1", "3"])
def test_gate_up_decode(g, monkeypatch, M, N, K, splits):
    """M <= 16 on the split-K kernel: ragged weight rows, K tails, and K split
    into pieces whose gate and up partials are summed apart before silu(g)*u."""
    if splits != "planned":
        monkeypatch.setenv("GB3_SKINNY_SPLITS", splits)
    p = g.gate_up_plan(M, N, K)
    assert p["kernel_name"] == "skinny_gate_up"
    if splits != "planned":
        kb = -(-K // 64)
        assert p["split_k"] == -(-kb // -(-kb // min(int(splits), kb)))
    check_gate_up(g, M, N, K, seed=M + N + K, dist_w=("normal", 1.0 / np.sqrt(K)))


@pytest.mark.slow
def test_workload_skinny_gate_up(g):
    """Full size, every entry."""
    w = workloads.WORKLOADS["skinny_gate_up_16x14336x4096"]
    assert g.gate_up_plan(w.M, w.N, w.K)["kernel_name"] == "skinny_gate_up"
    check_gate_up(g, w.M, w.N, w.K, w.seed, w.dist_b)


def test_gate_up_decode_matches_tiled_kernel(g, monkeypatch):
    """The decode path and the tiled gate/up kernel agree within tolerance of
    the oracle on the same inputs, and the decode path is deterministic."""
    M, N, K = 16, 2000, 3072
    X, Wg, Wu = workloads.gate_up_inputs(M, N, K, 81, ("normal", 1.0), ("normal", 1.0 / 55))
    Xd, Wgd, Wud = X.cuda(), Wg.cuda(), Wu.cuda()
    outs = [g.gate_up_silu(Xd, Wgd, Wud) for _ in range(2)]
    monkeypatch.setenv("GB3_GATE_UP_SKINNY", "0")
    assert g.gate_up_plan(M, N, K)["kernel_name"] == "gate_up"
    tiled = g.gate_up_silu(Xd, Wgd, Wud)
    torch.cuda.synchronize()
    assert torch.equal(outs[0].view(torch.int16), outs[1].view(torch.int16))
    rr, cc = np.meshgrid(np.arange(M), np.arange(N), indexing="ij")
    res = oracle.gate_up_entries(X, Wg, Wu, rr.ravel(), cc.ravel())
    tol = oracle.gate_up_tolerance(res)
    for name, y in (("decode", outs[0]), ("tiled", tiled)):
        assert_within(to_f64(y)[rr.ravel(), cc.ravel()], res["y"], tol, name)
    assert_status_ok(g)


@pytest.mark.slow
def test_workload_gate_up(g):
    w = workloads.WORKLOADS["gate_up_4096x14336x4096"]
    rows, cols = workloads.sample_entries(w.M, w.N, w.seed)
    check_gate_up(g, w.M, w.N, w.K, w.seed, w.dist_b, rows, cols)


# ---------------------------------------------------------------------------
# Edge cases and contracts
# ---------------------------------------------------------------------------
@pytest.mark.parametrize("K", [1, 16, 72, 2000])
def test_k_tails(g, K):
    M, N = 260, 300
    lda = max(8, (K + 7) // 8 * 8)
    A, B, _ = workloads.gemm_inputs(M, N, K, K, ("uniform",), ("uniform",))
    Ap = torch.zeros((M, lda), dtype=torch.bfloat16)
    Bp = torch.zeros((N, lda), dtype=torch.bfloat16)
    Ap[:, :K] = A
    Bp[:, :K] = B
    Ad, Bd = Ap.cuda()[:, :K], Bp.cuda()[:, :K]   # row pitch lda > K
    Cd = torch.empty((M, N), dtype=torch.float32, device="cuda")
    g.gemm(Ad, Bd, Cd)
    torch.cuda.synchronize()
    ref, ab = oracle.gemm_full(A, B)
    assert_within(to_f64(Cd), ref, oracle.gemm_tolerance(ref, ab, 1.0, 0.0), f"K={K}")


def test_leading_dimensions_larger_than_extents(g):
    M, N, K = 300, 260, 200
    A, B, C = workloads.gemm_inputs(M, N, K, 5, ("uniform",), ("uniform",), ("normal", 1.0))
    Abig = torch.zeros((M, K + 40), dtype=torch.bfloat16, device="cuda")
    Bbig = torch.zeros((N, K + 24), dtype=torch.bfloat16, device="cuda")
    Cbig = torch.full((M, N + 12), 7.0, dtype=torch.float32, device="cuda")
    Abig[:, :K] = A.cuda()
    Bbig[:, :K] = B.cuda()
    Cbig[:, :N] = C.cuda()
    g.gemm(Abig[:, :K], Bbig[:, :K], Cbig[:, :N], alpha=-1.0, beta=0.5)
    torch.cuda.synchronize()
    ref, ab = oracle.gemm_full(A, B, alpha=-1.0, beta=0.5, C=C)
    out = to_f64(Cbig)
    assert_within(out[:, :N], ref, oracle.gemm_tolerance(ref, ab, -1.0, 0.5, C.numpy()), "ld")
    assert np.all(out[:, N:] == 7.0)   # padding columns untouched


def test_beta_zero_does_not_read_nan_C(g):
    A, B, _ = workloads.gemm_inputs(256, 512, 256, 9, ("uniform",), ("uniform",))
    for dt in (torch.float32, torch.bfloat16):
        out = run_gemm(g, A, B, out_dtype=dt, fill=float("nan"))
        assert torch.isfinite(out).all()


def test_k_zero_scales_C(g):
    M, N = 70, 92
    C = torch.randn(M, N)
    Cd = C.cuda()
    A = torch.empty((M, 0), dtype=torch.bfloat16, device="cuda")
    B = torch.empty((N, 0), dtype=torch.bfloat16, device="cuda")
    g.gemm(A, B, Cd, alpha=3.0, beta=-2.0)
    torch.cuda.synchronize()
    assert torch.equal(Cd.cpu(), -2.0 * C)
    Cd = torch.full((M, N), float("nan"), device="cuda")
    g.gemm(A, B, Cd, beta=0.0)
    torch.cuda.synchronize()
    assert torch.equal(Cd.cpu(), torch.zeros(M, N))


def test_empty_problems_are_noops(g):
    A = torch.empty((0, 64), dtype=torch.bfloat16, device="cuda")
    B = torch.ones((32, 64), dtype=torch.bfloat16, device="cuda")
    C = torch.empty((0, 32), dtype=torch.float32, device="cuda")
    g.gemm(A, B, C)
    A = torch.ones((32, 64), dtype=torch.bfloat16, device="cuda")
    B = torch.empty((0, 64), dtype=torch.bfloat16, device="cuda")
    C = torch.empty((32, 0), dtype=torch.float32, device="cuda")
    g.gemm(A, B, C)
    torch.cuda.synchronize()
    assert_status_ok(g)


def test_modified_inputs_reuse_cached_descriptor(g):
    M, N, K = 256, 512, 512
    A, B, _ = int_inputs(M, N, K, 31)
    Ad, Bd = A.cuda(), B.cuda()
    Cd = torch.empty((M, N), dtype=torch.float32, device="cuda")
    g.gemm(Ad, Bd, Cd)
    Ad.mul_(-1)                    # same address, new values
    g.gemm(Ad, Bd, Cd)
    torch.cuda.synchronize()
    ref, _ = oracle.gemm_full(A, B)
    assert np.array_equal(to_f64(Cd), -ref)


def test_new_pointer_forces_new_descriptor(g):
    M, N, K = 200, 300, 128
    A1, B, _ = int_inputs(M, N, K, 32)
    A2, _, _ = int_inputs(M, N, K, 33)
    Bd = B.cuda()
    outs = []
    for A in (A1, A2, A1):
        Cd = torch.empty((M, N), dtype=torch.float32, device="cuda")
        g.gemm(A.cuda(), Bd, Cd)
        outs.append(Cd)
    torch.cuda.synchronize()
    for A, out in zip((A1, A2, A1), outs):
        ref, _ = oracle.gemm_full(A, B)
        assert np.array_equal(to_f64(out), ref)


@pytest.mark.parametrize("M", [512, 16])
def test_cuda_graph_capture_and_replay(g, M):
    N, K = 768, 1024
    A, B, _ = int_inputs(M, N, K, 34)
    Ad, Bd = A.cuda(), B.cuda()
    Cd = torch.empty((M, N), dtype=torch.bfloat16, device="cuda")
    g.gemm(Ad, Bd, Cd)      # eager call first: sets up descriptors and workspace
    torch.cuda.synchronize()
    eager = Cd.clone()
    Cd.zero_()
    s = torch.cuda.Stream()
    graph = torch.cuda.CUDAGraph()
    with torch.cuda.stream(s):
        with torch.cuda.graph(graph, stream=s):
            g.gemm(Ad, Bd, Cd, stream=s)
    for _ in range(3):
        Cd.zero_()
        graph.replay()
    torch.cuda.synchronize()
    assert torch.equal(Cd, eager)
    Ad.mul_(2)               # graph replay sees new values at the same address
    graph.replay()
    torch.cuda.synchronize()
    ref, _ = oracle.gemm_full(A, B, alpha=2.0)
    assert np.array_equal(bits(Cd.cpu()), oracle.round_to_bf16_bits(ref))


@pytest.mark.parametrize("M,K", [(512, 1024), (16, 2048)])
def test_sharding_over_N_matches_full_result(g, M, K):
    """Independent column shards (the multi-GPU split, run one after another
    here) concatenate to the unsharded result."""
    N, shards = 1536, 4
    A, B, _ = workloads.gemm_inputs(M, N, K, 35, ("normal", 1.0), ("normal", 1.0))
    Ad, Bd = A.cuda(), B.cuda()
    full = torch.empty((M, N), dtype=torch.float32, device="cuda")
    g.gemm(Ad, Bd, full)
    parts = torch.empty((M, N), dtype=torch.float32, device="cuda")
    w = N // shards
    for s in range(shards):
        g.gemm(Ad, Bd[s * w:(s + 1) * w], parts[:, s * w:(s + 1) * w])
    torch.cuda.synchronize()
    ref, ab = oracle.gemm_full(A, B)
    tol = oracle.gemm_tolerance(ref, ab, 1.0, 0.0)
    assert_within(to_f64(parts), ref, tol, "sharded")
    assert_within(to_f64(full), ref, tol, "full")
    if M > 16:   # tiled path: the per-entry K order does not depend on N
        assert torch.equal(parts, full)


def test_repeated_calls_are_deterministic(g):
    w = workloads.WORKLOADS["skinny_16x28672x8192"]
    A, B, _ = workloads.gemm_inputs(16, 4096, 8192, 36, ("normal", 1.0), ("normal", 0.01))
    Ad, Bd = A.cuda(), B.cuda()
    outs = []
    for _ in range(3):
        C = torch.empty((16, 4096), dtype=torch.float32, device="cuda")
        g.gemm(Ad, Bd, C)
        outs.append(C)
    torch.cuda.synchronize()
    assert torch.equal(outs[0], outs[1]) and torch.equal(outs[1], outs[2])
    del w


def test_plan_matches_device(g):
    p = g.plan(4096, 4096, 4096)
    props = torch.cuda.get_device_properties(0)
    assert p["grid"] == min(p["tiles"], props.multi_processor_count)
    assert (props.major, props.minor) == (10, 3)


def test_bounded_wait_reports_timeout(g):
    """A pipeline wait that nothing completes gives up after its limit and
    leaves GEMM_ERR_TIMEOUT in the device status word; the context stays
    usable."""
    from dense_bf16_gemm_gb300 import _native
    assert_status_ok(g)
    st = _native.gemm_selftest_wait_timeout(20_000_000, torch.cuda.current_stream().cuda_stream)
    assert st == 0
    st, site = g.device_status()
    assert st == _native.GEMM_ERR_TIMEOUT and site == 7
    st, site = g.device_status()        # reading clears the word
    assert st == 0
    # and the GPU still computes
    A, B, _ = int_inputs(128, 256, 64, 3)
    out = run_gemm(g, A, B, out_dtype=torch.float32)
    ref, _ = oracle.gemm_full(A, B)
    assert np.array_equal(to_f64(out), ref)


def test_gemm_pipeline_abort_path(g, monkeypatch):
    """A GEMM pipeline whose TMA producer stops after two k-blocks (the M <= 16
    kernel's self-test hook): the MMA thread's wait for the third runs out,
    every CTA leaves through its abort path (epilogue warps leave, the issued
    copies and MMAs are drained, Tensor Memory is freed), the status word names
    the MMA thread's wait (site 2), C is untouched, and the context still
    computes, the split-K kernel's arrival counters included."""
    from dense_bf16_gemm_gb300 import _native
    assert_status_ok(g)
    M, N, K = 16, 1024, 1024
    A, B, _ = int_inputs(M, N, K, 11)
    Ad, Bd = A.cuda(), B.cuda()
    Cd = torch.full((M, N), 7.0, dtype=torch.bfloat16, device="cuda")
    stream = torch.cuda.current_stream().cuda_stream
    st = _native.gemm_selftest_pipeline_timeout(M, N, K, Ad.data_ptr(), K, Bd.data_ptr(), K,
                                                Cd.data_ptr(), N, 2, stream)
    assert st == 0
    torch.cuda.synchronize()
    st, site = g.device_status()
    assert st == _native.GEMM_ERR_TIMEOUT and site == 2
    assert_status_ok(g)                 # reading cleared the word
    assert bool((Cd.float() == 7.0).all())
    # the same problem on the split-K kernel, forced to split K in 4 (so its
    # workspace and arrival counters are used), twice
    monkeypatch.setenv("GB3_GEMM_SMALL_M", "0")
    monkeypatch.setenv("GB3_SKINNY_SPLITS", "4")
    p = g.plan(M, N, K, torch.float32)
    assert p["kernel_name"] == "skinny_splitk" and p["split_k"] == 4
    ref, _ = oracle.gemm_full(A, B)
    for _ in range(2):
        out = run_gemm(g, A, B, out_dtype=torch.float32)
        assert np.array_equal(to_f64(out), ref)
    assert_status_ok(g)


@pytest.mark.parametrize("width", ["256", "224"])
@pytest.mark.parametrize("M,N,K", [(300, 520, 200), (512, 1000, 1000), (2000, 712, 136)])
@pytest.mark.parametrize("out_dtype", [torch.float32, torch.bfloat16])
def test_pair_widths_bit_exact(g, monkeypatch, width, M, N, K, out_dtype):
    """Every compiled CTA-pair tile width, forced, on integer inputs."""
    monkeypatch.setenv("GB3_GEMM_PAIR_TILE_N", width)
    p = g.plan(M, N, K, out_dtype)
    assert p["kernel_name"] == "pair" and p["tile_n"] == int(width)
    A, B, _ = int_inputs(M, N, K, seed=M + 3 * N + K)
    ref, _ = oracle.gemm_full(A, B)
    out = run_gemm(g, A, B, out_dtype=out_dtype)
    if out_dtype == torch.float32:
        assert np.array_equal(to_f64(out), ref)
    else:
        assert np.array_equal(bits(out.cpu()), oracle.round_to_bf16_bits(ref))
    assert_status_ok(g)


@pytest.mark.parametrize("pieces", ["2", "3", "5"])
@pytest.mark.parametrize("M,N,K", [(512, 1000, 1000), (300, 520, 704), (1000, 712, 2048)])
@pytest.mark.parametrize("out_dtype", [torch.float32, torch.bfloat16])
@pytest.mark.parametrize("ring", ["1", "0"])
def test_split_k_pieces_bit_exact(g, monkeypatch, pieces, M, N, K, out_dtype, ring):
    """Every pair tile cut into K pieces whose partials are summed by the last
    piece (which reads C through the staging ring, or with the register loads
    it replaced); integer inputs keep every partial exact."""
    monkeypatch.setenv("GB3_GEMM_SPLIT_ALL", pieces)
    monkeypatch.setenv("GB3_GEMM_C_RING", ring)
    p = g.plan(M, N, K, out_dtype)
    kb = -(-K // 64)
    kbp = -(-kb // min(int(pieces), kb))
    assert p["kernel_name"] == "pair" and p["split_k"] == -(-kb // kbp)   # pieces that get work
    A, B, C = int_inputs(M, N, K, seed=M + N + 7 * K)
    Cq = C.to(out_dtype)
    ref, _ = oracle.gemm_full(A, B, alpha=2.0, beta=-0.5, C=Cq.to(torch.float32))
    out = run_gemm(g, A, B, C=Cq, alpha=2.0, beta=-0.5, out_dtype=out_dtype)
    if out_dtype == torch.float32:
        assert np.array_equal(to_f64(out), ref)
    else:
        assert np.array_equal(bits(out.cpu()), oracle.round_to_bf16_bits(ref))
    assert_status_ok(g)


def test_split_k_is_deterministic_and_within_tolerance(g, monkeypatch):
    monkeypatch.setenv("GB3_GEMM_SPLIT_ALL", "4")
    M, N, K = 768, 1024, 4096
    A, B, _ = workloads.gemm_inputs(M, N, K, 51, ("normal", 1.0), ("normal", 1.0))
    Ad, Bd = A.cuda(), B.cuda()
    outs = []
    for _ in range(3):
        C = torch.empty((M, N), dtype=torch.float32, device="cuda")
        g.gemm(Ad, Bd, C)
        outs.append(C)
    torch.cuda.synchronize()
    assert torch.equal(outs[0], outs[1]) and torch.equal(outs[0], outs[2])
    ref, ab = oracle.gemm_full(A, B)
    assert_within(to_f64(outs[0]), ref, oracle.gemm_tolerance(ref, ab, 1.0, 0.0), "split 4")
    assert_status_ok(g)


@pytest.mark.parametrize("pieces", ["2", "3"])
def test_gate_up_split_k(g, monkeypatch, pieces):
    monkeypatch.setenv("GB3_GEMM_SPLIT_ALL", pieces)
    assert g.gate_up_plan(512, 640, 1024)["split_k"] == int(pieces)
    check_gate_up(g, 512, 640, 1024, seed=52, dist_w=("normal", 1.0 / 32))


# ---------------------------------------------------------------------------
# Batched GEMM (3-D descriptors) and FP16 operands / outputs
# ---------------------------------------------------------------------------
def batched_int_inputs(batch, M, N, K, seed, dtype):
    g_ = torch.Generator().manual_seed(seed)
    A = torch.randint(-2, 3, (batch, M, K), generator=g_).to(dtype)
    B = torch.randint(-2, 3, (batch, N, K), generator=g_).to(dtype)
    C = torch.randint(-3, 4, (batch, M, N), generator=g_).to(torch.float32)
    return A, B, C


def padded(t, rows_pad, cols_pad, fill):
    """Copy of a (b, r, c) CPU tensor into a CUDA buffer with extra rows and
    columns per matrix (so strides exceed the extents); returns (view, buffer)."""
    b, r, c = t.shape
    buf = torch.full((b, r + rows_pad, c + cols_pad), fill, dtype=t.dtype, device="cuda")
    buf[:, :r, :c] = t.cuda()
    return buf[:, :r, :c], buf


@pytest.mark.parametrize("M,N,K", [(300, 520, 200), (100, 264, 128), (7, 520, 1000)])
@pytest.mark.parametrize("out_dtype", [torch.float32, torch.bfloat16])
def test_batched_bit_exact_with_padded_strides(g, M, N, K, out_dtype):
    batch = 3
    A, B, C = batched_int_inputs(batch, M, N, K, M + N, torch.bfloat16)
    Cq = C.to(out_dtype)
    Ad, _ = padded(A, 5, 24, 7.0)     # pad values would show up if rows leaked
    Bd, _ = padded(B, 3, 8, -5.0)
    Cd, Cbuf = padded(Cq, 4, 16, 1024.0)
    g.gemm(Ad, Bd, Cd, alpha=2.0, beta=-0.5)
    torch.cuda.synchronize()
    for b in range(batch):
        ref, _ = oracle.gemm_full(A[b], B[b], alpha=2.0, beta=-0.5, C=Cq[b].to(torch.float32))
        if out_dtype == torch.float32:
            assert np.array_equal(to_f64(Cd[b]), ref), b
        else:
            assert np.array_equal(bits(Cd[b].cpu()), oracle.round_to_bf16_bits(ref)), b
    # padding rows and columns of C untouched
    pad_rows = Cbuf[:, M:, :].float().cpu()
    pad_cols = Cbuf[:, :, N:].float().cpu()
    assert torch.all(pad_rows == 1024.0) and torch.all(pad_cols == 1024.0)
    assert_status_ok(g)


def test_batched_plan_counts_every_matrix(g):
    p1 = g.batched_plan(1, 1024, 1024, 4096)
    p8 = g.batched_plan(8, 1024, 1024, 4096)
    assert p8["kernel_name"] == p1["kernel_name"] == "pair"
    assert p8["tiles"] >= 8 * (1024 // 256) * -(-1024 // p8["tile_n"])


@pytest.mark.parametrize("M,N,K", [(300, 520, 200), (64, 264, 136), (5, 1000, 2048)])
@pytest.mark.parametrize("out_dtype", [torch.float32, torch.float16, torch.bfloat16])
def test_f16_operands_bit_exact(g, M, N, K, out_dtype):
    A, B, C = batched_int_inputs(1, M, N, K, 3 * M + K, torch.float16)
    A, B, C = A[0], B[0], C[0]
    Cq = C.to(out_dtype)
    ref, _ = oracle.gemm_full(A, B, alpha=1.0, beta=0.5, C=Cq.to(torch.float32))
    out = run_gemm(g, A, B, C=Cq, alpha=1.0, beta=0.5, out_dtype=out_dtype)
    if out_dtype == torch.float32:
        assert np.array_equal(to_f64(out), ref)
    elif out_dtype == torch.float16:
        assert np.array_equal(bits(out.cpu()), oracle.round_to_f16_bits(ref))
    else:
        assert np.array_equal(bits(out.cpu()), oracle.round_to_bf16_bits(ref))
    assert_status_ok(g)


def test_f16_random_inputs_within_tolerance(g):
    M, N, K = 1000, 1536, 3072
    gen = torch.Generator().manual_seed(61)
    A = torch.randn(M, K, generator=gen).to(torch.float16)
    B = (torch.randn(N, K, generator=gen) / 32).to(torch.float16)
    out = run_gemm(g, A, B, out_dtype=torch.float16)
    ref, ab = oracle.gemm_full(A, B)
    tol = oracle.gemm_tolerance(ref, ab, 1.0, 0.0, out_f16=True)
    assert_within(to_f64(out), ref, tol, "fp16")
    assert_status_ok(g)


def test_batched_f16_split_pieces(g, monkeypatch):
    monkeypatch.setenv("GB3_GEMM_SPLIT_ALL", "2")
    batch, M, N, K = 2, 512, 768, 1024
    A, B, _ = batched_int_inputs(batch, M, N, K, 62, torch.float16)
    Cd = torch.empty((batch, M, N), dtype=torch.float32, device="cuda")
    g.gemm(A.cuda(), B.cuda(), Cd)
    torch.cuda.synchronize()
    for b in range(batch):
        ref, _ = oracle.gemm_full(A[b], B[b])
        assert np.array_equal(to_f64(Cd[b]), ref), b
    assert_status_ok(g)


# ---------------------------------------------------------------------------
# beta != 0 on CTA pairs: C is loaded with TMA into a ring of staging slots a
# few boxes ahead and each box is computed in place.  The register path
# (GB3_GEMM_C_RING=0) is the one it replaced; both must give the oracle's bits.
# ---------------------------------------------------------------------------
RING_SHAPES = [
    (300, 520, 200),     # one tile per pair; ragged rows and columns
    (2000, 3000, 136),   # two tiles on some pairs: the look-ahead crosses a tile
    (4000, 3896, 72),    # four tiles per pair: every slot reused many times
    (2304, 4136, 64),    # last column tile 40 (or 104) columns wide: partial and empty boxes
]


@pytest.mark.parametrize("width", ["256", "224"])
@pytest.mark.parametrize("M,N,K", RING_SHAPES)
@pytest.mark.parametrize("out_dtype", [torch.float32, torch.bfloat16, torch.float16])
def test_c_ring_bit_exact(g, monkeypatch, width, M, N, K, out_dtype):
    monkeypatch.setenv("GB3_GEMM_PAIR_TILE_N", width)
    monkeypatch.setenv("GB3_GEMM_TAIL_SPLIT", "0")   # whole tiles: the look-ahead cursor alone
    monkeypatch.setenv("GB3_GEMM_BALANCED", "0")
    A, B, C = int_inputs(M, N, K, seed=M + 5 * N + K)
    Cq = C.to(out_dtype)
    ref, _ = oracle.gemm_full(A, B, alpha=2.0, beta=-0.5, C=Cq.to(torch.float32))
    if out_dtype == torch.float32:
        want = ref
    elif out_dtype == torch.float16:
        want = oracle.round_to_f16_bits(ref)
    else:
        want = oracle.round_to_bf16_bits(ref)
    for ring in ("1", "0"):
        monkeypatch.setenv("GB3_GEMM_C_RING", ring)
        out = run_gemm(g, A, B, C=Cq, alpha=2.0, beta=-0.5, out_dtype=out_dtype)
        got = to_f64(out) if out_dtype == torch.float32 else bits(out.cpu())
        assert np.array_equal(got, want), f"ring={ring}"
    assert_status_ok(g)


def test_c_ring_matches_register_path_on_random_inputs(g, monkeypatch):
    """Same FP32 operations in the same order on both paths: identical bits."""
    M, N, K = 3000, 5000, 2000
    A, B, C = workloads.gemm_inputs(M, N, K, 71, ("normal", 1.0), ("normal", 1.0), ("normal", 1.0))
    Ad, Bd = A.cuda(), B.cuda()
    outs = {}
    for ring in ("1", "0"):
        monkeypatch.setenv("GB3_GEMM_C_RING", ring)
        Cd = C.cuda()
        g.gemm(Ad, Bd, Cd, alpha=0.75, beta=1.5)
        outs[ring] = Cd
    torch.cuda.synchronize()
    assert torch.equal(outs["1"], outs["0"])
    rows = np.random.default_rng(71).choice(M, 64, replace=False)
    ref, ab = oracle.gemm_entries(A, B, np.repeat(rows, N), np.tile(np.arange(N), rows.size),
                                  alpha=0.75, beta=1.5, C=C)
    got = to_f64(outs["1"])[np.repeat(rows, N), np.tile(np.arange(N), rows.size)]
    cm = C.numpy()[np.repeat(rows, N), np.tile(np.arange(N), rows.size)]
    assert_within(got, ref, oracle.gemm_tolerance(ref, ab, 0.75, 1.5, cm), "ring 3000x5000x2000")
    assert_status_ok(g)


@pytest.mark.parametrize("out_dtype", [torch.float32, torch.float16])
def test_c_ring_batched_padded(g, monkeypatch, out_dtype):
    """The third TMA coordinate (matrix of the batch) and a padded pitch of C
    on the ring's loads; padding of C untouched."""
    monkeypatch.setenv("GB3_GEMM_TAIL_SPLIT", "0")
    monkeypatch.setenv("GB3_GEMM_BALANCED", "0")
    batch, M, N, K = 3, 600, 1000, 136
    A, B, C = batched_int_inputs(batch, M, N, K, 72, torch.float16)
    Cq = C.to(out_dtype)
    Cd, Cbuf = padded(Cq, 4, 16, 1024.0)
    g.gemm(A.cuda(), B.cuda(), Cd, alpha=2.0, beta=-0.5)
    torch.cuda.synchronize()
    for b in range(batch):
        ref, _ = oracle.gemm_full(A[b], B[b], alpha=2.0, beta=-0.5, C=Cq[b].to(torch.float32))
        if out_dtype == torch.float32:
            assert np.array_equal(to_f64(Cd[b]), ref), b
        else:
            assert np.array_equal(bits(Cd[b].cpu()), oracle.round_to_f16_bits(ref)), b
    assert torch.all(Cbuf[:, M:, :].float().cpu() == 1024.0)
    assert torch.all(Cbuf[:, :, N:].float().cpu() == 1024.0)
    assert_status_ok(g)


@pytest.mark.parametrize("out_dtype", [torch.float32, torch.bfloat16])
def test_c_ring_with_split_tail(g, monkeypatch, out_dtype):
    """A planned split tail: the pieces' last arrivals load C on demand, then
    the whole tiles run the look-ahead cursor, in one launch."""
    monkeypatch.setenv("GB3_GEMM_BALANCED", "0")
    M, N, K = 2048, 2560, 3072
    p = g.plan(M, N, K, out_dtype)
    assert p["kernel_name"] == "pair" and p["split_k"] > 1
    A, B, C = int_inputs(M, N, K, seed=73)
    Cq = C.to(out_dtype)
    ref, _ = oracle.gemm_full(A, B, alpha=2.0, beta=-0.5, C=Cq.to(torch.float32))
    want = ref if out_dtype == torch.float32 else oracle.round_to_bf16_bits(ref)
    for ring in ("1", "0"):
        monkeypatch.setenv("GB3_GEMM_C_RING", ring)
        out = run_gemm(g, A, B, C=Cq, alpha=2.0, beta=-0.5, out_dtype=out_dtype)
        got = to_f64(out) if out_dtype == torch.float32 else bits(out.cpu())
        assert np.array_equal(got, want), f"ring={ring}"
    assert_status_ok(g)


# ---------------------------------------------------------------------------
# Balanced division of the CTA-pair kernels: every pair takes one contiguous
# range of the tiles' k-blocks; a tile cut by a range boundary is summed from
# its pieces by the last one to arrive.  Integer inputs keep every partial
# exact, so the result must equal the oracle bit for bit.
# ---------------------------------------------------------------------------
BALANCED_SHAPES = [
    (2304, 4136, 200),   # 153 tiles of 256 columns: ranges of ~8 k-blocks over 4-k-block tiles
    (4000, 3896, 72),    # 256 tiles, 2 k-blocks each: most tiles cut
    (3000, 5000, 264),   # the ragged workload's tiles with a short K (5 k-blocks, a K tail)
    (1300, 15000, 192),  # 6 x 59 tiles, 3 k-blocks
]


def split_tiles_planned(p, M, N):
    tiles = -(-M // 256) * -(-N // p["tile_n"])
    return p["tiles"] - tiles     # every cut tile adds one unit


@pytest.mark.parametrize("M,N,K", BALANCED_SHAPES)
@pytest.mark.parametrize("out_dtype", [torch.float32, torch.bfloat16])
@pytest.mark.parametrize("beta", [0.0, -0.5])
def test_balanced_division_bit_exact(g, monkeypatch, M, N, K, out_dtype, beta):
    monkeypatch.setenv("GB3_GEMM_BALANCED", "1")
    p = g.plan(M, N, K, out_dtype)
    assert p["kernel_name"] == "pair" and p["split_k"] >= 2 and split_tiles_planned(p, M, N) > 0
    A, B, C = int_inputs(M, N, K, seed=M + N + 3 * K)
    Cq = C.to(out_dtype) if beta != 0.0 else None
    ref, _ = oracle.gemm_full(A, B, alpha=2.0, beta=beta,
                              C=Cq.to(torch.float32) if Cq is not None else None)
    want = ref if out_dtype == torch.float32 else oracle.round_to_bf16_bits(ref)
    out = run_gemm(g, A, B, C=Cq, alpha=2.0, beta=beta, out_dtype=out_dtype)
    got = to_f64(out) if out_dtype == torch.float32 else bits(out.cpu())
    assert np.array_equal(got, want)
    assert_status_ok(g)


@pytest.mark.parametrize("width", ["256", "224"])
def test_balanced_division_random_inputs_within_tolerance(g, monkeypatch, width):
    """The ragged workload's shape on random inputs: the balanced division
    (pieces summed in K order by the last arrival) and the plan without it
    both sit within the bound, and the balanced result is identical from
    call to call."""
    monkeypatch.setenv("GB3_GEMM_PAIR_TILE_N", width)
    M, N, K = 3000, 5000, 2000
    A, B, C = workloads.gemm_inputs(M, N, K, 2, ("uniform",), ("uniform",), ("normal", 1.0))
    Ad, Bd = A.cuda(), B.cuda()
    outs = []
    for mode in ("1", "1", "0"):
        monkeypatch.setenv("GB3_GEMM_BALANCED", mode)
        Cd = C.cuda()
        g.gemm(Ad, Bd, Cd, alpha=0.5, beta=2.0)
        outs.append(Cd)
    torch.cuda.synchronize()
    assert torch.equal(outs[0], outs[1])
    rows = np.random.default_rng(81).choice(M, 48, replace=False)
    rr, cc = np.repeat(rows, N), np.tile(np.arange(N), rows.size)
    ref, ab = oracle.gemm_entries(A, B, rr, cc, alpha=0.5, beta=2.0, C=C)
    tol = oracle.gemm_tolerance(ref, ab, 0.5, 2.0, C.numpy()[rr, cc])
    for mode, o in (("balanced", outs[0]), ("whole tiles", outs[2])):
        assert_within(to_f64(o)[rr, cc], ref, tol, f"{mode} {width}")
    assert_status_ok(g)


def test_balanced_division_gate_up(g, monkeypatch):
    monkeypatch.setenv("GB3_GEMM_BALANCED", "1")
    M, N, K = 1024, 2600, 320           # 4 x 21 = 84 tiles of 128 output columns
    p = g.gate_up_plan(M, N, K)
    assert p["kernel_name"] == "pair_gate_up" and p["split_k"] >= 2
    check_gate_up(g, M, N, K, seed=83, dist_w=("normal", 1.0 / np.sqrt(K)))


def test_balanced_division_batched_f16(g, monkeypatch):
    """Ranges cross matrix boundaries of a batch: a tile's coordinates come
    from its index alone, so a range may end in one matrix and go on in the
    next."""
    monkeypatch.setenv("GB3_GEMM_BALANCED", "1")
    batch, M, N, K = 4, 1000, 2000, 200  # 4 x 4 x 8 = 128 tiles
    A, B, C = batched_int_inputs(batch, M, N, K, 84, torch.float16)
    Cd = C.cuda()
    g.gemm(A.cuda(), B.cuda(), Cd, alpha=2.0, beta=-0.5)
    torch.cuda.synchronize()
    for b in range(batch):
        ref, _ = oracle.gemm_full(A[b], B[b], alpha=2.0, beta=-0.5, C=C[b])
        assert np.array_equal(to_f64(Cd[b]), ref), b
    assert_status_ok(g)


def test_balanced_division_row_stats(g, monkeypatch):
    monkeypatch.setenv("GB3_GEMM_BALANCED", "1")
    M, N, K = 2304, 4136, 200           # 9 x 17 = 153 tiles of 4 k-blocks
    A, B, _ = workloads.gemm_inputs(M, N, K, 85, ("int", -2, 2), ("int", -2, 2))
    Cd = torch.full((M, N), float("nan"), dtype=torch.float32, device="cuda")
    Cd, rs, rmax, rmin = g.gemm_row_stats(A.cuda(), B.cuda(), Cd)
    torch.cuda.synchronize()
    ref = oracle.gemm_row_stats(A, B, np.arange(M))
    assert np.array_equal(to_f64(Cd), ref["values"])
    assert np.array_equal(to_f64(rs), ref["sum"])
    assert np.array_equal(to_f64(rmax), ref["max"])
    assert np.array_equal(to_f64(rmin), ref["min"])
    assert_status_ok(g)


# ---------------------------------------------------------------------------
# strips: the tail wave's 256-column tiles cut along N into four 64-column
# strips of the whole K (an MMA of N = 64 per strip, its own B boxes of 32
# rows per CTA, and the epilogue over its 64 columns).
# ---------------------------------------------------------------------------
STRIP_SHAPES = [
    (300, 520, 200),     # 6 tiles, 24 strips; of the last column block only strip 0 is inside C
    (1000, 712, 1000),   # 12 tiles, 48 strips
    (256, 256, 8),       # one tile, K below one k-block
    (3000, 5000, 264),   # 240 tiles: 3 waves, then 12 tiles as 48 strips; a K tail
    (2304, 4136, 200),   # 153 tiles: 2 waves, then 1 tile (its N ragged) as 4 strips
]


def strips_planned(p, M, N):
    tiles = -(-M // 256) * -(-N // 256)
    return p["tile_n"] == 256 and p["split_k"] == 1 and p["tiles"] > tiles and \
        (p["tiles"] - tiles) % 3 == 0


@pytest.mark.parametrize("M,N,K", STRIP_SHAPES)
@pytest.mark.parametrize("out_dtype", [torch.float32, torch.bfloat16])
@pytest.mark.parametrize("beta", [0.0, -0.5])
def test_strips_bit_exact(g, monkeypatch, M, N, K, out_dtype, beta):
    monkeypatch.setenv("GB3_GEMM_STRIPS", "1")
    monkeypatch.setenv("GB3_GEMM_PAIR_TILE_N", "256")
    monkeypatch.setenv("GB3_GEMM_BALANCED", "0")
    p = g.plan(M, N, K, out_dtype)
    assert p["kernel_name"] == "pair" and strips_planned(p, M, N), p
    A, B, C = int_inputs(M, N, K, seed=M + 2 * N + K)
    Cq = C.to(out_dtype) if beta != 0.0 else None
    ref, _ = oracle.gemm_full(A, B, alpha=2.0, beta=beta,
                              C=Cq.to(torch.float32) if Cq is not None else None)
    want = ref if out_dtype == torch.float32 else oracle.round_to_bf16_bits(ref)
    out = run_gemm(g, A, B, C=Cq, alpha=2.0, beta=beta, out_dtype=out_dtype)
    got = to_f64(out) if out_dtype == torch.float32 else bits(out.cpu())
    assert np.array_equal(got, want)
    assert_status_ok(g)


def test_strips_batched_f16(g, monkeypatch):
    """Strips of tiles of different matrices of a batch, FP16 operands."""
    monkeypatch.setenv("GB3_GEMM_STRIPS", "1")
    monkeypatch.setenv("GB3_GEMM_PAIR_TILE_N", "256")
    monkeypatch.setenv("GB3_GEMM_BALANCED", "0")
    batch, M, N, K = 2, 512, 1000, 200   # 2 x 2 x 4 = 16 tiles, all as strips
    A, B, C = batched_int_inputs(batch, M, N, K, 85, torch.float16)
    Cd = C.cuda()
    g.gemm(A.cuda(), B.cuda(), Cd, alpha=2.0, beta=-0.5)
    torch.cuda.synchronize()
    for b in range(batch):
        ref, _ = oracle.gemm_full(A[b], B[b], alpha=2.0, beta=-0.5, C=C[b])
        assert np.array_equal(to_f64(Cd[b]), ref), b
    assert_status_ok(g)


def test_strips_random_inputs_match_whole_tiles(g, monkeypatch):
    """The ragged workload (3000 x 5000 x 2000, alpha 0.5, beta 2, FP32 C) as
    planned (strips of its 12 tail tiles): within the bound of the oracle on
    sampled rows, identical from call to call, and identical to the same
    tiles run whole (an element's sum over K does not depend on the MMA's N)."""
    monkeypatch.setenv("GB3_GEMM_BALANCED", "0")
    M, N, K = 3000, 5000, 2000
    A, B, C = workloads.gemm_inputs(M, N, K, 2, ("uniform",), ("uniform",), ("normal", 1.0))
    Ad, Bd = A.cuda(), B.cuda()
    assert strips_planned(g.plan(M, N, K, torch.float32), M, N)
    outs = []
    for strips in ("-1", "-1", "0"):
        monkeypatch.setenv("GB3_GEMM_STRIPS", strips)
        monkeypatch.setenv("GB3_GEMM_PAIR_TILE_N", "256")
        Cd = C.cuda()
        g.gemm(Ad, Bd, Cd, alpha=0.5, beta=2.0)
        outs.append(Cd)
    torch.cuda.synchronize()
    assert torch.equal(outs[0], outs[1])
    assert torch.equal(outs[0], outs[2])
    rows = np.random.default_rng(86).choice(M, 48, replace=False)
    rr, cc = np.repeat(rows, N), np.tile(np.arange(N), rows.size)
    ref, ab = oracle.gemm_entries(A, B, rr, cc, alpha=0.5, beta=2.0, C=C)
    tol = oracle.gemm_tolerance(ref, ab, 0.5, 2.0, C.numpy()[rr, cc])
    assert_within(to_f64(outs[0])[rr, cc], ref, tol, "strips")
    assert_status_ok(g)


@pytest.mark.parametrize("beta", [0.0, 0.5])
def test_strips_f16_output(g, monkeypatch, beta):
    """Strips writing FP16 output (the 16-bit epilogue with its FP16 packing),
    with and without C read through the ring."""
    monkeypatch.setenv("GB3_GEMM_STRIPS", "1")
    monkeypatch.setenv("GB3_GEMM_PAIR_TILE_N", "256")
    monkeypatch.setenv("GB3_GEMM_BALANCED", "0")
    M, N, K = 1000, 712, 1000
    A, B, C = batched_int_inputs(1, M, N, K, 91, torch.float16)
    A, B, C = A[0], B[0], C[0]
    Cq = C.to(torch.float16) if beta != 0.0 else None
    ref, _ = oracle.gemm_full(A, B, alpha=1.0, beta=beta,
                              C=Cq.to(torch.float32) if Cq is not None else None)
    out = run_gemm(g, A, B, C=Cq, alpha=1.0, beta=beta, out_dtype=torch.float16)
    assert np.array_equal(bits(out.cpu()), oracle.round_to_f16_bits(ref))
    assert_status_ok(g)


def test_strips_under_graph_capture(g):
    """A plan with strips (the ragged workload's shape with a short K) captured
    into a CUDA graph on a fresh stream replays to the eager result: strips
    need no workspace, so nothing is allocated during capture."""
    M, N, K = 3000, 5000, 264
    assert strips_planned(g.plan(M, N, K, torch.float32), M, N)
    A, B, C = int_inputs(M, N, K, 35)
    Ad, Bd, C0 = A.cuda(), B.cuda(), C.cuda()
    Cd = C0.clone()
    g.gemm(Ad, Bd, Cd, alpha=2.0, beta=-0.5)
    torch.cuda.synchronize()
    eager = Cd.clone()
    s = torch.cuda.Stream()
    graph = torch.cuda.CUDAGraph()
    Cd.copy_(C0)
    torch.cuda.synchronize()
    with torch.cuda.stream(s):
        with torch.cuda.graph(graph, stream=s):
            g.gemm(Ad, Bd, Cd, alpha=2.0, beta=-0.5, stream=s)
    for _ in range(2):
        Cd.copy_(C0)
        graph.replay()
    torch.cuda.synchronize()
    assert torch.equal(Cd, eager)
    ref, _ = oracle.gemm_full(A, B, alpha=2.0, beta=-0.5, C=C)
    assert np.array_equal(to_f64(Cd), ref)
    assert_status_ok(g)


# the balanced division after data-parallel waves (GB3_GEMM_BALANCED=2): all
# whole waves but the last run whole tiles, the rest is divided into ranges
HYBRID_SHAPES = [
    (4096, 4096, 512),   # 256 tiles: 2 waves whole, 104 tiles (8 k-blocks each) divided
    (3000, 5000, 264),   # 240 tiles: 2 waves whole, 88 tiles divided; a K tail
    (2304, 4136, 200),   # 153 tiles: 1 wave whole, 77 tiles divided
]


@pytest.mark.parametrize("M,N,K", HYBRID_SHAPES)
@pytest.mark.parametrize("out_dtype", [torch.float32, torch.bfloat16])
@pytest.mark.parametrize("beta", [0.0, -0.5])
def test_balanced_after_whole_waves_bit_exact(g, monkeypatch, M, N, K, out_dtype, beta):
    monkeypatch.setenv("GB3_GEMM_BALANCED", "2")
    monkeypatch.setenv("GB3_GEMM_PAIR_TILE_N", "256")
    p = g.plan(M, N, K, out_dtype)
    tiles = -(-M // 256) * -(-N // 256)
    assert p["kernel_name"] == "pair" and p["split_k"] >= 2 and p["tiles"] > tiles
    A, B, C = int_inputs(M, N, K, seed=M + N + 5 * K)
    Cq = C.to(out_dtype) if beta != 0.0 else None
    ref, _ = oracle.gemm_full(A, B, alpha=2.0, beta=beta,
                              C=Cq.to(torch.float32) if Cq is not None else None)
    want = ref if out_dtype == torch.float32 else oracle.round_to_bf16_bits(ref)
    out = run_gemm(g, A, B, C=Cq, alpha=2.0, beta=beta, out_dtype=out_dtype)
    got = to_f64(out) if out_dtype == torch.float32 else bits(out.cpu())
    assert np.array_equal(got, want)
    assert_status_ok(g)


def test_balanced_after_whole_waves_random_and_deterministic(g, monkeypatch):
    monkeypatch.setenv("GB3_GEMM_BALANCED", "2")
    M, N, K = 4096, 4096, 4096
    A, B, _ = workloads.gemm_inputs(M, N, K, 3, ("uniform",), ("uniform",), None)
    Ad, Bd = A.cuda(), B.cuda()
    outs = []
    for _ in range(2):
        Cd = torch.empty((M, N), dtype=torch.float32, device="cuda")
        g.gemm(Ad, Bd, Cd)
        outs.append(Cd)
    torch.cuda.synchronize()
    assert torch.equal(outs[0], outs[1])
    rows = np.random.default_rng(87).choice(M, 24, replace=False)
    rr, cc = np.repeat(rows, N), np.tile(np.arange(N), rows.size)
    ref, ab = oracle.gemm_entries(A, B, rr, cc)
    tol = oracle.gemm_tolerance(ref, ab, 1.0, 0.0, None)
    assert_within(to_f64(outs[0])[rr, cc], ref, tol, "balanced after whole waves")
    assert_status_ok(g)
