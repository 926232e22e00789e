"""Parity of the row operations with the CPU oracle: the reductions along each
row of a GEMM result (sum, maximum, minimum), the row normalisation, and the
gate/up projection of a normalised activation.  Every call goes through the
C ABI via the thin torch binding."""
import numpy as np
import pytest
import torch

import oracle
import workloads

pytestmark = pytest.mark.gpu

F32, BF16, F16 = torch.float32, torch.bfloat16, torch.float16


@pytest.fixture(scope="module")
def g():
    from dense_bf16_gemm_gb300 import build
    build.build()
    import dense_bf16_gemm_gb300 as lib
    lib._native.lib()
    return lib


def to_f64(t):
    return t.detach().to("cpu").to(torch.float64).numpy()


def bits(t):
    return t.detach().cpu().contiguous().view(torch.int16).numpy().view(np.uint16)


def assert_within(got, ref, tol, what):
    err = np.abs(got - ref)
    bad = ~(err <= tol)
    if bad.any():
        i = tuple(np.argwhere(bad)[0])
        raise AssertionError(f"{what}: {bad.sum()} of {bad.size} out of tolerance; first {i}: "
                             f"got {got[i]!r} ref {ref[i]!r} tol {tol[i]!r}")


def assert_status_ok(g):
    st, site = g.device_status()
    assert st == 0, f"device status {st} at wait site {site}"


# ---------------------------------------------------------------------------
# Reductions along each row of the GEMM result
# ---------------------------------------------------------------------------
def row_stats_case(g, M, N, K, seed, alpha=1.0, beta=0.0, out=F32, in_dtype=BF16, dist=None,
                   rows=None):
    dist = dist or ("uniform",)
    A, B, C = workloads.gemm_inputs(M, N, K, seed, dist, dist,
                                    ("normal", 1.0) if beta != 0.0 else None, dtype=in_dtype)
    Cq = C.to(out) if C is not None else None
    Cd = Cq.cuda() if Cq is not None else torch.full((M, N), float("nan"), dtype=out,
                                                        device="cuda")
    _, rs, rmax, rmin = g.gemm_row_stats(A.cuda(), B.cuda(), Cd, alpha=alpha, beta=beta)
    torch.cuda.synchronize()
    rows = np.arange(M) if rows is None else np.asarray(rows)
    ref = oracle.gemm_row_stats(A, B, rows, alpha=alpha, beta=beta,
                                C=Cq.float() if Cq is not None else None)
    return A, B, Cq, Cd, (to_f64(rs)[rows], to_f64(rmax)[rows], to_f64(rmin)[rows]), ref, rows


@pytest.mark.parametrize("M,N,K,out", [
    (300, 520, 200, F32),     # ragged in every dimension, one pair tile wave
    (1000, 712, 1000, BF16),  # many tiles
    (16, 1000, 4096, BF16),   # M <= 16: the tiled kernel, not the swapped one
    (100, 300, 64, F32),      # single-CTA kernel, partial column tile
])
def test_row_stats_integer_inputs_exact(g, M, N, K, out):
    """Integer entries keep every product, partial and row sum exact in FP32
    (|row sum| < 2^24), so all three reductions equal the oracle exactly."""
    A, B, C = workloads.gemm_inputs(M, N, K, 3 * M + N, ("int", -2, 2), ("int", -2, 2))
    Cd = torch.full((M, N), float("nan"), dtype=out, device="cuda")
    Cd, rs, rmax, rmin = g.gemm_row_stats(A.cuda(), B.cuda(), Cd)
    torch.cuda.synchronize()
    ref = oracle.gemm_row_stats(A, B, np.arange(M))
    assert np.max(np.abs(ref["sum"])) < 2 ** 24
    assert np.array_equal(to_f64(rs), ref["sum"])
    assert np.array_equal(to_f64(rmax), ref["max"])
    assert np.array_equal(to_f64(rmin), ref["min"])
    # C itself is the plain GEMM's result
    if out == F32:
        assert np.array_equal(to_f64(Cd), ref["values"])
    else:
        assert np.array_equal(bits(Cd), oracle.round_to_bf16_bits(ref["values"]))
    assert_status_ok(g)


def test_row_stats_alpha_beta_within_tolerance(g):
    M, N, K, alpha, beta = 300, 520, 200, 0.5, 2.0
    *_, got, ref, _ = row_stats_case(g, M, N, K, 21, alpha=alpha, beta=beta)
    tol = oracle.row_stats_tolerance(ref, alpha, beta)
    for i, k in enumerate(("sum", "max", "min")):
        assert_within(got[i], ref[k], tol[k], k)
    assert_status_ok(g)


@pytest.mark.parametrize("in_dtype,out", [(BF16, F32), (F16, F16)])
def test_row_stats_normal_inputs(g, in_dtype, out):
    M, N, K = 520, 1000, 512
    *_, got, ref, _ = row_stats_case(g, M, N, K, 22, out=out, in_dtype=in_dtype,
                                     dist=("normal", 1.0))
    tol = oracle.row_stats_tolerance(ref, 1.0, 0.0)
    for i, k in enumerate(("sum", "max", "min")):
        assert_within(got[i], ref[k], tol[k], k)
    assert_status_ok(g)


def test_row_stats_C_matches_plain_gemm_bitwise(g):
    """Same plan, same epilogue arithmetic: the reductions do not change C."""
    M, N, K = 1000, 712, 1000
    A, B, _ = workloads.gemm_inputs(M, N, K, 23, ("normal", 1.0), ("normal", 1.0))
    Ad, Bd = A.cuda(), B.cuda()
    C1 = g.gemm(Ad, Bd, out_dtype=BF16)
    C2, *_ = g.gemm_row_stats(Ad, Bd, out_dtype=BF16)
    torch.cuda.synchronize()
    assert torch.equal(C1.view(torch.int16), C2.view(torch.int16))
    assert_status_ok(g)


def test_row_stats_deterministic(g):
    M, N, K = 4096, 4096, 1024
    A, B, _ = workloads.gemm_inputs(M, N, K, 24, ("normal", 1.0), ("normal", 1.0))
    Ad, Bd = A.cuda(), B.cuda()
    r1 = g.gemm_row_stats(Ad, Bd, out_dtype=BF16)
    r2 = g.gemm_row_stats(Ad, Bd, out_dtype=BF16)
    torch.cuda.synchronize()
    for a, b in zip(r1, r2):
        assert torch.equal(a.view(torch.int32) if a.dtype == F32 else a.view(torch.int16),
                           b.view(torch.int32) if b.dtype == F32 else b.view(torch.int16))
    assert_status_ok(g)


def test_row_stats_batched(g):
    bt, M, N, K = 3, 200, 296, 128
    A, B, _ = workloads.gemm_inputs(M, N, K, 25, ("int", -2, 2), ("int", -2, 2), batch=bt)
    C, rs, rmax, rmin = g.gemm_row_stats(A.cuda(), B.cuda(), out_dtype=F32)
    torch.cuda.synchronize()
    assert rs.shape == (bt, M)
    for b in range(bt):
        ref = oracle.gemm_row_stats(A[b], B[b], np.arange(M))
        assert np.array_equal(to_f64(rs[b]), ref["sum"])
        assert np.array_equal(to_f64(rmax[b]), ref["max"])
        assert np.array_equal(to_f64(rmin[b]), ref["min"])
    assert_status_ok(g)


def test_row_stats_K0_and_N0(g):
    M, N = 70, 96
    C = torch.randn(M, N, generator=torch.Generator().manual_seed(26))
    A = torch.empty((M, 0), dtype=BF16, device="cuda")
    B = torch.empty((N, 0), dtype=BF16, device="cuda")
    Cd = C.cuda()
    _, rs, rmax, rmin = g.gemm_row_stats(A, B, Cd, alpha=1.0, beta=-0.5)
    torch.cuda.synchronize()
    v = -0.5 * C.double().numpy()          # beta * C, exact in FP32
    assert np.allclose(rs.cpu().double().numpy(), v.sum(axis=1), rtol=0, atol=1e-4)
    assert np.array_equal(rmax.cpu().double().numpy(), v.max(axis=1))
    assert np.array_equal(rmin.cpu().double().numpy(), v.min(axis=1))
    assert np.array_equal(Cd.cpu().double().numpy(), v)
    # no columns: empty reductions
    A0 = torch.empty((M, 64), dtype=BF16, device="cuda")
    B0 = torch.empty((0, 64), dtype=BF16, device="cuda")
    _, rs, rmax, rmin = g.gemm_row_stats(A0, B0, out_dtype=F32)
    torch.cuda.synchronize()
    assert torch.all(rs == 0) and torch.all(rmax == -float("inf"))
    assert torch.all(rmin == float("inf"))
    assert_status_ok(g)


@pytest.mark.slow
def test_workload_gemm_row_stats_4096(g):
    """Full size, in the configuration the benchmark times: 64 whole rows
    (the first and last 16 and 32 drawn) against the oracle."""
    w = workloads.WORKLOADS["gemm_row_stats_4096"]
    gen = np.random.default_rng(w.seed)
    rows = np.unique(np.concatenate([np.arange(16), np.arange(w.M - 16, w.M),
                                     gen.choice(w.M, 32, replace=False)]))
    *_, got, ref, _ = row_stats_case(g, w.M, w.N, w.K, w.seed, out=BF16,
                                     dist=w.dist_a, rows=rows)
    tol = oracle.row_stats_tolerance(ref, 1.0, 0.0)
    for i, k in enumerate(("sum", "max", "min")):
        assert_within(got[i], ref[k], tol[k], k)
    assert_status_ok(g)


# ---------------------------------------------------------------------------
# Row normalisation ("Tiles and shared memory", section "A complete kernel")
# ---------------------------------------------------------------------------
KIND = {F32: "f32", BF16: "bf16", F16: "f16"}


def norm_case(g, rows, D, x_dtype, y_dtype, seed, ld=None, eps=1e-6, check_rows=None):
    X, G = workloads.rms_norm_inputs(rows, D, seed, x_dtype)
    ld = ld or D
    Xd = torch.zeros((rows, ld), dtype=x_dtype, device="cuda")
    Xd[:, :D] = X.cuda()
    Yd = torch.full((rows, ld), float("nan"), dtype=y_dtype, device="cuda")
    g.rms_norm(Xd[:, :D], G.cuda(), eps, Y=Yd[:, :D])
    torch.cuda.synchronize()
    r = np.arange(rows) if check_rows is None else np.asarray(check_rows)
    ref, _ = oracle.rms_norm(X, G, eps, r)
    got = to_f64(Yd[:, :D])[r]
    tol = oracle.rms_norm_tolerance(ref, D, out_bf16=y_dtype == BF16, out_f16=y_dtype == F16)
    assert_within(got, ref, tol, f"rms_norm {rows}x{D} {KIND[x_dtype]}->{KIND[y_dtype]}")
    # the padding past D is untouched
    if ld > D:
        assert torch.isnan(Yd[:, D:].float()).all()
    return X, G, Yd


@pytest.mark.parametrize("rows,D,xd,yd,ld", [
    (37, 256, F32, F32, None),       # the pages' kernel: D = 256, FP32
    (100, 4096, BF16, BF16, None),   # whole row held in registers
    (64, 1000, F16, F32, None),
    (50, 1004, BF16, BF16, 1008),    # scalar tail of 4 elements, padded pitch
    (33, 8196, BF16, F16, 8200),     # longer than the register cache, plus a tail
    (257, 3, F32, BF16, 8),          # shorter than one vector: all scalar
    (1, 20000, F32, F32, None),      # one long row, second pass from L2
])
@pytest.mark.parametrize("row_warps", ["2", "1"])
def test_rms_norm_within_tolerance(g, monkeypatch, rows, D, xd, yd, ld, row_warps):
    """Long rows run on two warps per row by default; GB3_NORM_ROW_WARPS=1
    keeps them on one (short rows always take one)."""
    monkeypatch.setenv("GB3_NORM_ROW_WARPS", row_warps)
    norm_case(g, rows, D, xd, yd, seed=rows + D, ld=ld)
    assert_status_ok(g)


def test_rms_norm_in_place_equals_out_of_place(g):
    rows, D = 300, 4096
    X, G = workloads.rms_norm_inputs(rows, D, 31, BF16)
    Gd = G.cuda()
    Y = g.rms_norm(X.cuda(), Gd, 1e-6)
    Xi = X.cuda()
    g.rms_norm(Xi, Gd, 1e-6, Y=Xi)
    torch.cuda.synchronize()
    assert torch.equal(Y.view(torch.int16), Xi.view(torch.int16))
    assert_status_ok(g)


def test_rms_norm_eps_dominates_tiny_rows(g):
    """Rows far below sqrt(eps): inv ~ 1/sqrt(eps), so eps must enter."""
    rows, D = 16, 512
    X = torch.randn(rows, D, generator=torch.Generator().manual_seed(32)) * 1e-5
    G = torch.ones(D)
    Y = g.rms_norm(X.cuda(), G.cuda(), 0.25)
    torch.cuda.synchronize()
    ref, _ = oracle.rms_norm(X, G, 0.25)
    assert_within(to_f64(Y), ref, oracle.rms_norm_tolerance(ref, D), "eps")
    assert_status_ok(g)


@pytest.mark.slow
@pytest.mark.parametrize("name", ["rms_norm_262144x256_f32", "rms_norm_16384x4096_bf16"])
def test_workload_rms_norm(g, name):
    """Full size, as the benchmark runs it; 4096 sampled rows (the first and
    last 256 among them) against the oracle."""
    w = workloads.WORKLOADS[name]
    X, G = workloads.inputs_for(w)
    Y = g.rms_norm(X.cuda(), G.cuda(), w.eps, out_dtype=w.out_dtype)
    torch.cuda.synchronize()
    gen = np.random.default_rng(w.seed)
    rows = np.unique(np.concatenate([np.arange(256), np.arange(w.M - 256, w.M),
                                     gen.choice(w.M, 3584, replace=False)]))
    ref, _ = oracle.rms_norm(X, G, w.eps, rows)
    tol = oracle.rms_norm_tolerance(ref, w.K, out_bf16=w.out_bf16)
    assert_within(to_f64(Y)[rows], ref, tol, name)
    assert_status_ok(g)


# ---------------------------------------------------------------------------
# The gate/up projection of the normalised activation
# ---------------------------------------------------------------------------
def check_rmsnorm_gate_up(g, M, N, K, seed, rows=None, cols=None, dist_w=("normal", 0.0625)):
    X, G, Wg, Wu = workloads.rmsnorm_gate_up_inputs(M, N, K, seed, dist_w)
    Xd, Gd, Wgd, Wud = X.cuda(), G.cuda(), Wg.cuda(), Wu.cuda()
    Y, Xn = g.rmsnorm_gate_up_silu(Xd, Gd, 1e-6, Wgd, Wud)
    torch.cuda.synchronize()
    # the normalised activation is the standalone normalisation, bit for bit,
    # and the projection is the plain gate/up of it, bit for bit
    Xn2 = g.rms_norm(Xd, Gd, 1e-6, out_dtype=BF16)
    Y2 = g.gate_up_silu(Xn2, Wgd, Wud)
    torch.cuda.synchronize()
    assert torch.equal(Xn.view(torch.int16), Xn2.view(torch.int16))
    assert torch.equal(Y.view(torch.int16), Y2.view(torch.int16))
    if rows is None:
        rr, cc = np.meshgrid(np.arange(M), np.arange(N), indexing="ij")
        rows, cols = rr.ravel(), cc.ravel()
    res = oracle.rmsnorm_gate_up_entries(X, G, 1e-6, Wg, Wu, rows, cols)
    tol = oracle.gate_up_tolerance(res, rel=oracle.rmsnorm_gate_up_rel(K))
    assert_within(to_f64(Y)[rows, cols], res["y"], tol, f"rmsnorm gate/up {M}x{N}x{K}")
    # Xn against the normalisation oracle, with the BF16 output rounding
    xr = np.unique(rows)
    ref, _ = oracle.rms_norm(X, G, 1e-6, xr)
    assert_within(to_f64(Xn)[xr], ref, oracle.rms_norm_tolerance(ref, K, out_bf16=True), "Xn")
    assert_status_ok(g)


@pytest.fixture(params=["two_launches", "single_launch"])
def launches(request, monkeypatch):
    """Both forms of the normalised gate/up: the default two launches, and
    (GB3_RMSNORM_SINGLE_LAUNCH=1, M > 128) one launch of the pair gate/up
    kernel that normalises its rows of X first, with the geometry the
    standalone normalisation takes (one warp per row for K <= 1024, two
    warps for longer rows), so the bits are the same."""
    monkeypatch.setenv("GB3_RMSNORM_SINGLE_LAUNCH", "1" if request.param == "single_launch" else "0")
    return request.param


@pytest.mark.parametrize("M,N,K", [(200, 296, 256), (300, 520, 1000), (16, 256, 4096),
                                   (512, 1000, 4096), (1100, 2600, 320)])
def test_rmsnorm_gate_up(g, launches, M, N, K):
    check_rmsnorm_gate_up(g, M, N, K, seed=M + N + K)


def test_rmsnorm_gate_up_two_launches_when_forced(g, monkeypatch):
    """With the standalone normalisation forced onto one warp per long row the
    call takes the two-launch path, still bit-identical to the two steps."""
    monkeypatch.setenv("GB3_NORM_ROW_WARPS", "1")
    check_rmsnorm_gate_up(g, 300, 520, 2048, seed=91)


def test_rmsnorm_gate_up_rows_of_partial_vectors(g):
    """K = 1004 (rows of 2008 bytes, not whole 16-byte vectors) in a padded X:
    the call takes the two-launch path, bit-identical to the two steps."""
    M, N, K = 300, 520, 1004
    X, G, Wg, Wu = workloads.rmsnorm_gate_up_inputs(M, N, K, 94, ("normal", 0.0625))
    Xbuf = torch.zeros((M, 1008), dtype=torch.bfloat16, device="cuda")
    Xbuf[:, :K] = X.cuda()
    Xd = Xbuf[:, :K]
    Wgb = torch.zeros((N, 1008), dtype=torch.bfloat16, device="cuda")
    Wub = torch.zeros((N, 1008), dtype=torch.bfloat16, device="cuda")
    Wgb[:, :K], Wub[:, :K] = Wg.cuda(), Wu.cuda()
    Gd = G.cuda()
    Y, Xn = g.rmsnorm_gate_up_silu(Xd, Gd, 1e-6, Wgb[:, :K], Wub[:, :K],
                                   Xn=torch.zeros((M, 1008), dtype=torch.bfloat16,
                                                  device="cuda")[:, :K])
    Xn2 = g.rms_norm(Xd, Gd, 1e-6, Y=torch.zeros((M, 1008), dtype=BF16, device="cuda")[:, :K])
    torch.cuda.synchronize()
    assert torch.equal(Xn.contiguous().view(torch.int16), Xn2.contiguous().view(torch.int16))
    rr, cc = np.meshgrid(np.arange(M), np.arange(N), indexing="ij")
    res = oracle.rmsnorm_gate_up_entries(X, G, 1e-6, Wg, Wu, rr.ravel(), cc.ravel())
    tol = oracle.gate_up_tolerance(res, rel=oracle.rmsnorm_gate_up_rel(K))
    assert_within(to_f64(Y).ravel(), res["y"], tol, "rmsnorm gate/up K=1004")
    assert_status_ok(g)


def test_rmsnorm_gate_up_in_place(g, launches):
    """Xn may be X itself: each row is read by the threads that then write it."""
    M, N, K = 400, 704, 2048
    X, G, Wg, Wu = workloads.rmsnorm_gate_up_inputs(M, N, K, 92, ("normal", 0.0625))
    Gd, Wgd, Wud = G.cuda(), Wg.cuda(), Wu.cuda()
    Xd = X.cuda()
    Y, Xn = g.rmsnorm_gate_up_silu(Xd, Gd, 1e-6, Wgd, Wud, Xn=Xd)
    torch.cuda.synchronize()
    assert Xn.data_ptr() == Xd.data_ptr()
    Xn2 = g.rms_norm(X.cuda(), Gd, 1e-6, out_dtype=BF16)
    Y2 = g.gate_up_silu(Xn2, Wgd, Wud)
    torch.cuda.synchronize()
    assert torch.equal(Xn.view(torch.int16), Xn2.view(torch.int16))
    assert torch.equal(Y.view(torch.int16), Y2.view(torch.int16))
    assert_status_ok(g)


def test_rmsnorm_gate_up_grids_of_different_sizes_back_to_back(g, monkeypatch):
    """The single launch's grid-wide barrier counters return to zero after every
    launch, so launches with grids of different sizes (20 CTAs, then all
    resident pairs, then 20 again) each wait for exactly their own CTAs."""
    monkeypatch.setenv("GB3_RMSNORM_SINGLE_LAUNCH", "1")
    shapes = [(300, 520, 1024), (2048, 4096, 512), (300, 520, 1024)]
    for i, (M, N, K) in enumerate(shapes):
        X, G, Wg, Wu = workloads.rmsnorm_gate_up_inputs(M, N, K, 93 + i, ("normal", 0.0625))
        Xd, Gd, Wgd, Wud = X.cuda(), G.cuda(), Wg.cuda(), Wu.cuda()
        Y, Xn = g.rmsnorm_gate_up_silu(Xd, Gd, 1e-6, Wgd, Wud)
        Xn2 = g.rms_norm(Xd, Gd, 1e-6, out_dtype=BF16)
        Y2 = g.gate_up_silu(Xn2, Wgd, Wud)
        torch.cuda.synchronize()
        assert torch.equal(Xn.view(torch.int16), Xn2.view(torch.int16)), (M, N, K)
        assert torch.equal(Y.view(torch.int16), Y2.view(torch.int16)), (M, N, K)
    assert_status_ok(g)


@pytest.mark.slow
def test_workload_rmsnorm_gate_up(g):
    w = workloads.WORKLOADS["rmsnorm_gate_up_4096x14336x4096"]
    rows, cols = workloads.sample_entries(w.M, w.N, w.seed)
    check_rmsnorm_gate_up(g, w.M, w.N, w.K, w.seed, rows, cols, w.dist_b)
