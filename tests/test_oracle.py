"""Pins of the CPU oracle to facts that do not come from the oracle itself:
closed forms, identities, brute force on tiny shapes written independently
here, and library routines (numpy float64 matmul, torch's BF16 rounding)."""
import math
import struct

import numpy as np
import pytest
import torch

import oracle
import workloads

ONE_BF16 = 0x3F80  # 1.0 in BF16


def bits(t: torch.Tensor) -> np.ndarray:
    return t.contiguous().view(torch.int16).numpy().view(np.uint16)


def py_bf16(b: int) -> float:
    """BF16 bits -> float, via struct (independent of the oracle's decoder)."""
    return struct.unpack("<f", struct.pack("<I", (int(b) & 0xFFFF) << 16))[0]


def brute_gemm(A, B, alpha, beta, C):
    """Triple loop in Python floats (binary64)."""
    a, b = bits(A), bits(B)
    M, K = a.shape
    N = b.shape[0]
    out = [[0.0] * N for _ in range(M)]
    for m in range(M):
        for n in range(N):
            s = 0.0
            for k in range(K):
                s += py_bf16(a[m, k]) * py_bf16(b[n, k])
            v = alpha * s
            if beta != 0.0:
                v += beta * float(C[m, n])
            out[m][n] = v
    return np.array(out)


def rand_inputs(M, N, K, seed, dist=("uniform",)):
    A, B, C = workloads.gemm_inputs(M, N, K, seed, dist, dist, ("normal", 1.0))
    return A, B, C


# ---------------------------------------------------------------------------
# GEMM
# ---------------------------------------------------------------------------
@pytest.mark.parametrize("M,N,K", [(1, 1, 1), (3, 5, 7), (17, 13, 33), (40, 9, 130)])
def test_ones_times_ones_is_K(M, N, K):
    A = np.full((M, K), ONE_BF16, np.uint16)
    B = np.full((N, K), ONE_BF16, np.uint16)
    v, ab = oracle.gemm_full(A, B)
    assert np.all(v == K)
    assert np.all(ab == K)


def test_identity_left_and_right():
    A, B, _ = rand_inputs(24, 24, 24, seed=11)
    eye = np.where(np.eye(24, dtype=bool), ONE_BF16, 0).astype(np.uint16)
    # A . I = A   (I stored (N, K) is its own transpose)
    v, _ = oracle.gemm_full(A, eye)
    assert np.array_equal(v, oracle.bf16_bits_to_f64(bits(A)))
    # I . B = B^T-storage: (I.B)(m, n) = b(m, n) = B[n, m]
    v, _ = oracle.gemm_full(eye, B)
    assert np.array_equal(v, oracle.bf16_bits_to_f64(bits(B)).T)


def test_identity_rectangular_selects_columns():
    # A (M,K) times a K x N selector picking column j -> k = perm[j]
    A, _, _ = rand_inputs(9, 1, 31, seed=12)
    perm = np.array([30, 0, 7, 7, 19])
    sel = np.zeros((perm.size, 31), np.uint16)
    sel[np.arange(perm.size), perm] = ONE_BF16
    v, _ = oracle.gemm_full(A, sel)
    assert np.array_equal(v, oracle.bf16_bits_to_f64(bits(A))[:, perm])


def test_transpose_identity_by_storage_swap():
    A, B, _ = rand_inputs(37, 23, 71, seed=13)
    v, ab = oracle.gemm_full(A, B)
    vt, abt = oracle.gemm_full(B, A)   # B^T . A^T with the same storage
    assert np.allclose(vt, v.T, rtol=0, atol=1e-12 * np.max(ab))
    assert np.array_equal(abt, ab.T) or np.allclose(abt, ab.T, rtol=1e-15)


@pytest.mark.parametrize("alpha", [2.0, 0.25, -4.0])
def test_alpha_power_of_two_scales_exactly(alpha):
    A, B, _ = rand_inputs(20, 30, 50, seed=14)
    v1, _ = oracle.gemm_full(A, B)
    va, _ = oracle.gemm_full(A, B, alpha=alpha)
    assert np.array_equal(va, alpha * v1)


def test_beta_term_is_separable():
    A, B, C = rand_inputs(20, 30, 50, seed=15)
    v0, ab = oracle.gemm_full(A, B, alpha=0.5)
    vb, _ = oracle.gemm_full(A, B, alpha=0.5, beta=2.0, C=C)
    expect = v0 + 2.0 * C.numpy().astype(np.float64)
    assert np.allclose(vb, expect, rtol=0, atol=1e-13 * (np.max(ab) + 10))
    # alpha = 0 leaves exactly beta * C
    vz, _ = oracle.gemm_full(A, B, alpha=0.0, beta=-3.0, C=C)
    assert np.array_equal(vz, -3.0 * C.numpy().astype(np.float64))


def test_beta_zero_never_reads_C():
    A, B, C = rand_inputs(8, 8, 8, seed=16)
    nanC = torch.full_like(C, float("nan"))
    v, _ = oracle.gemm_full(A, B, beta=0.0, C=nanC)
    assert np.isfinite(v).all()


@pytest.mark.parametrize("M,N,K", [(1, 1, 1), (3, 5, 7), (17, 13, 33)])
def test_matches_bruteforce_triple_loop(M, N, K):
    A, B, C = rand_inputs(M, N, K, seed=M * 100 + N)
    alpha, beta = 0.75, -1.5
    v, _ = oracle.gemm_full(A, B, alpha=alpha, beta=beta, C=C)
    ref = brute_gemm(A, B, alpha, beta, C.numpy())
    assert np.allclose(v, ref, rtol=1e-14, atol=1e-14)


def test_matches_numpy_float64_matmul():
    A, B, C = rand_inputs(64, 48, 300, seed=17, dist=("normal", 1.0))
    a = oracle.bf16_bits_to_f64(bits(A))
    b = oracle.bf16_bits_to_f64(bits(B))
    v, ab = oracle.gemm_full(A, B, alpha=1.5, beta=0.5, C=C)
    ref = 1.5 * (a @ b.T) + 0.5 * C.numpy().astype(np.float64)
    assert np.allclose(v, ref, rtol=0, atol=1e-12 * np.max(ab))
    assert np.allclose(ab, np.abs(a) @ np.abs(b).T, rtol=1e-13)


def test_entries_match_full():
    A, B, C = rand_inputs(50, 70, 90, seed=18)
    v, ab = oracle.gemm_full(A, B, alpha=-0.5, beta=2.0, C=C)
    rows = np.array([0, 49, 13, 13, 7])
    cols = np.array([0, 69, 5, 6, 68])
    ve, abe = oracle.gemm_entries(A, B, rows, cols, alpha=-0.5, beta=2.0, C=C)
    assert np.array_equal(ve, v[rows, cols])
    assert np.array_equal(abe, ab[rows, cols])


def test_dropped_term_or_transposed_operand_is_caught():
    """Planted mistakes (made here, on the CPU) fail the brute-force pin."""
    A, B, _ = rand_inputs(6, 6, 6, seed=19)
    ref = brute_gemm(A, B, 1.0, 0.0, None)
    a = oracle.bf16_bits_to_f64(bits(A))
    b = oracle.bf16_bits_to_f64(bits(B))
    good = a @ b.T
    dropped = a[:, :-1] @ b[:, :-1].T        # last k term lost
    transposed = a @ b                       # B read as (K, N) storage
    sign = a @ (-b).T + 2 * a[:, :1] @ b[:, :1].T  # one term with the wrong sign
    assert np.allclose(good, ref, rtol=1e-13, atol=1e-13)
    for wrong in (dropped, transposed, sign):
        assert not np.allclose(wrong, ref, rtol=1e-6, atol=1e-6)


# ---------------------------------------------------------------------------
# SiLU and gate/up
# ---------------------------------------------------------------------------
def test_silu_closed_forms():
    assert oracle.silu(0.0) == 0.0
    for t in [0.1, 0.5, 1.0, 2.3994, 7.0, 30.0]:
        # silu(t) - silu(-t) = t
        assert math.isclose(oracle.silu(t) - oracle.silu(-t), t, rel_tol=1e-14, abs_tol=1e-15)
        # independent tanh form: t * (1 + tanh(t/2)) / 2
        assert math.isclose(oracle.silu(t), t * 0.5 * (1.0 + math.tanh(t / 2.0)), rel_tol=1e-14)
    assert math.isclose(oracle.silu(60.0) / 60.0, 1.0, rel_tol=1e-20 + 1e-15)
    assert abs(oracle.silu(-60.0)) < 1e-20
    # the Lipschitz constant used by the tolerance bounds |silu'|
    ts = np.linspace(-20, 20, 200001)
    d = np.gradient(ts / (1 + np.exp(-ts)), ts)
    assert np.max(np.abs(d)) <= oracle.SILU_LIPSCHITZ


def brute_gate_up(X, Wg, Wu):
    x, g_, u_ = bits(X), bits(Wg), bits(Wu)
    M, K = x.shape
    N = g_.shape[0]
    out = np.zeros((M, N))
    for m in range(M):
        for n in range(N):
            g = sum(py_bf16(x[m, k]) * py_bf16(g_[n, k]) for k in range(K))
            u = sum(py_bf16(x[m, k]) * py_bf16(u_[n, k]) for k in range(K))
            out[m, n] = g * 0.5 * (1.0 + math.tanh(g / 2.0)) * u
    return out


def test_gate_up_matches_bruteforce():
    X, Wg, Wu = workloads.gate_up_inputs(6, 7, 19, seed=21, dist_w=("normal", 0.5))
    rows, cols = np.meshgrid(np.arange(6), np.arange(7), indexing="ij")
    res = oracle.gate_up_entries(X, Wg, Wu, rows.ravel(), cols.ravel())
    ref = brute_gate_up(X, Wg, Wu).ravel()
    assert np.allclose(res["y"], ref, rtol=1e-13, atol=1e-14)


def test_gate_up_against_gemm_oracle_and_numpy():
    X, Wg, Wu = workloads.gate_up_inputs(33, 40, 70, seed=22, dist_w=("normal", 0.2))
    x = oracle.bf16_bits_to_f64(bits(X))
    g = x @ oracle.bf16_bits_to_f64(bits(Wg)).T
    u = x @ oracle.bf16_bits_to_f64(bits(Wu)).T
    rows, cols = np.meshgrid(np.arange(33), np.arange(40), indexing="ij")
    res = oracle.gate_up_entries(X, Wg, Wu, rows.ravel(), cols.ravel())
    ref = (g * 0.5 * (1 + np.tanh(g / 2)) * u).ravel()
    assert np.allclose(res["g"], g.ravel(), rtol=0, atol=1e-12)
    assert np.allclose(res["u"], u.ravel(), rtol=0, atol=1e-12)
    assert np.allclose(res["y"], ref, rtol=1e-12, atol=1e-13)


# ---------------------------------------------------------------------------
# BF16 encoding
# ---------------------------------------------------------------------------
def torch_bf16_bits(x32: np.ndarray) -> np.ndarray:
    t = torch.from_numpy(np.ascontiguousarray(x32, dtype=np.float32)).to(torch.bfloat16)
    return t.view(torch.int16).numpy().view(np.uint16)


def test_round_to_bf16_matches_torch_on_fp32_patterns():
    rng = np.random.default_rng(5)
    pats = rng.integers(0, 2**32, size=1_000_000, dtype=np.uint64).astype(np.uint32)
    x = pats.view(np.float32)
    x = x[np.isfinite(x)]
    mine = oracle.round_to_bf16_bits(x.astype(np.float64))
    assert np.array_equal(mine, torch_bf16_bits(x))


def test_round_to_bf16_ties_and_edges():
    # exact ties between two BF16 neighbours go to the even mantissa
    base = np.arange(0, 1 << 16, 97, dtype=np.uint32) << 16
    ties = (base | 0x8000).view(np.float32)
    ties = ties[np.isfinite(ties)]
    assert np.array_equal(oracle.round_to_bf16_bits(ties.astype(np.float64)), torch_bf16_bits(ties))
    specials = np.array([0.0, -0.0, 1.0, -1.0, 2.0**-133, 2.0**-134, 3 * 2.0**-135,
                         2.0**-126, 3.3895313892515355e38, 3.3961e38, 1e39, -1e39,
                         float("inf"), float("-inf")])
    got = oracle.round_to_bf16_bits(specials)
    with np.errstate(over="ignore"):
        want = torch_bf16_bits(specials.astype(np.float32))
    assert np.array_equal(got, want)
    assert oracle.round_to_bf16_bits(np.array([float("nan")]))[0] == 0x7FC0


def test_bf16_widening_matches_torch():
    b = np.arange(0, 1 << 16, dtype=np.uint32).astype(np.uint16)
    t = torch.from_numpy(b.view(np.int16)).view(torch.bfloat16).to(torch.float64).numpy()
    mine = oracle.bf16_bits_to_f64(b)
    fin = np.isfinite(t)
    assert np.array_equal(mine[fin], t[fin])
    assert np.array_equal(np.isnan(mine), np.isnan(t))


def test_half_ulp_bounds_rounding_error():
    assert oracle.bf16_half_ulp(1.0) == 2.0**-8
    assert oracle.bf16_half_ulp(1.99) == 2.0**-8
    assert oracle.bf16_half_ulp(2.0) == 2.0**-7
    assert oracle.bf16_half_ulp(0.75) == 2.0**-9
    assert oracle.bf16_half_ulp(0.0) == 2.0**-134
    rng = np.random.default_rng(6)
    x = rng.standard_normal(200000) * np.exp2(rng.integers(-30, 30, 200000))
    err = np.abs(oracle.bf16_bits_to_f64(oracle.round_to_bf16_bits(x)) - x)
    assert np.all(err <= oracle.bf16_half_ulp(x))


def test_tolerance_flags_a_planted_error():
    A, B, C = rand_inputs(16, 16, 64, seed=23, dist=("normal", 1.0))
    v, ab = oracle.gemm_full(A, B, alpha=0.5, beta=2.0, C=C)
    tol = oracle.gemm_tolerance(v, ab, 0.5, 2.0, C.numpy(), out_bf16=False)
    assert np.all(tol > 0)
    bad = v.copy()
    bad[3, 4] += 2.0 * tol[3, 4]
    assert np.sum(np.abs(bad - v) > tol) == 1


# ---------------------------------------------------------------------------
# FP16 operands and outputs
# ---------------------------------------------------------------------------
def py_f16(b: int) -> float:
    """binary16 bits -> float via struct's 'e' format (independent of numpy)."""
    return struct.unpack("<e", struct.pack("<H", int(b) & 0xFFFF))[0]


def test_decode16_every_pattern():
    pats = np.arange(1 << 16, dtype=np.uint32).astype(np.uint16)
    f16_np = pats.view(np.float16).astype(np.float64)
    bf16_t = torch.from_numpy(pats.view(np.int16)).view(torch.bfloat16).to(torch.float64).numpy()
    for i in range(0, 1 << 16, 7):            # a seventh of them through ctypes
        a, b = oracle.decode16(i, True), oracle.decode16(i, False)
        assert (a == f16_np[i]) or (math.isnan(a) and math.isnan(f16_np[i]))
        assert (b == bf16_t[i]) or (math.isnan(b) and math.isnan(bf16_t[i]))
        if not math.isnan(a):
            assert a == py_f16(i)


def test_round_to_f16_matches_struct_half_rounding():
    rng = np.random.default_rng(7)
    x = rng.standard_normal(20000) * np.exp2(rng.integers(-26, 16, 20000))
    # exact ties between neighbours, including subnormals, must go to even
    ties = np.array([1 + 2.0**-11, 1 + 3 * 2.0**-11, 2.0**-24 * 1.5, 2.0**-24 * 2.5,
                     65504 + 16, 65520.0, -65520.0, 2.0**-25, 3 * 2.0**-26])
    for v in np.concatenate([x, ties]):
        try:
            want = struct.unpack("<H", struct.pack("<e", float(v)))[0]
        except OverflowError:            # struct refuses values that round to inf
            want = 0x7C00 if v > 0 else 0xFC00
        assert oracle.round_to_f16_bits(v) == want, v


def test_f16_half_ulp_bounds_rounding_error():
    assert oracle.f16_half_ulp(1.0) == 2.0**-11
    assert oracle.f16_half_ulp(1024.0) == 0.5
    assert oracle.f16_half_ulp(0.0) == 2.0**-25
    rng = np.random.default_rng(8)
    x = rng.standard_normal(100000) * np.exp2(rng.integers(-20, 14, 100000))
    err = np.abs(oracle.f16_bits_to_f64(oracle.round_to_f16_bits(x)) - x)
    assert np.all(err <= oracle.f16_half_ulp(x))


def test_f16_operands_match_bruteforce_and_numpy():
    g = torch.Generator().manual_seed(9)
    A = (torch.rand(7, 19, generator=g) * 4 - 2).to(torch.float16)
    B = (torch.rand(5, 19, generator=g) * 4 - 2).to(torch.float16)
    v, ab = oracle.gemm_full(A, B)
    a = A.view(torch.int16).numpy().view(np.uint16)
    b = B.view(torch.int16).numpy().view(np.uint16)
    brute = np.array([[sum(py_f16(a[m, k]) * py_f16(b[n, k]) for k in range(19))
                       for n in range(5)] for m in range(7)])
    assert np.allclose(v, brute, rtol=1e-14, atol=1e-14)
    assert np.allclose(v, A.double().numpy() @ B.double().numpy().T, rtol=1e-13, atol=1e-13)
    # the same bits read as BF16 give a different product: the flag is honoured
    vb, _ = oracle.gemm_full(a, b)
    assert not np.allclose(vb, v)
    ve, _ = oracle.gemm_entries(A, B, [0, 6], [4, 0])
    assert np.array_equal(ve, v[[0, 6], [4, 0]])


# ---------------------------------------------------------------------------
# Row normalisation ("Tiles and shared memory", section "A complete kernel")
# ---------------------------------------------------------------------------
@pytest.mark.parametrize("c,eps", [(3.0, 1e-6), (1e-4, 1e-6), (3.0, 0.5), (-2.5, 0.0)])
def test_rms_norm_constant_row_closed_form(c, eps):
    """A row of D equal values c: mean square c^2, so y_k = c g_k / sqrt(c^2 + eps)."""
    D = 48
    X = np.full((2, D), c, np.float32)
    G = (np.arange(D) % 7 + 1).astype(np.float32) / 4.0
    y, inv = oracle.rms_norm(X, G, eps)
    c32 = float(np.float32(c))
    want_inv = 1.0 / math.sqrt(c32 * c32 + eps)
    assert np.allclose(inv, want_inv, rtol=1e-15, atol=0)
    assert np.allclose(y, c32 * want_inv * G.astype(np.float64), rtol=1e-15, atol=0)


def test_rms_norm_one_hot_row():
    """Only x_j = c is nonzero: the mean square is c^2 / D (a sum of |x| or a
    divisor other than D would give another value)."""
    D, j, c, eps = 64, 11, 3.0, 1e-6
    X = np.zeros((1, D), np.float32)
    X[0, j] = c
    G = np.linspace(0.5, 2.0, D).astype(np.float32)
    y, inv = oracle.rms_norm(X, G, eps)
    want = c / math.sqrt(c * c / D + eps) * float(G[j])
    assert math.isclose(y[0, j], want, rel_tol=1e-15)
    assert np.count_nonzero(y) == 1


def test_rms_norm_has_unit_rms_without_eps():
    """With unit gains and eps = 0 every output row has mean square exactly 1
    (up to float64 rounding)."""
    X = torch.randn(20, 333, generator=torch.Generator().manual_seed(5)) * 7.0
    y, _ = oracle.rms_norm(X, np.ones(333, np.float32), 0.0)
    assert np.allclose((y * y).mean(axis=1), 1.0, rtol=1e-13, atol=0)


@pytest.mark.parametrize("j", [-3, 1, 5])
def test_rms_norm_power_of_two_scale_invariance(j):
    """Scaling a row by 2^j scales its root mean square by 2^j exactly, so
    with eps = 0 the result is bit-identical."""
    X = torch.randn(6, 96, generator=torch.Generator().manual_seed(6))
    G = torch.rand(96, generator=torch.Generator().manual_seed(7)) + 0.5
    y0, _ = oracle.rms_norm(X, G, 0.0)
    y1, _ = oracle.rms_norm(X * 2.0 ** j, G, 0.0)
    assert np.array_equal(y0, y1)


@pytest.mark.parametrize("dtype", [torch.bfloat16, torch.float16])
def test_rms_norm_16bit_inputs_equal_their_fp32_widening(dtype):
    X = torch.randn(9, 200, generator=torch.Generator().manual_seed(8)).to(dtype)
    G = torch.rand(200, generator=torch.Generator().manual_seed(9)) + 0.5
    y16, inv16 = oracle.rms_norm(X, G, 1e-6, rows=[0, 4, 8])
    y32, inv32 = oracle.rms_norm(X.float(), G, 1e-6, rows=[0, 4, 8])
    assert np.array_equal(y16, y32) and np.array_equal(inv16, inv32)


def _fp32_lane_rms_norm(x64, g, eps):
    """The normalisation evaluated in binary32 with 32 lanes each summing
    every 32nd element in order, then a pairwise combination of the lanes."""
    x = x64.astype(np.float32)
    D = x.shape[0]
    lanes = np.zeros(32, np.float32)
    for k in range(D):
        lanes[k % 32] = np.float32(lanes[k % 32] + x[k] * x[k])
    while lanes.size > 1:
        lanes = (lanes[: lanes.size // 2] + lanes[lanes.size // 2:]).astype(np.float32)
    ms = np.float32(lanes[0] / np.float32(D))
    inv = np.float32(np.float32(1.0) / np.sqrt(np.float32(ms + np.float32(eps))))
    return (x * inv).astype(np.float32) * g.astype(np.float32)


def test_rms_norm_tolerance_covers_fp32_evaluation():
    D = 4096
    gen = torch.Generator().manual_seed(10)
    X = (torch.randn(8, D, generator=gen) * torch.rand(8, 1, generator=gen) * 50).to(torch.bfloat16)
    G = (torch.rand(D, generator=gen) + 0.5).numpy().astype(np.float32)
    y, _ = oracle.rms_norm(X, G, 1e-6)
    tol = oracle.rms_norm_tolerance(y, D)
    xf = X.float().numpy().astype(np.float64)
    for r in range(8):
        y32 = _fp32_lane_rms_norm(xf[r], G, 1e-6).astype(np.float64)
        assert np.all(np.abs(y32 - y[r]) <= tol[r])
        # and the BF16-rounded operand stays within the gate/up perturbation bound
        yb = oracle.bf16_bits_to_f64(oracle.round_to_bf16_bits(y32))
        d = oracle.rmsnorm_gate_up_rel(D) - oracle.REL_ACC * (1 + 2.0 ** -8)
        assert np.all(np.abs(yb - y[r]) <= d * np.abs(y[r]) + 1e-300)


def test_rmsnorm_gate_up_reduces_to_gate_up_on_exact_rows():
    """Rows of +-2 have root mean square 2, so with eps = 0 and power-of-two
    gains the normalised row is +-g exactly and BF16; the projection must then
    equal the plain gate/up oracle on that row."""
    M, N, K = 6, 40, 96
    gen = torch.Generator().manual_seed(11)
    sign = torch.where(torch.rand(M, K, generator=gen) < 0.5, -1.0, 1.0)
    X = (2.0 * sign).to(torch.bfloat16)
    G = 2.0 ** torch.randint(-1, 3, (K,), generator=gen).float()
    Wg = torch.randn(N, K, generator=gen).to(torch.bfloat16)
    Wu = torch.randn(N, K, generator=gen).to(torch.bfloat16)
    Xn = (sign * G).to(torch.bfloat16)
    rows = np.repeat(np.arange(M), N)
    cols = np.tile(np.arange(N), M)
    a = oracle.rmsnorm_gate_up_entries(X, G, 0.0, Wg, Wu, rows, cols)
    b = oracle.gate_up_entries(Xn, Wg, Wu, rows, cols)
    for k in ("y", "g", "u", "abs_g", "abs_u"):
        assert np.array_equal(a[k], b[k]), k


def test_rmsnorm_gate_up_against_numpy_composition():
    M, N, K = 5, 33, 128
    gen = torch.Generator().manual_seed(12)
    X = torch.randn(M, K, generator=gen).to(torch.bfloat16)
    G = torch.rand(K, generator=gen) + 0.5
    Wg = (torch.randn(N, K, generator=gen) / 8).to(torch.bfloat16)
    Wu = (torch.randn(N, K, generator=gen) / 8).to(torch.bfloat16)
    x = X.double().numpy()
    xn = x / np.sqrt((x * x).mean(axis=1, keepdims=True) + 1e-6) * G.double().numpy()
    g = xn @ Wg.double().numpy().T
    u = xn @ Wu.double().numpy().T
    y = g / (1.0 + np.exp(-g)) * u
    rows = np.repeat(np.arange(M), N)
    cols = np.tile(np.arange(N), M)
    res = oracle.rmsnorm_gate_up_entries(X, G, 1e-6, Wg, Wu, rows, cols)
    assert np.allclose(res["y"], y.ravel(), rtol=1e-12, atol=1e-14)
    assert np.allclose(res["abs_g"], (np.abs(xn) @ np.abs(Wg.double().numpy()).T).ravel(),
                       rtol=1e-12)


# ---------------------------------------------------------------------------
# Reductions along a row of the GEMM result
# ---------------------------------------------------------------------------
def test_row_stats_of_ones_product():
    M, N, K, alpha = 3, 10, 12, -0.5
    A = np.full((M, K), ONE_BF16, np.uint16)
    B = np.full((N, K), ONE_BF16, np.uint16)
    s = oracle.gemm_row_stats(A, B, np.arange(M), alpha=alpha)
    assert np.all(s["sum"] == N * K * alpha)
    assert np.all(s["max"] == K * alpha) and np.all(s["min"] == K * alpha)


def test_row_stats_of_identity_product_are_the_rows_of_A():
    M, K = 7, 24
    A = torch.randn(M, K, generator=torch.Generator().manual_seed(13)).to(torch.bfloat16)
    I = torch.eye(K).to(torch.bfloat16)
    s = oracle.gemm_row_stats(A, I, np.arange(M))
    a = A.double().numpy()
    assert np.array_equal(s["max"], a.max(axis=1)) and np.array_equal(s["min"], a.min(axis=1))
    assert np.allclose(s["sum"], a.sum(axis=1), rtol=1e-15, atol=1e-15)


def test_row_stats_against_numpy_with_beta():
    M, N, K = 9, 31, 70
    A, B, C = rand_inputs(M, N, K, seed=14)
    rows = np.array([0, 3, 8])
    s = oracle.gemm_row_stats(A, B, rows, alpha=0.5, beta=2.0, C=C)
    v = 0.5 * (A.double().numpy() @ B.double().numpy().T) + 2.0 * C.double().numpy()
    v = v[rows]
    assert np.allclose(s["sum"], v.sum(axis=1), rtol=1e-13, atol=1e-12)
    assert np.allclose(s["max"], v.max(axis=1), rtol=1e-14)
    assert np.allclose(s["min"], v.min(axis=1), rtol=1e-14)


def test_row_stats_tolerance_flags_a_planted_error():
    M, N, K = 4, 50, 64
    A, B, _ = rand_inputs(M, N, K, seed=15)
    s = oracle.gemm_row_stats(A, B, np.arange(M))
    tol = oracle.row_stats_tolerance(s, 1.0, 0.0)
    for k in ("sum", "max", "min"):
        assert np.all(tol[k] > 0)
        assert not np.any(np.abs((s[k] + 2 * tol[k]) - s[k]) <= tol[k])
    # FP32 evaluation of the same sums stays inside the bound
    v32 = s["values"].astype(np.float32)
    assert np.all(np.abs(v32.sum(axis=1, dtype=np.float32) - s["sum"]) <= tol["sum"])


# ---------------------------------------------------------------------------
# Attention ("Tiles and shared memory", section "How long a tile lives")
# ---------------------------------------------------------------------------
def _attn_inputs(H, Nq, Nk, D, seed):
    gen = torch.Generator().manual_seed(seed)
    Q = torch.randn(H, Nq, D, generator=gen).to(torch.bfloat16)
    K = torch.randn(H, Nk, D, generator=gen).to(torch.bfloat16)
    V = torch.randn(H, Nk, D, generator=gen).to(torch.bfloat16)
    return Q, K, V


def _all_rows(H, Nq):
    hh, rr = np.meshgrid(np.arange(H), np.arange(Nq), indexing="ij")
    return hh.ravel(), rr.ravel()


def test_attention_zero_scale_is_the_mean_of_V():
    """With scale 0 every score is equal: the output is the plain mean of V."""
    Q, K, V = _attn_inputs(2, 3, 9, 8, 40)
    h, r = _all_rows(2, 3)
    res = oracle.attention_rows(Q, K, V, 0.0, h, r)
    mean = V.double().mean(dim=1).numpy()
    assert np.allclose(res["o"], mean[h], rtol=1e-14, atol=1e-15)


def test_attention_single_key_returns_its_value():
    Q, K, V = _attn_inputs(2, 4, 1, 16, 41)
    h, r = _all_rows(2, 4)
    res = oracle.attention_rows(Q, K, V, 0.7, h, r)
    assert np.array_equal(res["o"], V.double().numpy()[h, 0])


def test_attention_identical_keys_give_the_mean_of_V():
    """Equal keys give equal scores whatever the query (a wrong axis in the
    score, or a missing normalisation, would not)."""
    Q, K, V = _attn_inputs(1, 5, 6, 8, 42)
    K = K[:, :1].expand(1, 6, 8).contiguous()
    h, r = _all_rows(1, 5)
    res = oracle.attention_rows(Q, K, V, 1.3, h, r)
    assert np.allclose(res["o"], V.double().mean(dim=1).numpy()[h], rtol=1e-13, atol=1e-14)


def test_attention_dominant_key_selects_its_value():
    """One key scoring 100 above the rest carries weight 1 - O(e^-100)."""
    D, Nk = 8, 5
    Q = torch.zeros(1, 1, D)
    Q[0, 0, 0] = 10.0
    K = torch.zeros(1, Nk, D)
    K[0, 3, 0] = 10.0
    V = torch.randn(1, Nk, D, generator=torch.Generator().manual_seed(43))
    res = oracle.attention_rows(Q.to(torch.bfloat16), K.to(torch.bfloat16),
                                V.to(torch.bfloat16), 1.0, [0], [0])
    assert np.allclose(res["o"][0], V.to(torch.bfloat16).double().numpy()[0, 3], rtol=0,
                       atol=1e-40)


def test_attention_is_invariant_to_key_order():
    Q, K, V = _attn_inputs(1, 4, 11, 16, 44)
    perm = torch.randperm(11, generator=torch.Generator().manual_seed(45))
    h, r = _all_rows(1, 4)
    a = oracle.attention_rows(Q, K, V, 0.3, h, r)
    b = oracle.attention_rows(Q, K[:, perm], V[:, perm], 0.3, h, r)
    assert np.allclose(a["o"], b["o"], rtol=1e-13, atol=1e-14)


def test_attention_against_torch_float64_softmax():
    Q, K, V = _attn_inputs(3, 6, 37, 32, 46)
    h, r = _all_rows(3, 6)
    res = oracle.attention_rows(Q, K, V, 32 ** -0.5, h, r)
    s = 32 ** -0.5 * Q.double() @ K.double().transpose(1, 2)
    w = torch.softmax(s, dim=-1)
    ref = (w @ V.double()).numpy()[h, r]
    assert np.allclose(res["o"], ref, rtol=1e-12, atol=1e-14)
    assert np.allclose(res["abs_o"], (w @ V.double().abs()).numpy()[h, r], rtol=1e-12)
    amax = (Q.double().abs() @ K.double().abs().transpose(1, 2)).amax(dim=-1).numpy()[h, r]
    assert np.allclose(res["smax"], 32 ** -0.5 * amax, rtol=1e-13)


def _fp32_flash(q, k, v, scale, block=128, lag=0.0):
    """An FP32 flash loop over key blocks with BF16 probabilities, as the
    GPU computes it, in numpy (independent of the oracle).  With lag > 0 the
    maximum the probabilities are taken against moves only when a block's
    maximum exceeds it by more than lag, so probabilities reach exp(lag)."""
    q, k, v = (np.asarray(x, np.float32) for x in (q, k, v))
    m, l = np.float32(-np.inf), np.float32(0)
    acc = np.zeros(q.shape[-1], np.float32)
    for j0 in range(0, k.shape[0], block):
        s = (k[j0:j0 + block] @ q).astype(np.float32) * np.float32(scale)
        m_new = np.float32(s.max()) if s.max() > m + lag else m
        alpha = np.float32(np.exp(np.float32(m - m_new))) if m != -np.inf else np.float32(0)
        p = np.exp((s - m_new).astype(np.float32)).astype(np.float32)
        pb = oracle.bf16_bits_to_f64(oracle.round_to_bf16_bits(p)).astype(np.float32)
        l = np.float32(l * alpha + p.sum(dtype=np.float32))
        acc = (acc * alpha + pb @ v[j0:j0 + block]).astype(np.float32)
        m = m_new
    return (acc / l).astype(np.float64)


def _fp32_flash_two_chains(q, k, v, scale, block=128, lag=0.0):
    """The FP32 flash loop run as two independent chains, the even key blocks
    in one and the odd ones in the other (each with its own maximum, sum and
    accumulator, BF16 probabilities), merged at the end in FP32:
    O = (acc_0 f_0 + acc_1 f_1) / (l_0 f_0 + l_1 f_1), f_c = exp(m_c - m),
    m = max(m_0, m_1).  Numpy, independent of the oracle."""
    q, k, v = (np.asarray(x, np.float32) for x in (q, k, v))
    m = [np.float32(-np.inf)] * 2
    l = [np.float32(0)] * 2
    acc = [np.zeros(q.shape[-1], np.float32) for _ in range(2)]
    for j, j0 in enumerate(range(0, k.shape[0], block)):
        c = j % 2
        s = (k[j0:j0 + block] @ q).astype(np.float32) * np.float32(scale)
        m_new = np.float32(s.max()) if s.max() > m[c] + lag else m[c]
        alpha = np.float32(np.exp(np.float32(m[c] - m_new))) if m[c] != -np.inf else np.float32(0)
        p = np.exp((s - m_new).astype(np.float32)).astype(np.float32)
        pb = oracle.bf16_bits_to_f64(oracle.round_to_bf16_bits(p)).astype(np.float32)
        l[c] = np.float32(l[c] * alpha + p.sum(dtype=np.float32))
        acc[c] = (acc[c] * alpha + pb @ v[j0:j0 + block]).astype(np.float32)
        m[c] = m_new
    mm = max(m)
    f = [np.float32(np.exp(np.float32(mc - mm))) if mc != -np.inf else np.float32(0) for mc in m]
    num = (acc[0] * f[0] + acc[1] * f[1]).astype(np.float32)
    den = np.float32(l[0] * f[0] + l[1] * f[1])
    return (num / den).astype(np.float64)


@pytest.mark.parametrize("Nk,scale,lag", [(600, None, 0.0), (1153, None, 8.0), (520, 1.0, 8.0)])
def test_attention_tolerance_covers_two_merged_chains(Nk, scale, lag):
    """Key blocks dealt to two chains and merged at the end (lazy maxima that
    lag by up to 8 in base 2, peaked rows at scale 1): the bound still holds,
    so the merge's extra roundings are inside it."""
    H, Nq, D = 1, 24, 64
    Q, K, V = _attn_inputs(H, Nq, Nk, D, Nk)
    h, r = _all_rows(H, Nq)
    sc = D ** -0.5 if scale is None else scale
    res = oracle.attention_rows(Q, K, V, sc, h, r)
    tol = oracle.attention_tolerance(res, D, Nk, out_bf16=False)
    qf, kf, vf = Q.float().numpy(), K.float().numpy(), V.float().numpy()
    blocks = [np.arange(j0, min(j0 + 128, Nk)) for j0 in range(0, Nk, 128)]
    even, odd = np.concatenate(blocks[0::2]), np.concatenate(blocks[1::2])
    flagged = 0
    for i in range(Nq):
        got = _fp32_flash_two_chains(qf[0, i], kf[0], vf[0], sc, lag=lag * np.log(2.0))
        assert np.all(np.abs(got - res["o"][i]) <= tol[i]), i
        # a merge that weights the two chains' outputs equally is caught
        wrong = (_fp32_flash(qf[0, i], kf[0][even], vf[0][even], sc) +
                 _fp32_flash(qf[0, i], kf[0][odd], vf[0][odd], sc)) / 2
        flagged += bool(np.any(np.abs(wrong - res["o"][i]) > tol[i]))
    assert flagged >= Nq // 2


def test_attention_tolerance_covers_an_fp32_flash_loop():
    H, Nq, Nk, D = 1, 8, 600, 64
    Q, K, V = _attn_inputs(H, Nq, Nk, D, 47)
    h, r = _all_rows(H, Nq)
    res = oracle.attention_rows(Q, K, V, D ** -0.5, h, r)
    tol = oracle.attention_tolerance(res, D, Nk, out_bf16=False)
    qf, kf, vf = Q.float().numpy(), K.float().numpy(), V.float().numpy()
    for i in range(Nq):
        got = _fp32_flash(qf[0, i], kf[0], vf[0], D ** -0.5)
        assert np.all(np.abs(got - res["o"][i]) <= tol[i])
    # the bound is tight enough to flag a dropped or doubled key
    assert np.all(tol > 0)
    dropped = oracle.attention_rows(Q[:, :, :], K[:, 1:], V[:, 1:], D ** -0.5, h, r)
    assert np.any(np.abs(dropped["o"] - res["o"]) > tol)


def test_attention_tolerance_covers_probabilities_above_one():
    """Peaked rows (scale 1) whose probabilities are taken against a maximum
    that lags by up to 8 (base 2): every probability, the dominant ones
    included, carries a BF16 rounding of up to 2^-8 relative.  Some of these
    rows land between the 2^-9 and the 2^-8 forms of the bound."""
    H, Nq, Nk, D = 1, 48, 520, 64
    Q, K, V = _attn_inputs(H, Nq, Nk, D, 5)
    h, r = _all_rows(H, Nq)
    res = oracle.attention_rows(Q, K, V, 1.0, h, r)
    tol = oracle.attention_tolerance(res, D, Nk, out_bf16=False)
    qf, kf, vf = Q.float().numpy(), K.float().numpy(), V.float().numpy()
    worst = 0.0
    for i in range(Nq):
        got = _fp32_flash(qf[0, i], kf[0], vf[0], 1.0, lag=8.0 * np.log(2.0))
        err = np.abs(got - res["o"][i])
        assert np.all(err <= tol[i]), i
        worst = max(worst, float(np.max(err / res["abs_o"][i])))
    assert worst > 2.0 ** -9        # a bound with 2^-9 for BF16 would not hold here
