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
