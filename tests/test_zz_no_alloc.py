"""The allocation-free decode-shaped GEMM (gemm_bf16_skinny_noalloc).

It serves callers that may not allocate device memory during a call (for
example code whose memory pool must own every byte, or that cannot afford the
synchronization an allocation can cause): its split-K partial sums live in a
fixed array compiled into the library.  These tests call it through the C ABI
and check every entry against the CPU oracle, and against gemm_bf16 on the
same inputs, on calls made back to back, so that state left in the shared
array by one call cannot leak into the next.

This file is named to be collected last.
"""
import numpy as np
import pytest
import torch

import oracle
import workloads

pytestmark = pytest.mark.gpu


@pytest.fixture(scope="module")
def native():
    from dense_bf16_gemm_gb300 import _native, build
    build.build()
    _native.lib()
    return _native


def _call(fn, A, B, C, alpha, beta):
    M, K = A.shape
    N = B.shape[0]
    code = 1 if C.dtype == torch.bfloat16 else 0
    return fn(M, N, K, alpha, A.data_ptr(), A.stride(0), B.data_ptr(), B.stride(0), beta,
              C.data_ptr(), C.stride(0), code, torch.cuda.current_stream().cuda_stream)


def _stream():
    return torch.cuda.current_stream().cuda_stream


def _status_ok(native):
    st, site = native.gemm_get_device_status(_stream())
    assert st == 0, (st, site)


def _split_of(native, M, N, K, monkeypatch):
    """The split the allocation-free entry point runs: the split-K kernel's
    own plan (what gemm_bf16 plans when the small-M kernel is switched off)."""
    with monkeypatch.context() as m:
        m.setenv("GB3_GEMM_SMALL_M", "0")
        st, plan = native.gemm_bf16_plan(M, N, K, native.GEMM_OUT_BF16, 0)
    assert st == 0 and plan.as_dict()["kernel_name"] == "skinny_splitk"
    return plan.split_k


def _check_against_oracle(A, B, C0, got, alpha, beta, out_dtype):
    """Every entry within the stated bound of the oracle's FP64 result."""
    ref, ab = oracle.gemm_full(A, B, alpha=alpha, beta=beta,
                               C=C0.float().cpu() if beta != 0.0 else None)
    tol = oracle.gemm_tolerance(ref, ab, alpha, beta,
                                C0.double().cpu().numpy() if beta != 0.0 else None,
                                out_bf16=out_dtype == torch.bfloat16)
    err = np.abs(got.double().cpu().numpy() - ref)
    assert np.all(err <= tol), f"max err {err.max()} (worst ratio {np.max(err / tol)})"
    return tol


# (M, N, K, alpha, beta, seed): the decode workload's shape (split-K), a ragged
# one that reads C, one whose plan has a single split, and one with many splits.
CASES = [
    (16, 28672, 8192, 1.0, 0.0, 41),
    (5, 3000, 4096, 0.5, 2.0, 42),
    (16, 19456, 512, 1.0, -1.0, 43),
    (9, 1000, 6144, 2.0, 0.5, 44),
]


@pytest.mark.parametrize("out_dtype", [torch.bfloat16, torch.float32])
def test_noalloc_matches_gemm_bf16_on_two_calls_in_a_row(native, monkeypatch, out_dtype):
    """Each case runs twice back to back (and the cases, whose splits differ,
    follow one another), so counters or partial sums left in the shared array
    by one call would show in the next.  Every result is checked against the
    oracle, and against gemm_bf16 on the same inputs: bit for bit when both
    run the split-K kernel with the same split, else within twice the bound
    (each is within the bound of the exact result)."""
    splits = [_split_of(native, M, N, K, monkeypatch) for M, N, K, *_ in CASES]
    assert 1 in splits and len(set(splits)) >= 3, splits
    for M, N, K, alpha, beta, seed in CASES:
        A, B, C = workloads.gemm_inputs(M, N, K, seed, ("normal", 1.0),
                                        ("normal", K ** -0.5), ("normal", 1.0))
        Ad, Bd = A.cuda(), B.cuda()
        C0 = C.to(out_dtype).cuda()
        outs = []
        for _ in range(2):
            c_new = C0.clone()
            assert _call(native.gemm_bf16_skinny_noalloc, Ad, Bd, c_new, alpha, beta) == 0
            outs.append(c_new)
        c_ref = C0.clone()
        assert _call(native.gemm_bf16, Ad, Bd, c_ref, alpha, beta) == 0
        torch.cuda.synchronize()
        _status_ok(native)
        assert torch.equal(outs[0], outs[1])
        tol = _check_against_oracle(A, B, C0, outs[0], alpha, beta, out_dtype)
        diff = np.abs(outs[0].double().cpu().numpy() - c_ref.double().cpu().numpy())
        assert np.all(diff <= 2 * tol)
        with monkeypatch.context() as m:       # gemm_bf16 on the split-K kernel too
            m.setenv("GB3_GEMM_SMALL_M", "0")
            c_same = C0.clone()
            assert _call(native.gemm_bf16, Ad, Bd, c_same, alpha, beta) == 0
            torch.cuda.synchronize()
        assert torch.equal(outs[0], c_same)


def test_noalloc_k_zero_scales_C(native):
    M, N = 7, 1000
    C0 = torch.randn(M, N, generator=torch.Generator().manual_seed(45)).cuda()
    A = torch.zeros((M, 0), dtype=torch.bfloat16, device="cuda")
    B = torch.zeros((N, 0), dtype=torch.bfloat16, device="cuda")
    C = C0.clone()
    assert native.gemm_bf16_skinny_noalloc(M, N, 0, 1.0, A.data_ptr(), 1, B.data_ptr(), 1, 0.5,
                                           C.data_ptr(), N, 0, _stream()) == 0
    torch.cuda.synchronize()
    _status_ok(native)
    assert torch.equal(C, C0 * 0.5)    # beta * C, exact for a power of two


def test_noalloc_after_a_wait_that_timed_out(native):
    """A kernel that gave up leaves its status word set; reading it clears the
    word, and the next allocation-free call (which clears its own counters)
    is exact again."""
    assert native.gemm_selftest_wait_timeout(20_000_000, _stream()) == 0
    st, site = native.gemm_get_device_status(_stream())
    assert st == native.GEMM_ERR_TIMEOUT and site == 7
    M, N, K = 16, 28672, 8192
    A, B, _ = workloads.gemm_inputs(M, N, K, 46, ("normal", 1.0), ("normal", K ** -0.5))
    C = torch.full((M, N), float("nan"), dtype=torch.bfloat16, device="cuda")
    assert _call(native.gemm_bf16_skinny_noalloc, A.cuda(), B.cuda(), C, 1.0, 0.0) == 0
    torch.cuda.synchronize()
    _status_ok(native)
    _check_against_oracle(A, B, C, C, 1.0, 0.0, torch.bfloat16)


def test_noalloc_rejects_problems_larger_than_its_array(native):
    """A decode problem whose partial sums exceed the 8 MiB array is refused
    before any launch.  Real buffers are used so that nothing could touch an
    invalid address even if the call were accepted."""
    M = 16
    for N, K in ((77952, 16384), (86016, 8192), (155648, 16384), (163840, 32768)):
        st, plan = native.gemm_bf16_plan(M, N, K, native.GEMM_OUT_BF16, 0)
        assert st == 0
        if plan.split_k > 1 and plan.split_k * M * N * 4 > 8 << 20:
            break
    else:
        pytest.fail("no candidate shape splits K with partials beyond the array")
    A = torch.zeros((M, K), dtype=torch.bfloat16, device="cuda")
    B = torch.zeros((N, K), dtype=torch.bfloat16, device="cuda")
    C = torch.zeros((M, N), dtype=torch.bfloat16, device="cuda")
    assert _call(native.gemm_bf16_skinny_noalloc, A, B, C, 1.0, 0.0) == native.GEMM_ERR_INVALID_ARG
    # M above the decode-shaped limit is refused too
    A = torch.zeros((17, 64), dtype=torch.bfloat16, device="cuda")
    B = torch.zeros((64, 64), dtype=torch.bfloat16, device="cuda")
    C = torch.zeros((17, 64), dtype=torch.bfloat16, device="cuda")
    assert _call(native.gemm_bf16_skinny_noalloc, A, B, C, 1.0, 0.0) == native.GEMM_ERR_INVALID_ARG
    del A, B, C
    torch.cuda.empty_cache()
