"""The allocation-free decode-shaped GEMM (gemm_bf16_skinny_noalloc).

It serves callers that may not allocate device memory during a call (for
example code whose memory pool must own every byte, or that cannot afford the
synchronization an allocation can cause): its split-K partial sums live in a
fixed array compiled into the library.  These tests call it through the C ABI
and compare it with gemm_bf16 on the same inputs, two calls in a row, so that
state left in the shared array by one call cannot leak into the next.

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


@pytest.mark.parametrize("out_dtype", [torch.bfloat16, torch.float32])
def test_noalloc_matches_gemm_bf16_on_two_calls_in_a_row(native, out_dtype):
    cases = [
        # (M, N, K, alpha, beta, seed)
        (16, 28672, 8192, 1.0, 0.0, 41),   # the decode workload's shape, split-K
        (5, 3000, 4096, 0.5, 2.0, 42),     # ragged M and N, beta reads C
    ]
    for M, N, K, alpha, beta, seed in cases:
        A, B, C = workloads.gemm_inputs(M, N, K, seed, ("normal", 1.0),
                                        ("normal", K ** -0.5), ("normal", 1.0))
        Ad, Bd = A.cuda(), B.cuda()
        C0 = C.to(out_dtype).cuda()
        c_ref = C0.clone()
        c_new = C0.clone()
        assert _call(native.gemm_bf16, Ad, Bd, c_ref, alpha, beta) == 0
        assert _call(native.gemm_bf16_skinny_noalloc, Ad, Bd, c_new, alpha, beta) == 0
        torch.cuda.synchronize()
        st, site = native.gemm_get_device_status(torch.cuda.current_stream().cuda_stream)
        assert st == 0, (st, site)
        # tolerance of the parity tests, scaled from the oracle's sum |a b|
        rows = np.arange(M).repeat(256)
        cols = np.tile(np.linspace(0, N - 1, 256).astype(np.int64), M)
        _, ab = oracle.gemm_entries(A, B, rows, cols, alpha=alpha, beta=beta,
                                    C=C0.float().cpu())
        got = c_new.double().cpu().numpy()
        ref = c_ref.double().cpu().numpy()
        c_in = C0.double().cpu().numpy()[rows, cols]
        tol = oracle.gemm_tolerance(ref[rows, cols], ab, alpha, beta, c_in,
                                    out_bf16=out_dtype == torch.bfloat16)
        assert np.all(np.abs(got[rows, cols] - ref[rows, cols]) <= tol)
        # every entry, against the allocating entry point's own result
        full_tol = 4e-3 * (np.abs(ref) + 1.0)
        assert np.all(np.abs(got - ref) <= full_tol)


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
