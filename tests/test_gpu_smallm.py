"""Parity of the small-M kernel (64-row weight tiles; the k-blocks of all tiles
divided evenly over the CTAs, shared tiles summed in piece order by their last
piece) with the CPU oracle.  GB3_GEMM_SMALL_M = 1 routes every M <= 128 call
to it, whatever the planner would choose; GB3_SMALL_M_STREAM_K = 0 gives each
CTA whole tiles instead."""
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


@pytest.fixture
def small_m(monkeypatch):
    monkeypatch.setenv("GB3_GEMM_SMALL_M", "1")


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


def expect_small_m(g, batch, M, N, K, in_dtype=BF16, out=BF16):
    assert g.batched_plan(batch, M, N, K, in_dtype, out)["kernel_name"] == "small_m"


SHAPES = [
    (1, 64, 64),        # one tile, one k-block, one activation row
    (16, 1000, 4096),   # decode-sized, ragged N; 8 CTAs share each tile
    (17, 296, 64),      # NX = 32
    (33, 520, 200),     # NX = 64, ragged N and K; one CTA per tile
    (100, 296, 136),    # NX = 128, ragged everything
    (128, 640, 1024),   # the widest activation tile, full; 2 CTAs per tile
    (40, 1800, 8008),   # ragged K, tiles shared by 11 or 12 CTAs
    (64, 14336, 512),   # 112 tiles: one whole tile per CTA
]


@pytest.fixture(params=["1", "0"], ids=["stream_k", "whole_tiles"])
def division(request, monkeypatch):
    monkeypatch.setenv("GB3_SMALL_M_STREAM_K", request.param)
    return request.param


@pytest.mark.parametrize("M,N,K", SHAPES)
@pytest.mark.parametrize("out", [F32, BF16])
def test_small_m_integer_inputs_exact(g, small_m, division, M, N, K, out):
    """Integer entries make every FP32 partial sum exact: the result equals the
    oracle bit for bit (after RNE for a BF16 output), alpha and beta included,
    however K is divided."""
    A, B, C = workloads.gemm_inputs(M, N, K, 7 * M + K, ("int", -2, 2), ("int", -2, 2),
                                    ("int", -3, 3))
    expect_small_m(g, 1, M, N, K, out=out)
    Cq = C.to(out)
    ref, _ = oracle.gemm_full(A, B, alpha=2.0, beta=-0.5, C=Cq.float())
    Cd = Cq.cuda()
    g.gemm(A.cuda(), B.cuda(), Cd, alpha=2.0, beta=-0.5)
    torch.cuda.synchronize()
    if out == F32:
        assert np.array_equal(to_f64(Cd), ref)
    else:
        assert np.array_equal(bits(Cd), oracle.round_to_bf16_bits(ref))
    assert_status_ok(g)


@pytest.mark.parametrize("M,N,K", [(16, 1000, 4096), (64, 1000, 2000), (128, 520, 512),
                                   (64, 2000, 8192)])
def test_small_m_normal_inputs_within_tolerance(g, small_m, division, M, N, K):
    A, B, _ = workloads.gemm_inputs(M, N, K, 11, ("normal", 1.0), ("normal", 0.03))
    C = torch.full((M, N), float("nan"), dtype=BF16, device="cuda")
    g.gemm(A.cuda(), B.cuda(), C)
    torch.cuda.synchronize()
    ref, ab = oracle.gemm_full(A, B)
    assert_within(to_f64(C), ref, oracle.gemm_tolerance(ref, ab, 1.0, 0.0, out_bf16=True),
                  f"small-M {M}x{N}x{K}")
    assert_status_ok(g)


def test_small_m_fp16(g, small_m):
    M, N, K = 40, 392, 320
    A, B, _ = workloads.gemm_inputs(M, N, K, 12, ("int", -2, 2), ("int", -2, 2), dtype=F16)
    expect_small_m(g, 1, M, N, K, F16, F16)
    C = g.gemm(A.cuda(), B.cuda(), out_dtype=F16)
    torch.cuda.synchronize()
    ref, _ = oracle.gemm_full(A, B)
    assert np.array_equal(bits(C), oracle.round_to_f16_bits(ref))
    assert_status_ok(g)


@pytest.mark.parametrize("K", [136, 2048])   # whole tiles; 4 CTAs per tile
def test_small_m_batched_padded_strides(g, small_m, K):
    """With K = 2048 the CTAs' ranges run from the last tile of one matrix into
    the first tile of the next."""
    bt, M, N = 3, 40, 200
    A, B, _ = workloads.gemm_inputs(M, N, K, 13, ("int", -2, 2), ("int", -2, 2), batch=bt)
    # every matrix padded in its pitch and in its stride
    Ab = torch.zeros(bt, M + 3, K + 8, dtype=BF16, device="cuda")
    Bb = torch.zeros(bt, N + 5, K + 8, dtype=BF16, device="cuda")
    Cb = torch.full((bt, M + 2, N + 8), float("nan"), dtype=F32, device="cuda")
    Ab[:, :M, :K] = A.cuda()
    Bb[:, :N, :K] = B.cuda()
    expect_small_m(g, bt, M, N, K, out=F32)
    g.gemm(Ab[:, :M, :K], Bb[:, :N, :K], Cb[:, :M, :N])
    torch.cuda.synchronize()
    for b in range(bt):
        ref, _ = oracle.gemm_full(A[b], B[b])
        assert np.array_equal(to_f64(Cb[b, :M, :N]), ref)
    # the padding is untouched
    assert torch.isnan(Cb[:, M:, :]).all() and torch.isnan(Cb[:, :, N:]).all()
    assert_status_ok(g)


def test_small_m_matches_split_k_within_tolerance_and_is_deterministic(g, monkeypatch):
    M, N, K = 16, 3000, 4096
    A, B, _ = workloads.gemm_inputs(M, N, K, 14, ("normal", 1.0), ("normal", 0.02))
    Ad, Bd = A.cuda(), B.cuda()
    monkeypatch.setenv("GB3_GEMM_SMALL_M", "1")
    C1 = g.gemm(Ad, Bd, out_dtype=F32)
    C2 = g.gemm(Ad, Bd, out_dtype=F32)
    monkeypatch.setenv("GB3_GEMM_SMALL_M", "0")
    C3 = g.gemm(Ad, Bd, out_dtype=F32)
    torch.cuda.synchronize()
    assert torch.equal(C1, C2)
    ref, ab = oracle.gemm_full(A, B)
    tol = oracle.gemm_tolerance(ref, ab, 1.0, 0.0)
    assert_within(to_f64(C1), ref, tol, "small-M")
    assert_within(to_f64(C3), ref, tol, "split-K")
    assert_status_ok(g)


def test_small_m_whole_tiles_capture_without_workspace(g, small_m, monkeypatch):
    """One CTA per whole tile allocates nothing, so the call can be captured
    without an eager call first."""
    monkeypatch.setenv("GB3_SMALL_M_STREAM_K", "0")
    M, N, K = 16, 2048, 1024
    assert g.batched_plan(1, M, N, K, BF16, F32)["split_k"] == 1
    A, B, _ = workloads.gemm_inputs(M, N, K, 15, ("int", -2, 2), ("int", -2, 2))
    Ad, Bd = A.cuda(), B.cuda()
    C = torch.full((M, N), float("nan"), dtype=F32, device="cuda")
    stream = torch.cuda.Stream()
    graph = torch.cuda.CUDAGraph()
    with torch.cuda.graph(graph, stream=stream):
        g.gemm(Ad, Bd, C)
    graph.replay()
    torch.cuda.synchronize()
    ref, _ = oracle.gemm_full(A, B)
    assert np.array_equal(to_f64(C), ref)
    assert_status_ok(g)


def test_small_m_stream_k_capture_and_replay(g, small_m):
    """Shared tiles need the workspace: an eager call sets it up, after which
    replays of a captured call reuse it and leave its counters at zero."""
    M, N, K = 16, 2048, 1024
    assert g.batched_plan(1, M, N, K, BF16, F32)["split_k"] > 1
    A, B, _ = workloads.gemm_inputs(M, N, K, 16, ("int", -2, 2), ("int", -2, 2))
    Ad, Bd = A.cuda(), B.cuda()
    C = torch.full((M, N), float("nan"), dtype=F32, device="cuda")
    g.gemm(Ad, Bd, C)
    torch.cuda.synchronize()
    stream = torch.cuda.Stream()
    graph = torch.cuda.CUDAGraph()
    with torch.cuda.stream(stream):
        with torch.cuda.graph(graph, stream=stream):
            g.gemm(Ad, Bd, C, stream=stream)
    ref, _ = oracle.gemm_full(A, B)
    for _ in range(3):
        C.fill_(float("nan"))
        graph.replay()
        torch.cuda.synchronize()
        assert np.array_equal(to_f64(C), ref)
    assert_status_ok(g)


@pytest.mark.parametrize("out,N,pad", [(BF16, 600, 8), (BF16, 602, 6), (F32, 600, 4),
                                       (F32, 601, 3), (F16, 597, 11)])
def test_small_m_shared_tiles_padded_ragged(g, small_m, out, N, pad):
    """The combine of shared tiles writes four outputs at once, and one at a
    time in the last group of a row whose N is not a multiple of 4; both give
    the oracle's bits, with alpha and beta, and leave the padding alone."""
    M, K = 40, 4096
    in_dtype = F16 if out == F16 else BF16
    assert g.batched_plan(1, M, N, K, in_dtype, out)["split_k"] > 1
    A, B, C = workloads.gemm_inputs(M, N, K, 19 + pad, ("int", -2, 2), ("int", -2, 2),
                                    ("int", -3, 3), dtype=in_dtype)
    Cq = C.to(out)
    buf = torch.full((M, N + pad), float("nan"), dtype=out, device="cuda")
    buf[:, :N] = Cq.cuda()
    Cv = buf[:, :N]
    g.gemm(A.cuda(), B.cuda(), Cv, alpha=2.0, beta=-0.5)
    torch.cuda.synchronize()
    ref, _ = oracle.gemm_full(A, B, alpha=2.0, beta=-0.5, C=Cq.float())
    if out == F32:
        assert np.array_equal(to_f64(Cv), ref)
    elif out == BF16:
        assert np.array_equal(bits(Cv), oracle.round_to_bf16_bits(ref))
    else:
        assert np.array_equal(bits(Cv), oracle.round_to_f16_bits(ref))
    assert torch.isnan(buf[:, N:].float()).all()
    assert_status_ok(g)


_PREPARE_THEN_CAPTURE = r"""
import numpy as np, torch
import dense_bf16_gemm_gb300 as g, oracle, workloads
M, N, K = 100, 3000, 4096
assert g.batched_plan(1, M, N, K, torch.bfloat16, torch.float32)["split_k"] > 1
A, B, _ = workloads.gemm_inputs(M, N, K, 18, ("int", -2, 2), ("int", -2, 2))
Ad, Bd = A.cuda(), B.cuda()
C = torch.full((M, N), float("nan"), dtype=torch.float32, device="cuda")
g.prepare(N)
torch.cuda.synchronize()
stream = torch.cuda.Stream()
graph = torch.cuda.CUDAGraph()
with torch.cuda.stream(stream):
    with torch.cuda.graph(graph, stream=stream):
        g.gemm(Ad, Bd, C, stream=stream)
graph.replay()
torch.cuda.synchronize()
ref, _ = oracle.gemm_full(A, B)
assert np.array_equal(C.double().cpu().numpy(), ref)
assert g.device_status()[0] == 0
print("prepared capture ok")
"""


def test_small_m_prepare_then_capture_in_fresh_process(g):
    """gemm_prepare(N) sizes the workspace for every M <= 128: a fresh process
    captures a small-M call with shared tiles without any eager call first."""
    import os
    import subprocess
    import sys
    root = os.path.dirname(os.path.dirname(os.path.abspath(__file__)))
    env = dict(os.environ, GB3_GEMM_SMALL_M="1")
    r = subprocess.run([sys.executable, "-c", _PREPARE_THEN_CAPTURE], cwd=root, env=env,
                       capture_output=True, text=True, timeout=600)
    assert r.returncode == 0, r.stdout[-2000:] + r.stderr[-2000:]
    assert "prepared capture ok" in r.stdout


def test_small_m_stream_k_deterministic(g, small_m):
    """The shared tiles are summed in piece order, so repeated calls agree bit
    for bit on inputs whose partial sums round."""
    M, N, K = 64, 2000, 8192
    A, B, _ = workloads.gemm_inputs(M, N, K, 17, ("normal", 1.0), ("normal", 0.02))
    Ad, Bd = A.cuda(), B.cuda()
    assert g.batched_plan(1, M, N, K, BF16, F32)["split_k"] > 1
    outs = [g.gemm(Ad, Bd, out_dtype=F32) for _ in range(4)]
    torch.cuda.synchronize()
    for o in outs[1:]:
        assert torch.equal(o, outs[0])
    assert_status_ok(g)


@pytest.mark.slow
@pytest.mark.parametrize("name", ["skinny_16x28672x8192", "smallm_64x28672x8192",
                                  "smallm_64x8192x8192"])
def test_workload_small_m(g, small_m, name):
    """Full size: every entry within 256 columns of either edge, every row,
    plus 65,536 sampled entries."""
    w = workloads.WORKLOADS[name]
    A, B, _ = workloads.inputs_for(w)
    expect_small_m(g, 1, w.M, w.N, w.K)
    C = torch.full((w.M, w.N), float("nan"), dtype=BF16, device="cuda")
    # (the planner itself picks the small-M kernel for the last of these)
    g.gemm(A.cuda(), B.cuda(), C)
    torch.cuda.synchronize()
    rows, cols = workloads.sample_entries(w.M, w.N, w.seed)
    ref, ab = oracle.gemm_entries(A, B, rows, cols)
    tol = oracle.gemm_tolerance(ref, ab, 1.0, 0.0, out_bf16=True)
    assert_within(to_f64(C)[rows, cols], ref, tol, name)
    assert_status_ok(g)
