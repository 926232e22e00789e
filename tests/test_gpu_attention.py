"""Parity of the attention kernel with the CPU oracle: softmax(scale Q.K^T).V
per head, through the C ABI (via the thin torch binding)."""
import numpy as np
import pytest
import torch

import oracle
import workloads

pytestmark = pytest.mark.gpu

F32, BF16 = torch.float32, torch.bfloat16


@pytest.fixture(scope="module")
def g():
    from dense_bf16_gemm_gb300 import build
    build.build()
    import dense_bf16_gemm_gb300 as lib
    lib._native.lib()
    return lib


def to_f64(t):
    return t.detach().to("cpu").to(torch.float64).numpy()


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


def check(g, H, Nq, Nk, D, seed, scale=None, out=BF16, rows=None):
    Q, K, V = workloads.attention_inputs(H, Nq, Nk, D, seed)
    scale = D ** -0.5 if scale is None else scale
    O = torch.full((H, Nq, D), float("nan"), dtype=out, device="cuda")
    g.attention(Q.cuda(), K.cuda(), V.cuda(), scale, O=O)
    torch.cuda.synchronize()
    if rows is None:
        hh, rr = np.meshgrid(np.arange(H), np.arange(Nq), indexing="ij")
        hh, rr = hh.ravel(), rr.ravel()
    else:
        hh, rr = rows
    res = oracle.attention_rows(Q, K, V, scale, hh, rr)
    tol = oracle.attention_tolerance(res, D, Nk, out_bf16=out == BF16)
    assert_within(to_f64(O)[hh, rr], res["o"], tol, f"attention {H}x{Nq}x{Nk}x{D}")
    assert_status_ok(g)
    return Q, K, V, O


@pytest.mark.parametrize("H,Nq,Nk,D", [
    (1, 128, 128, 64),     # one query block, one key block
    (1, 128, 128, 128),
    (2, 200, 300, 128),    # ragged queries and keys
    (3, 1, 1, 64),         # one query, one key
    (1, 129, 1000, 128),   # a second query block of one row; eight key blocks, ragged
    (2, 256, 2048, 64),    # many key blocks: the ring and both score buffers wrap
])
@pytest.mark.parametrize("out", [BF16, F32])
def test_attention_within_tolerance(g, H, Nq, Nk, D, out):
    check(g, H, Nq, Nk, D, seed=H + Nq + Nk + D, out=out)


@pytest.mark.parametrize("scale", [0.0, 1.0, -0.3])
def test_attention_scales(g, scale):
    check(g, 2, 160, 520, 64, seed=5, scale=scale, out=F32)


def test_attention_zero_scale_is_the_mean_of_V(g):
    """Scale 0: every probability is exactly 1 (and exact in BF16), so the
    output is the FP32 mean of V."""
    H, Nq, Nk, D = 2, 130, 700, 128
    Q, K, V = workloads.attention_inputs(H, Nq, Nk, D, 6)
    O = g.attention(Q.cuda(), K.cuda(), V.cuda(), 0.0, out_dtype=F32)
    torch.cuda.synchronize()
    mean = V.double().mean(dim=1, keepdim=True).expand(H, Nq, D).numpy()
    assert np.allclose(to_f64(O), mean, rtol=0, atol=1e-5)
    assert_status_ok(g)


def test_attention_dominant_key(g):
    """A key far above the others in every query's score selects its value."""
    H, Nq, Nk, D = 1, 128, 384, 64
    Q = torch.zeros(H, Nq, D)
    Q[..., 0] = 8.0
    K = torch.zeros(H, Nk, D)
    K[0, 300, 0] = 8.0          # score 64 against 0 for every other key
    V = torch.randn(H, Nk, D, generator=torch.Generator().manual_seed(7))
    Q, K, V = (x.to(BF16) for x in (Q, K, V))
    O = g.attention(Q.cuda(), K.cuda(), V.cuda(), 1.0, out_dtype=F32)
    torch.cuda.synchronize()
    want = V.double()[0, 300].expand(Nq, D).numpy()
    assert np.allclose(to_f64(O)[0], want, rtol=0, atol=1e-6)
    assert_status_ok(g)


@pytest.mark.parametrize("direction", ["growing", "shrinking"])
def test_attention_running_maximum_moves(g, direction):
    """Scores that climb by about 17 (base 2) from one key block to the next
    move every row's running maximum past the rescaling threshold on every
    block (the output accumulator is rescaled each time); falling scores never
    move it after the first block."""
    H, Nq, Nk, D = 2, 200, 1000, 64
    gen = torch.Generator().manual_seed(11)
    Q = torch.randn(H, Nq, D, generator=gen) * 0.1
    Q[..., 0] = 1.0
    K = torch.randn(H, Nk, D, generator=gen) * 0.1
    ramp = torch.arange(Nk, dtype=torch.float32) / 128.0 * 12.0
    K[..., 0] = ramp if direction == "growing" else ramp.flip(0)
    V = torch.randn(H, Nk, D, generator=gen)
    Q, K, V = (x.to(BF16) for x in (Q, K, V))
    O = g.attention(Q.cuda(), K.cuda(), V.cuda(), 1.0, out_dtype=F32)
    torch.cuda.synchronize()
    hh, rr = np.meshgrid(np.arange(H), np.arange(Nq), indexing="ij")
    res = oracle.attention_rows(Q, K, V, 1.0, hh.ravel(), rr.ravel())
    tol = oracle.attention_tolerance(res, D, Nk, out_bf16=False)
    assert_within(to_f64(O)[hh.ravel(), rr.ravel()], res["o"], tol, direction)
    assert_status_ok(g)


def test_attention_padded_strides_and_2d(g):
    H, Nq, Nk, D = 3, 150, 260, 64
    Q, K, V = workloads.attention_inputs(H, Nq, Nk, D, 8)
    # padded pitches and head strides
    Qp = torch.zeros(H, Nq + 5, D + 8, dtype=BF16, device="cuda")
    Kp = torch.zeros(H, Nk + 3, D + 16, dtype=BF16, device="cuda")
    Vp = torch.zeros(H, Nk + 7, D + 8, dtype=BF16, device="cuda")
    Op = torch.full((H, Nq + 2, D + 8), float("nan"), dtype=F32, device="cuda")
    Qp[:, :Nq, :D], Kp[:, :Nk, :D], Vp[:, :Nk, :D] = Q.cuda(), K.cuda(), V.cuda()
    g.attention(Qp[:, :Nq, :D], Kp[:, :Nk, :D], Vp[:, :Nk, :D], 0.125, O=Op[:, :Nq, :D])
    torch.cuda.synchronize()
    hh, rr = np.meshgrid(np.arange(H), np.arange(Nq), indexing="ij")
    res = oracle.attention_rows(Q, K, V, 0.125, hh.ravel(), rr.ravel())
    tol = oracle.attention_tolerance(res, D, Nk, out_bf16=False)
    assert_within(to_f64(Op[:, :Nq, :D])[hh.ravel(), rr.ravel()], res["o"], tol, "padded")
    assert torch.isnan(Op[:, Nq:, :]).all() and torch.isnan(Op[:, :, D:]).all()
    # one head through the 2-D form equals the batched result for that head
    O1 = g.attention(Q[1].cuda(), K[1].cuda(), V[1].cuda(), 0.125, out_dtype=F32)
    torch.cuda.synchronize()
    assert torch.equal(O1, Op[1, :Nq, :D])
    assert_status_ok(g)


def test_attention_deterministic(g):
    Q, K, V = workloads.attention_inputs(4, 512, 1024, 128, 9)
    Qd, Kd, Vd = Q.cuda(), K.cuda(), V.cuda()
    O1 = g.attention(Qd, Kd, Vd)
    O2 = g.attention(Qd, Kd, Vd)
    torch.cuda.synchronize()
    assert torch.equal(O1.view(torch.int16), O2.view(torch.int16))
    assert_status_ok(g)


@pytest.mark.slow
@pytest.mark.parametrize("name", ["attention_32x4096x4096x128", "attention_32x4096x4096x64"])
def test_workload_attention(g, name):
    """Full size: the first and last 128 query rows and 256 drawn ones, in
    the first, a middle and the last head."""
    w = workloads.WORKLOADS[name]
    Q, K, V = workloads.inputs_for(w)
    O = g.attention(Q.cuda(), K.cuda(), V.cuda(), w.K ** -0.5)
    torch.cuda.synchronize()
    gen = np.random.default_rng(w.seed)
    rows = np.unique(np.concatenate([np.arange(128), np.arange(w.M - 128, w.M),
                                     gen.choice(w.M, 256, replace=False)]))
    heads = np.array([0, w.batch // 2, w.batch - 1])
    hh, rr = np.repeat(heads, rows.size), np.tile(rows, heads.size)
    res = oracle.attention_rows(Q, K, V, w.K ** -0.5, hh, rr)
    tol = oracle.attention_tolerance(res, w.K, w.N, out_bf16=True)
    assert_within(to_f64(O)[hh, rr], res["o"], tol, name)
    assert_status_ok(g)


@pytest.mark.parametrize("Nk,key", [(384, 200), (384, 290), (129, 128), (256, 255), (640, 520)])
def test_attention_dominant_key_in_either_chain(g, Nk, key):
    """The key blocks are dealt to two loops (even and odd blocks) merged at
    the end: a dominant key in an odd block (chain 1), in the only key of the
    second block, or in a later even block, selects its value exactly as one
    in block 0 does."""
    H, Nq, D = 1, 200, 64
    Q = torch.zeros(H, Nq, D)
    Q[..., 0] = 8.0
    K = torch.zeros(H, Nk, D)
    K[0, key, 0] = 8.0          # score 64 against 0 for every other key
    V = torch.randn(H, Nk, D, generator=torch.Generator().manual_seed(Nk + key))
    Q, K, V = (x.to(BF16) for x in (Q, K, V))
    O = g.attention(Q.cuda(), K.cuda(), V.cuda(), 1.0, out_dtype=F32)
    torch.cuda.synchronize()
    want = V.double()[0, key].expand(Nq, D).numpy()
    assert np.allclose(to_f64(O)[0], want, rtol=0, atol=1e-6)
    assert_status_ok(g)


@pytest.mark.parametrize("D", [64, 128])
@pytest.mark.parametrize("Nk", [129, 256, 257, 1152])
def test_attention_chains_with_different_maxima(g, Nk, D):
    """Scores whose scale differs between even and odd key blocks (odd blocks
    ~20 higher in base 2, then lower), so the two loops' maxima and sums
    differ and the merge's scaling decides the result; checked against the
    oracle within the derived bound."""
    H, Nq = 2, 160
    gen = torch.Generator().manual_seed(Nk + D)
    Q = torch.randn(H, Nq, D, generator=gen) * 0.3
    Q[..., 0] = 1.0
    K = torch.randn(H, Nk, D, generator=gen) * 0.3
    blk = (torch.arange(Nk) // 128) % 2
    K[..., 0] = torch.where(blk == 1, torch.tensor(14.0), torch.tensor(0.0)) \
        - (torch.arange(Nk) >= 768).float() * 28.0
    V = torch.randn(H, Nk, D, generator=gen)
    Q, K, V = (x.to(BF16) for x in (Q, K, V))
    O = g.attention(Q.cuda(), K.cuda(), V.cuda(), 1.0, out_dtype=F32)
    torch.cuda.synchronize()
    hh, rr = np.meshgrid(np.arange(H), np.arange(Nq), indexing="ij")
    res = oracle.attention_rows(Q, K, V, 1.0, hh.ravel(), rr.ravel())
    tol = oracle.attention_tolerance(res, D, Nk, out_bf16=False)
    assert_within(to_f64(O)[hh.ravel(), rr.ravel()], res["o"], tol, f"Nk={Nk}")
    assert_status_ok(g)
