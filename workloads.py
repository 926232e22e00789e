"""Seeded synthetic inputs for the GEMM and gate/up workloads.

This module holds the random-number recipe only and none of the arithmetic of
the method: it draws float32 values with a seeded ``torch.Generator`` on the
CPU, rounds them to BF16 (round-to-nearest-even, ``Tensor.to``) and returns the
CPU tensors.  The CUDA path receives device copies of exactly these bytes and
the oracle reads the same host bytes, so both sides see identical inputs.

Storage (both operands K-contiguous):
  A  (M, K)  a(m,k) = A[m, k]
  B  (N, K)  b(k,n) = B[n, k]
  C  (M, N)  float32, only for beta != 0
Gate/up:  X (M, K), Wg (N, K), Wu (N, K).
Row normalisation:  X (rows, D) with a per-row magnitude exp(N(0,1)) so that
rows of very different scale meet; gains G (D,) uniform on [0.5, 1.5).

Draw order within one generator: A, then B, then C (or X, Wg, Wu).
"uniform" is ``2 * rand - 1`` (uniform on [-1, 1)); "normal" is
``std * randn``.
"""
from __future__ import annotations

import math
from dataclasses import dataclass, field

import numpy as np
import torch


@dataclass(frozen=True)
class Workload:
    name: str
    kind: str                 # "gemm", "gate_up", "gemm_row_stats", "rms_norm",
                              # "rmsnorm_gate_up" or "attention" (M = Nq, N = Nk,
                              # K = head dimension D, batch = heads)
    M: int
    N: int
    K: int
    seed: int
    dist_a: tuple             # ("uniform",) or ("normal", std)
    dist_b: tuple
    alpha: float = 1.0
    beta: float = 0.0
    dist_c: tuple | None = None
    out_bf16: bool = False
    check: str = "full"       # "full" or "sampled"
    notes: str = ""
    batch: int = 1            # independent matrices (gemm only)
    in_f16: bool = False      # FP16 operands instead of BF16
    out_f16: bool = False     # FP16 output
    norm_in: str = "bf16"     # rms_norm input element type: "f32", "bf16" or "f16"
    eps: float = 1e-6         # rms_norm constant

    @property
    def out_dtype(self):
        if self.out_f16:
            return torch.float16
        return torch.bfloat16 if self.out_bf16 else torch.float32

    @property
    def flops(self) -> float:
        """Useful floating-point operations: 2MNK per GEMM (two for gate/up)."""
        if self.kind == "rms_norm":
            return 3.0 * self.M * self.K
        if self.kind == "attention":   # Q.K^T and P.V
            return 4.0 * self.batch * self.M * self.N * self.K
        per = 2.0 * self.M * self.N * self.K * self.batch
        return 2.0 * per if self.kind in ("gate_up", "rmsnorm_gate_up") else per

    @property
    def algorithmic_bytes(self) -> int:
        """Compulsory HBM bytes: each input read once, the output written once
        (plus C read when beta != 0)."""
        out_elem = 2 if (self.out_bf16 or self.out_f16) else 4
        if self.kind == "rms_norm":
            in_elem = 4 if self.norm_in == "f32" else 2
            return self.M * self.K * (in_elem + out_elem) + 4 * self.K
        if self.kind == "gate_up":
            return 2 * (self.M * self.K + 2 * self.N * self.K + self.M * self.N)
        if self.kind == "attention":   # Q and O once, K and V once per head
            return self.batch * (2 * self.M * self.K + 4 * self.N * self.K +
                                 out_elem * self.M * self.K)
        if self.kind == "rmsnorm_gate_up":
            # X read, Xn written, both weights read, Y written (Xn is re-read from L2)
            return 2 * (2 * self.M * self.K + 2 * self.N * self.K + self.M * self.N) + 4 * self.K
        b = 2 * (self.M * self.K + self.N * self.K) + out_elem * self.M * self.N
        if self.beta != 0.0:
            b += out_elem * self.M * self.N
        if self.kind == "gemm_row_stats":
            b += 3 * 4 * self.M
        return b * self.batch


WORKLOADS = {
    "gemm_256_f32": Workload(
        "gemm_256_f32", "gemm", 256, 256, 256, seed=0,
        dist_a=("uniform",), dist_b=("uniform",), out_bf16=False,
        notes="M=N=K=256, FP32 output, alpha=1, beta=0"),
    "gemm_4096_bf16": Workload(
        "gemm_4096_bf16", "gemm", 4096, 4096, 4096, seed=1,
        dist_a=("normal", 1.0), dist_b=("normal", 1.0), out_bf16=True,
        notes="M=N=K=4096, BF16 output, alpha=1, beta=0"),
    "gemm_ragged_3000x5000x2000": Workload(
        "gemm_ragged_3000x5000x2000", "gemm", 3000, 5000, 2000, seed=2,
        dist_a=("uniform",), dist_b=("uniform",), alpha=0.5, beta=2.0,
        dist_c=("normal", 1.0), out_bf16=False,
        notes="ragged tails in M, N and K; FP32 C read and written"),
    "gate_up_4096x14336x4096": Workload(
        "gate_up_4096x14336x4096", "gate_up", 4096, 14336, 4096, seed=3,
        dist_a=("normal", 1.0), dist_b=("normal", 1.0 / 64.0), out_bf16=True,
        check="sampled",
        notes="Y = silu(X Wg) * (X Wu), BF16 [4096, 14336]"),
    # The gate/up projection at a decode batch of 16: HBM-bound on Wg and Wu.
    "skinny_gate_up_16x14336x4096": Workload(
        "skinny_gate_up_16x14336x4096", "gate_up", 16, 14336, 4096, seed=14,
        dist_a=("normal", 1.0), dist_b=("normal", 1.0 / 64.0), out_bf16=True,
        check="sampled",
        notes="Y = silu(X Wg) * (X Wu) for 16 rows, Wg and Wu 117 MB each"),
    "skinny_16x28672x8192": Workload(
        "skinny_16x28672x8192", "gemm", 16, 28672, 8192, seed=4,
        dist_a=("normal", 1.0), dist_b=("normal", 1.0 / math.sqrt(8192)),
        out_bf16=True, check="sampled",
        notes="decode-shaped, weight 470 MB, HBM-bound"),
    # Batched and FP16 variants (the next row after the five workloads above).
    "gemm_4096_f16": Workload(
        "gemm_4096_f16", "gemm", 4096, 4096, 4096, seed=5,
        dist_a=("normal", 1.0), dist_b=("normal", 1.0), out_f16=True, in_f16=True,
        notes="M=N=K=4096, FP16 operands and output"),
    "gemm_batched_8x2048": Workload(
        "gemm_batched_8x2048", "gemm", 2048, 2048, 2048, seed=6,
        dist_a=("normal", 1.0), dist_b=("normal", 1.0), out_bf16=True, batch=8,
        notes="8 independent 2048^3 BF16 GEMMs, one call"),
    # A decode batch of 64 rows: the small-M kernel's home ground.
    "smallm_64x28672x8192": Workload(
        "smallm_64x28672x8192", "gemm", 64, 28672, 8192, seed=10,
        dist_a=("normal", 1.0), dist_b=("normal", 1.0 / math.sqrt(8192)),
        out_bf16=True, check="sampled",
        notes="decode batch of 64, weight 470 MB, HBM-bound"),
    "smallm_64x8192x8192": Workload(
        "smallm_64x8192x8192", "gemm", 64, 8192, 8192, seed=11,
        dist_a=("normal", 1.0), dist_b=("normal", 1.0 / math.sqrt(8192)),
        out_bf16=True, check="sampled",
        notes="decode batch of 64 through an 8192 x 8192 projection (134 MB): 64 weight "
              "tiles of 128 rows, their k-blocks divided over every SM"),
    # Softmax attention (the flash-attention loop).
    "attention_32x4096x4096x128": Workload(
        "attention_32x4096x4096x128", "attention", 4096, 4096, 128, seed=12,
        dist_a=("normal", 1.0), dist_b=("normal", 1.0), out_bf16=True, batch=32,
        check="sampled", notes="32 heads, 4096 queries and keys, D = 128, scale 1/sqrt(D)"),
    "attention_32x4096x4096x64": Workload(
        "attention_32x4096x4096x64", "attention", 4096, 4096, 64, seed=13,
        dist_a=("normal", 1.0), dist_b=("normal", 1.0), out_bf16=True, batch=32,
        check="sampled", notes="32 heads, 4096 queries and keys, D = 64, scale 1/sqrt(D)"),
    # Row reductions and the row normalisation (the row after those).
    "gemm_row_stats_4096": Workload(
        "gemm_row_stats_4096", "gemm_row_stats", 4096, 4096, 4096, seed=1,
        dist_a=("normal", 1.0), dist_b=("normal", 1.0), out_bf16=True, check="sampled",
        notes="the 4096^3 BF16 GEMM plus the sum, max and min of every row"),
    "rms_norm_262144x256_f32": Workload(
        "rms_norm_262144x256_f32", "rms_norm", 262144, 256, 256, seed=7,
        dist_a=("normal", 1.0), dist_b=("uniform",), norm_in="f32", check="sampled",
        notes="row normalisation, D=256, FP32 in and out"),
    "rms_norm_16384x4096_bf16": Workload(
        "rms_norm_16384x4096_bf16", "rms_norm", 16384, 4096, 4096, seed=8,
        dist_a=("normal", 1.0), dist_b=("uniform",), norm_in="bf16", out_bf16=True,
        check="sampled", notes="row normalisation, D=4096, BF16 in and out"),
    "rmsnorm_gate_up_4096x14336x4096": Workload(
        "rmsnorm_gate_up_4096x14336x4096", "rmsnorm_gate_up", 4096, 14336, 4096, seed=9,
        dist_a=("normal", 1.0), dist_b=("normal", 1.0 / 64.0), out_bf16=True,
        check="sampled", notes="Y = silu(Xn Wg) * (Xn Wu), Xn = rms_norm(X)"),
}

# The workload the benchmark times by default.
HEADLINE = "gemm_4096_bf16"


def _draw(gen: torch.Generator, shape, dist) -> torch.Tensor:
    if dist[0] == "uniform":
        return torch.rand(shape, generator=gen, dtype=torch.float32) * 2.0 - 1.0
    if dist[0] == "normal":
        return torch.randn(shape, generator=gen, dtype=torch.float32) * float(dist[1])
    if dist[0] == "int":
        lo, hi = dist[1], dist[2]
        return torch.randint(lo, hi + 1, shape, generator=gen).to(torch.float32)
    raise ValueError(f"unknown distribution {dist!r}")


def gemm_inputs(M: int, N: int, K: int, seed: int, dist_a=("uniform",),
                dist_b=("uniform",), dist_c=None, batch: int = 1, dtype=torch.bfloat16):
    """CPU tensors ``A`` (M,K), ``B`` (N,K) of ``dtype`` (bf16 or f16) and ``C``
    (M,N) f32 or None; with batch > 1 each gains a leading batch dimension."""
    gen = torch.Generator(device="cpu").manual_seed(int(seed))
    lead = (batch,) if batch > 1 else ()
    A = _draw(gen, lead + (M, K), dist_a).to(dtype)
    B = _draw(gen, lead + (N, K), dist_b).to(dtype)
    C = _draw(gen, lead + (M, N), dist_c) if dist_c is not None else None
    return A, B, C


def gate_up_inputs(M: int, N: int, K: int, seed: int, dist_x=("normal", 1.0),
                   dist_w=("normal", 1.0)):
    """CPU tensors ``X`` (M,K), ``Wg`` (N,K), ``Wu`` (N,K), all bf16."""
    gen = torch.Generator(device="cpu").manual_seed(int(seed))
    X = _draw(gen, (M, K), dist_x).to(torch.bfloat16)
    Wg = _draw(gen, (N, K), dist_w).to(torch.bfloat16)
    Wu = _draw(gen, (N, K), dist_w).to(torch.bfloat16)
    return X, Wg, Wu


_NORM_TYPES = {"f32": torch.float32, "bf16": torch.bfloat16, "f16": torch.float16}


def rms_norm_inputs(rows: int, D: int, seed: int, dtype=torch.float32):
    """CPU tensors ``X`` (rows, D) of ``dtype`` and gains ``G`` (D,) float32.

    Draw order: the row magnitudes (rows, 1), then X, then G."""
    gen = torch.Generator(device="cpu").manual_seed(int(seed))
    mag = torch.exp(_draw(gen, (rows, 1), ("normal", 1.0)))
    X = (_draw(gen, (rows, D), ("normal", 1.0)) * mag).to(dtype)
    G = torch.rand(D, generator=gen, dtype=torch.float32) + 0.5
    return X, G


def rmsnorm_gate_up_inputs(M: int, N: int, K: int, seed: int, dist_w=("normal", 1.0)):
    """CPU tensors ``X`` (M,K) bf16 with per-row magnitudes, ``G`` (K,) float32,
    ``Wg``, ``Wu`` (N,K) bf16, drawn in that order from one generator."""
    gen = torch.Generator(device="cpu").manual_seed(int(seed))
    mag = torch.exp(_draw(gen, (M, 1), ("normal", 1.0)))
    X = (_draw(gen, (M, K), ("normal", 1.0)) * mag).to(torch.bfloat16)
    G = torch.rand(K, generator=gen, dtype=torch.float32) + 0.5
    Wg = _draw(gen, (N, K), dist_w).to(torch.bfloat16)
    Wu = _draw(gen, (N, K), dist_w).to(torch.bfloat16)
    return X, G, Wg, Wu


def attention_inputs(heads: int, Nq: int, Nk: int, D: int, seed: int, dist=("normal", 1.0)):
    """CPU bf16 tensors Q (heads, Nq, D), K and V (heads, Nk, D), drawn in that order."""
    gen = torch.Generator(device="cpu").manual_seed(int(seed))
    Q = _draw(gen, (heads, Nq, D), dist).to(torch.bfloat16)
    K = _draw(gen, (heads, Nk, D), dist).to(torch.bfloat16)
    V = _draw(gen, (heads, Nk, D), dist).to(torch.bfloat16)
    return Q, K, V


def inputs_for(w: Workload):
    if w.kind == "attention":
        return attention_inputs(w.batch, w.M, w.N, w.K, w.seed, w.dist_a)
    if w.kind == "gate_up":
        return gate_up_inputs(w.M, w.N, w.K, w.seed, w.dist_a, w.dist_b)
    if w.kind == "rms_norm":
        return rms_norm_inputs(w.M, w.K, w.seed, _NORM_TYPES[w.norm_in])
    if w.kind == "rmsnorm_gate_up":
        return rmsnorm_gate_up_inputs(w.M, w.N, w.K, w.seed, w.dist_b)
    return gemm_inputs(w.M, w.N, w.K, w.seed, w.dist_a, w.dist_b, w.dist_c, w.batch,
                       torch.float16 if w.in_f16 else torch.bfloat16)


def sample_entries(M: int, N: int, seed: int, count: int = 65536, edge: int = 256):
    """Output coordinates to check for a large result.

    Every entry within ``edge`` rows of the top or bottom edge or within
    ``edge`` columns of the left or right edge, plus ``count`` further
    distinct entries drawn uniformly (without replacement, by a generator
    seeded with ``seed + 1000``).  Returns ``(rows, cols)`` int64 arrays.
    """
    mask = np.zeros((M, N), dtype=bool) if M * N <= (1 << 28) else None
    rows_e, cols_e = [], []
    r_edge = np.unique(np.concatenate([np.arange(min(edge, M)),
                                       np.arange(max(M - edge, 0), M)]))
    c_edge = np.unique(np.concatenate([np.arange(min(edge, N)),
                                       np.arange(max(N - edge, 0), N)]))
    rr, cc = np.meshgrid(r_edge, np.arange(N), indexing="ij")
    rows_e.append(rr.ravel()); cols_e.append(cc.ravel())
    mid = np.setdiff1d(np.arange(M), r_edge)
    rr, cc = np.meshgrid(mid, c_edge, indexing="ij")
    rows_e.append(rr.ravel()); cols_e.append(cc.ravel())
    rows_e = np.concatenate(rows_e).astype(np.int64)
    cols_e = np.concatenate(cols_e).astype(np.int64)
    if mask is not None:
        mask[rows_e, cols_e] = True
    total = M * N
    gen = torch.Generator(device="cpu").manual_seed(int(seed) + 1000)
    want = min(count, total - rows_e.size)
    picked = np.empty(0, dtype=np.int64)
    draws = max(2 * want, 1024)
    while picked.size < want:
        r = torch.randint(0, total, (draws,), generator=gen).numpy()
        _, first = np.unique(r, return_index=True)
        r = r[np.sort(first)]
        if mask is not None:
            r = r[~mask.ravel()[r]]
        else:
            rm, cm = r // N, r % N
            in_edge = (rm < edge) | (rm >= M - edge) | (cm < edge) | (cm >= N - edge)
            r = r[~in_edge]
        if picked.size:
            r = r[~np.isin(r, picked)]   # keeps draw order
        picked = np.concatenate([picked, r])[:want]
    rows = np.concatenate([rows_e, picked // N])
    cols = np.concatenate([cols_e, picked % N])
    return rows, cols
