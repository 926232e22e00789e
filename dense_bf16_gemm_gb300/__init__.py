"""GB300 (sm_103a) dense BF16 GEMM and fused gate/up projection.

The computation runs in the CUDA library declared by ``include/gemm_bf16.h``
(tcgen05 tensor cores, TMA, Tensor Memory).  This module only marshals torch
tensors into that C ABI: PyTorch supplies device memory and streams.

    C = alpha * A @ B + beta * C       gemm(A, B, C, alpha, beta)   (2-D or batched 3-D,
                                                                     BF16 or FP16 operands)
    ... and row sum/max/min of it      gemm_row_stats(A, B, C, alpha, beta)
    Y = silu(X @ Wg) * (X @ Wu)        gate_up_silu(X, Wg, Wu)
    Y = x / rms(x) * g  (per row)      rms_norm(X, G, eps)
    Y = gate_up_silu(rms_norm(X), ..)  rmsnorm_gate_up_silu(X, G, eps, Wg, Wu)
    O = softmax(s Q.K^T) . V per head  attention(Q, K, V, scale)

Operands are K-contiguous: ``A`` is (M, K) and ``B`` is passed as its (N, K)
storage, so ``gemm(A, B)`` equals ``A @ B.T`` in torch notation.
"""
from __future__ import annotations

import torch

from . import _native
from ._native import (GEMM_ERR_ALIGNMENT, GEMM_ERR_CUDA, GEMM_ERR_INVALID_ARG,  # noqa: F401
                      GEMM_ERR_TIMEOUT, GEMM_ERR_UNSUPPORTED, GEMM_IN_BF16, GEMM_IN_F16,
                      GEMM_OK, GEMM_OUT_BF16, GEMM_OUT_F16, GEMM_OUT_F32, GemmError)

__all__ = ["gemm", "gemm_row_stats", "gate_up_silu", "rms_norm", "rmsnorm_gate_up_silu", "attention",
           "device_status", "plan", "batched_plan", "row_stats_plan", "gate_up_plan", "prepare",
           "GemmError", "library_path"]

_OUT_CODES = {torch.float32: GEMM_OUT_F32, torch.bfloat16: GEMM_OUT_BF16,
              torch.float16: GEMM_OUT_F16}
_IN_CODES = {torch.bfloat16: GEMM_IN_BF16, torch.float16: GEMM_IN_F16}


def library_path() -> str:
    return _native.library_path()


def _stream(stream, device) -> int:
    if stream is None:
        stream = torch.cuda.current_stream(device)
    return int(stream.cuda_stream)


def _check_operand(name, t, dtypes=(torch.bfloat16,), dims=(2,)):
    if not isinstance(t, torch.Tensor):
        raise TypeError(f"{name} must be a tensor")
    if not t.is_cuda:
        raise ValueError(f"{name} must be a CUDA tensor (there is no CPU path)")
    if t.dtype not in dtypes:
        raise TypeError(f"{name} must be one of {dtypes}, got {t.dtype}")
    if t.dim() not in dims or (t.numel() > 0 and t.stride(-1) != 1):
        raise ValueError(f"{name} must be {dims}-D with a contiguous last dimension")


def _ld(t) -> int:
    """Row pitch in elements of a (.., rows, cols) tensor."""
    return max(t.stride(-2), t.shape[-1]) if t.numel() > 0 else t.shape[-1]


def _bstride(t) -> int:
    return t.stride(0) if t.dim() == 3 else 0


def _gemm_operands(A, B, C, beta, out_dtype):
    """Checks A, B (and C, created when None); returns (C, batched, batch, M, N, K)."""
    _check_operand("A", A, tuple(_IN_CODES), (2, 3))
    _check_operand("B", B, tuple(_IN_CODES), (A.dim(),))
    if B.dtype != A.dtype:
        raise TypeError("A and B must have the same dtype")
    batched = A.dim() == 3
    batch = A.shape[0] if batched else 1
    M, K = A.shape[-2:]
    N, K2 = B.shape[-2:]
    if K2 != K or (batched and B.shape[0] != batch):
        raise ValueError(f"shapes differ: A {tuple(A.shape)}, B {tuple(B.shape)}")
    shape = (batch, M, N) if batched else (M, N)
    if C is None:
        if beta != 0.0:
            raise ValueError("beta != 0 needs an input C")
        C = torch.empty(shape, dtype=out_dtype or A.dtype, device=A.device)
    else:
        if out_dtype is not None and C.dtype != out_dtype:
            raise TypeError("C dtype and out_dtype differ")
        _check_operand("C", C, tuple(_OUT_CODES), (A.dim(),))
        if tuple(C.shape) != shape:
            raise ValueError(f"C must be {shape}")
    return C, batched, batch, M, N, K


def gemm(A: torch.Tensor, B: torch.Tensor, C: torch.Tensor | None = None,
         alpha: float = 1.0, beta: float = 0.0, out_dtype: torch.dtype | None = None,
         stream: torch.cuda.Stream | None = None) -> torch.Tensor:
    """``C = alpha * A.B + beta * C`` with FP32 accumulation.

    A: (M, K) or a batch (b, M, K).  B: (N, K) or (b, N, K): the K-contiguous
    storage of the (K, N) operand.  A and B are both bfloat16 or both float16.
    C: (M, N) or (b, M, N), float32, bfloat16 or float16; created when None
    (then ``beta`` must be 0).  Asynchronous on ``stream`` (default: current).
    """
    C, batched, batch, M, N, K = _gemm_operands(A, B, C, beta, out_dtype)
    code = _OUT_CODES[C.dtype]
    with torch.cuda.device(A.device):
        if not batched and A.dtype == torch.bfloat16:
            st = _native.gemm_bf16(M, N, K, float(alpha), A.data_ptr(), _ld(A), B.data_ptr(),
                                   _ld(B), float(beta), C.data_ptr(), _ld(C), code,
                                   _stream(stream, A.device))
        else:
            st = _native.gemm_batched(batch, M, N, K, float(alpha), A.data_ptr(), _ld(A),
                                      _bstride(A), B.data_ptr(), _ld(B), _bstride(B),
                                      float(beta), C.data_ptr(), _ld(C), _bstride(C),
                                      _IN_CODES[A.dtype], code, _stream(stream, A.device))
    if st != GEMM_OK:
        raise GemmError(st, "gemm")
    return C


def gemm_row_stats(A: torch.Tensor, B: torch.Tensor, C: torch.Tensor | None = None,
                   alpha: float = 1.0, beta: float = 0.0, out_dtype: torch.dtype | None = None,
                   stream: torch.cuda.Stream | None = None, stats=None):
    """``gemm`` plus the sum, maximum and minimum along each row of the FP32
    result (before its output rounding).

    Returns ``(C, row_sum, row_max, row_min)``; the three are float32 of
    shape (M,) or (b, M), created unless ``stats`` gives them (any may be
    None there: that reduction is not written).
    """
    C, batched, batch, M, N, K = _gemm_operands(A, B, C, beta, out_dtype)
    lead = (batch, M) if batched else (M,)
    if stats is None:
        stats = [torch.empty(lead, dtype=torch.float32, device=A.device) for _ in range(3)]
    stats = list(stats)
    for t in stats:
        if t is not None and (not t.is_cuda or t.dtype != torch.float32 or
                              tuple(t.shape) != lead or not t.is_contiguous()):
            raise ValueError(f"row statistics must be contiguous CUDA float32 {lead}")
    with torch.cuda.device(A.device):
        st = _native.gemm_row_stats(batch, M, N, K, float(alpha), A.data_ptr(), _ld(A),
                                    _bstride(A), B.data_ptr(), _ld(B), _bstride(B),
                                    float(beta), C.data_ptr(), _ld(C), _bstride(C),
                                    _IN_CODES[A.dtype], _OUT_CODES[C.dtype],
                                    *(t.data_ptr() if t is not None else 0 for t in stats),
                                    _stream(stream, A.device))
    if st != GEMM_OK:
        raise GemmError(st, "gemm_row_stats")
    return (C, *stats)


def rms_norm(X: torch.Tensor, G: torch.Tensor, eps: float = 1e-6, Y: torch.Tensor | None = None,
             out_dtype: torch.dtype | None = None,
             stream: torch.cuda.Stream | None = None) -> torch.Tensor:
    """``Y = X * rsqrt(mean(X^2, dim=1) + eps) * G`` row by row.

    X: (rows, D) float32, bfloat16 or float16; G: (D,) float32; Y: (rows, D)
    created when None (dtype ``out_dtype``, default X's).  Y may be X itself.
    """
    _check_operand("X", X, tuple(_OUT_CODES))
    rows, D = X.shape
    if not isinstance(G, torch.Tensor) or not G.is_cuda or G.dtype != torch.float32 or \
            G.numel() != D or not G.is_contiguous():
        raise ValueError("G must be a contiguous CUDA float32 tensor of D gains")
    if Y is None:
        Y = torch.empty((rows, D), dtype=out_dtype or X.dtype, device=X.device)
    else:
        _check_operand("Y", Y, tuple(_OUT_CODES))
        if tuple(Y.shape) != (rows, D):
            raise ValueError(f"Y must be ({rows}, {D})")
    with torch.cuda.device(X.device):
        st = _native.gemm_rms_norm(rows, D, X.data_ptr(), _ld(X), _OUT_CODES[X.dtype],
                                   G.data_ptr(), float(eps), Y.data_ptr(), _ld(Y),
                                   _OUT_CODES[Y.dtype], _stream(stream, X.device))
    if st != GEMM_OK:
        raise GemmError(st, "gemm_rms_norm")
    return Y


def rmsnorm_gate_up_silu(X: torch.Tensor, G: torch.Tensor, eps: float, Wg: torch.Tensor,
                         Wu: torch.Tensor, Xn: torch.Tensor | None = None,
                         Y: torch.Tensor | None = None,
                         stream: torch.cuda.Stream | None = None):
    """``Y = silu(Xn.Wg) * (Xn.Wu)`` with ``Xn = rms_norm(X, G, eps)`` (BF16).

    X (M, K) bf16, G (K,) float32, Wg/Wu stored (N, K) bf16.  Returns (Y, Xn);
    Xn is created when None (it may be X itself for an in-place normalisation).
    """
    _check_operand("X", X)
    _check_operand("Wg", Wg)
    _check_operand("Wu", Wu)
    M, K = X.shape
    N = Wg.shape[0]
    if tuple(Wg.shape) != (N, K) or tuple(Wu.shape) != (N, K) or Wg.stride(0) != Wu.stride(0):
        raise ValueError("Wg and Wu must both be (N, K) with one row pitch")
    if not isinstance(G, torch.Tensor) or not G.is_cuda or G.dtype != torch.float32 or \
            G.numel() != K or not G.is_contiguous():
        raise ValueError("G must be a contiguous CUDA float32 tensor of K gains")
    if Xn is None:
        Xn = torch.empty((M, K), dtype=torch.bfloat16, device=X.device)
    else:
        _check_operand("Xn", Xn)
        if tuple(Xn.shape) != (M, K):
            raise ValueError(f"Xn must be ({M}, {K})")
    if Y is None:
        Y = torch.empty((M, N), dtype=torch.bfloat16, device=X.device)
    else:
        _check_operand("Y", Y)
        if tuple(Y.shape) != (M, N):
            raise ValueError(f"Y must be ({M}, {N})")
    with torch.cuda.device(X.device):
        st = _native.gemm_rmsnorm_gate_up_silu(M, N, K, X.data_ptr(), _ld(X), G.data_ptr(),
                                               float(eps), Wg.data_ptr(), Wu.data_ptr(), _ld(Wg),
                                               Xn.data_ptr(), _ld(Xn), Y.data_ptr(), _ld(Y),
                                               _stream(stream, X.device))
    if st != GEMM_OK:
        raise GemmError(st, "gemm_rmsnorm_gate_up_silu")
    return Y, Xn


def attention(Q: torch.Tensor, K: torch.Tensor, V: torch.Tensor, scale: float | None = None,
              O: torch.Tensor | None = None, out_dtype: torch.dtype = torch.bfloat16,
              stream: torch.cuda.Stream | None = None) -> torch.Tensor:
    """``O = softmax(scale * Q.K^T) . V`` per head (softmax over the keys).

    Q: (heads, Nq, D) or (Nq, D); K, V: (heads, Nk, D) or (Nk, D); bfloat16,
    D = 64 or 128.  ``scale`` defaults to 1/sqrt(D).  O: created when None
    (``out_dtype`` float32 or bfloat16).
    """
    squeeze = Q.dim() == 2
    if squeeze:
        Q, K, V = Q.unsqueeze(0), K.unsqueeze(0), V.unsqueeze(0)
        if O is not None:
            O = O.unsqueeze(0)
    for name, t in (("Q", Q), ("K", K), ("V", V)):
        _check_operand(name, t, (torch.bfloat16,), (3,))
    H, Nq, D = Q.shape
    Nk = K.shape[1]
    if tuple(K.shape) != (H, Nk, D) or tuple(V.shape) != (H, Nk, D):
        raise ValueError("K and V must be (heads, Nk, D) with Q's heads and D")
    if scale is None:
        scale = D ** -0.5
    if O is None:
        O = torch.empty((H, Nq, D), dtype=out_dtype, device=Q.device)
    else:
        _check_operand("O", O, (torch.float32, torch.bfloat16), (3,))
        if tuple(O.shape) != (H, Nq, D):
            raise ValueError(f"O must be {(H, Nq, D)}")
    with torch.cuda.device(Q.device):
        st = _native.gemm_attention(H, Nq, Nk, D, float(scale), Q.data_ptr(), _ld(Q), _bstride(Q),
                                    K.data_ptr(), _ld(K), _bstride(K), V.data_ptr(), _ld(V),
                                    _bstride(V), O.data_ptr(), _ld(O), _bstride(O),
                                    _OUT_CODES[O.dtype], _stream(stream, Q.device))
    if st != GEMM_OK:
        raise GemmError(st, "gemm_attention")
    return O[0] if squeeze else O


def gate_up_silu(X: torch.Tensor, Wg: torch.Tensor, Wu: torch.Tensor,
                 Y: torch.Tensor | None = None,
                 stream: torch.cuda.Stream | None = None) -> torch.Tensor:
    """``Y = silu(X.Wg) * (X.Wu)``; X (M, K), Wg and Wu stored (N, K), Y (M, N), all bf16."""
    _check_operand("X", X)
    _check_operand("Wg", Wg)
    _check_operand("Wu", Wu)
    M, K = X.shape
    N = Wg.shape[0]
    if tuple(Wg.shape) != (N, K) or tuple(Wu.shape) != (N, K):
        raise ValueError("Wg and Wu must both be (N, K)")
    if Wg.stride(0) != Wu.stride(0):
        raise ValueError("Wg and Wu must share a row pitch")
    if Y is None:
        Y = torch.empty((M, N), dtype=torch.bfloat16, device=X.device)
    else:
        _check_operand("Y", Y)
        if tuple(Y.shape) != (M, N):
            raise ValueError(f"Y must be ({M}, {N})")
    with torch.cuda.device(X.device):
        st = _native.gemm_gate_up_silu(M, N, K, X.data_ptr(), _ld(X), Wg.data_ptr(),
                                       Wu.data_ptr(), _ld(Wg), Y.data_ptr(), _ld(Y),
                                       _stream(stream, X.device))
    if st != GEMM_OK:
        raise GemmError(st, "gemm_gate_up_silu")
    return Y


def device_status(stream: torch.cuda.Stream | None = None, device=None):
    """Synchronize ``stream`` and return (status, site) of the device status
    word, clearing it."""
    dev = torch.device("cuda", torch.cuda.current_device()) if device is None else device
    with torch.cuda.device(dev):
        return _native.gemm_get_device_status(_stream(stream, dev))


def prepare(max_n: int, stream: torch.cuda.Stream | None = None, device=None) -> None:
    """Allocate the split-K workspace for M <= 16 calls up to ``max_n`` columns."""
    dev = torch.device("cuda", torch.cuda.current_device()) if device is None else device
    with torch.cuda.device(dev):
        st = _native.gemm_prepare(int(max_n), _stream(stream, dev))
    if st != GEMM_OK:
        raise GemmError(st, "gemm_prepare")


def plan(M: int, N: int, K: int, out_dtype: torch.dtype = torch.bfloat16, num_sms: int = 0) -> dict:
    """How ``gemm`` would run a problem (host-side planning)."""
    st, p = _native.gemm_bf16_plan(M, N, K, _OUT_CODES[out_dtype], num_sms)
    if st != GEMM_OK:
        raise GemmError(st, "gemm_bf16_plan")
    return p.as_dict()


def batched_plan(batch: int, M: int, N: int, K: int, in_dtype: torch.dtype = torch.bfloat16,
                 out_dtype: torch.dtype = torch.bfloat16, num_sms: int = 0) -> dict:
    """How ``gemm`` would run a batch of problems (host-side planning)."""
    st, p = _native.gemm_batched_plan(batch, M, N, K, _IN_CODES[in_dtype], _OUT_CODES[out_dtype],
                                      num_sms)
    if st != GEMM_OK:
        raise GemmError(st, "gemm_batched_plan")
    return p.as_dict()


def row_stats_plan(batch: int, M: int, N: int, K: int, in_dtype: torch.dtype = torch.bfloat16,
                   out_dtype: torch.dtype = torch.bfloat16, num_sms: int = 0) -> dict:
    """How ``gemm_row_stats`` would run a batch of problems (host-side planning)."""
    st, p = _native.gemm_row_stats_plan(batch, M, N, K, _IN_CODES[in_dtype],
                                        _OUT_CODES[out_dtype], num_sms)
    if st != GEMM_OK:
        raise GemmError(st, "gemm_row_stats_plan")
    return p.as_dict()


def gate_up_plan(M: int, N: int, K: int, num_sms: int = 0) -> dict:
    st, p = _native.gemm_gate_up_plan(M, N, K, num_sms)
    if st != GEMM_OK:
        raise GemmError(st, "gemm_gate_up_plan")
    return p.as_dict()
