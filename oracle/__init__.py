"""CPU oracle for the dense BF16 GEMM and the fused gate/up projection.

TEST INFRASTRUCTURE ONLY.  Only ``tests/``, ``__graft_entry__.smoke()`` and the
CPU-baseline leg of ``bench.py`` may import this package.  The product library
(``dense_bf16_gemm_gb300``) never imports, links or runs anything here, and this
package never imports the product: the two share no code.

Contents
--------
* ``gemm_full`` / ``gemm_entries``: ``alpha * A.B + beta * C`` in float64 from
  the BF16 inputs, one running double sum per output (C implementation in
  ``gemm_oracle.c``).  The epilogue semantics follow "Tiles and shared memory",
  section "var and let" (``C[...] = alpha * acc + beta * c_old``); the operand
  storage follows "TMA and Hopper WGMMA", section "The same storage contract
  on both sides" (A(M,K) with K contiguous, B(K,N) stored with K inner, i.e.
  ``B[n*ldb + k]``).
* ``gate_up_entries``: ``silu(X.Wg) * (X.Wu)`` in float64 ("TMA and Hopper
  WGMMA", sections "TMA and Hopper WGMMA" and "Worked consumers and current
  validation", which name the fused gate/up projection; it is read as the
  SwiGLU form with no bias and no scaling).
* FP16 operands (``in_f16``) are decoded exactly as IEEE binary16; FP16
  outputs are rounded with ``round_to_f16_bits`` ("TMEM tiles and transfers",
  section "Representation and windows": pack(Float16, f)).
* ``bf16_bits_to_f64`` / ``round_to_bf16_bits``: exact BF16 widening and
  round-to-nearest-even narrowing ("TMEM tiles and transfers", section
  "Representation and windows": ``pack(BFloat16, f)`` converts FP32 values to
  BF16; the rounding mode is not stated there and is read as nearest-even).
* ``rms_norm``: ``y = x * inv * g`` with ``inv = 1/sqrt(mean_k x^2 + eps)``
  per row ("Tiles and shared memory", section "A complete kernel").
* ``rmsnorm_gate_up_entries``: the gate/up projection of ``rms_norm(X)``, the
  normalised activation kept in float64 (the steps on either side of the
  projection).
* ``gemm_row_stats``: sum, maximum and minimum along each row of
  ``alpha * A.B + beta * C`` ("TMEM tiles and transfers", section "Storage and
  a transfer": a reduction along the second axis of a loaded accumulator;
  "TMA and Hopper WGMMA", section "WGMMA values and ownership": sum, maximum
  and minimum along axis 2 of a finished accumulator), over the whole row.
* ``attention_rows``: ``softmax(scale * q.K^T) . V`` for chosen query rows
  ("Tiles and shared memory", section "How long a tile lives": the
  flash-attention loop with a running maximum and sum, finished by acc / l),
  evaluated directly over all keys.
* ``gemm_tolerance`` / ``gate_up_tolerance`` / ``rms_norm_tolerance`` /
  ``row_stats_tolerance`` / ``attention_tolerance``: the admissible distance
  between a result computed in FP32 and the float64 reference.

Every function here is pinned in ``tests/test_oracle.py`` to closed forms,
identities, brute force on tiny shapes and library routines.
"""
from __future__ import annotations

import ctypes
import os
import subprocess
import threading

import numpy as np

_HERE = os.path.dirname(os.path.abspath(__file__))
_SRC = os.path.join(_HERE, "gemm_oracle.c")
_BUILD_DIR = os.path.join(_HERE, "_build")
_LIB_PATH = os.path.join(_BUILD_DIR, "liboracle.so")

_lock = threading.Lock()
_lib = None

_i64 = ctypes.c_int64
_dbl = ctypes.c_double
_vp = ctypes.c_void_p


def build(force: bool = False) -> str:
    """Compile the C oracle with the host compiler (plain -O2, OpenMP)."""
    if not force and os.path.exists(_LIB_PATH) and \
            os.path.getmtime(_LIB_PATH) >= os.path.getmtime(_SRC):
        return _LIB_PATH
    os.makedirs(_BUILD_DIR, exist_ok=True)
    tmp = _LIB_PATH + f".tmp{os.getpid()}"
    cmd = ["gcc", "-O2", "-fopenmp", "-fPIC", "-shared", "-std=c99",
           "-o", tmp, _SRC, "-lm"]
    subprocess.run(cmd, check=True)
    os.replace(tmp, _LIB_PATH)
    return _LIB_PATH


def _load():
    global _lib
    with _lock:
        if _lib is None:
            build()
            lib = ctypes.CDLL(_LIB_PATH)
            lib.oracle_num_threads.restype = ctypes.c_int
            lib.oracle_silu.restype = _dbl
            lib.oracle_silu.argtypes = [_dbl]
            lib.oracle_gemm_entries.restype = None
            lib.oracle_gemm_entries.argtypes = [
                _i64, _dbl, _vp, _i64, _vp, _i64, _dbl, _vp, _i64,
                _i64, _vp, _vp, _vp, _vp, ctypes.c_int]
            lib.oracle_gemm_full.restype = None
            lib.oracle_gemm_full.argtypes = [
                _i64, _i64, _i64, _dbl, _vp, _i64, _vp, _i64, _dbl, _vp, _i64,
                _vp, _vp, ctypes.c_int]
            lib.oracle_decode16.restype = _dbl
            lib.oracle_decode16.argtypes = [ctypes.c_uint16, ctypes.c_int]
            lib.oracle_rms_norm_rows.restype = None
            lib.oracle_rms_norm_rows.argtypes = [
                _i64, _vp, _i64, ctypes.c_int, _vp, _dbl, _i64, _vp, _vp, _vp]
            lib.oracle_gate_up_entries_f64.restype = None
            lib.oracle_gate_up_entries_f64.argtypes = [
                _i64, _vp, _i64, _vp, _vp, _i64,
                _i64, _vp, _vp, _vp, _vp, _vp, _vp, _vp]
            lib.oracle_attention_rows.restype = None
            lib.oracle_attention_rows.argtypes = [
                _i64, _i64, _i64, _dbl, _vp, _vp, _vp, _i64, _vp, _vp, _vp, _vp, _vp]
            lib.oracle_gate_up_entries.restype = None
            lib.oracle_gate_up_entries.argtypes = [
                _i64, _vp, _i64, _vp, _vp, _i64,
                _i64, _vp, _vp, _vp, _vp, _vp, _vp, _vp]
            _lib = lib
    return _lib


def num_threads() -> int:
    """OpenMP threads the oracle uses (``OMP_NUM_THREADS`` or all cores)."""
    return int(_load().oracle_num_threads())


def _ptr(a: np.ndarray | None):
    return None if a is None else a.ctypes.data


def _as_bits(x) -> np.ndarray:
    """Accept a uint16 array of 16-bit patterns or a torch bfloat16/float16 tensor."""
    if isinstance(x, np.ndarray):
        if x.dtype != np.uint16:
            raise TypeError("16-bit operands are passed as uint16 bit patterns")
        return np.ascontiguousarray(x)
    import torch  # only for accepting CPU tensors from the input generator
    if not isinstance(x, torch.Tensor) or x.dtype not in (torch.bfloat16, torch.float16):
        raise TypeError("expected a bfloat16/float16 tensor or uint16 bits")
    return np.ascontiguousarray(x.contiguous().view(torch.int16).numpy()).view(np.uint16)


def _is_f16(*xs) -> int:
    """1 when the operands are float16 tensors (uint16 bits are BF16 unless
    in_f16 is given explicitly)."""
    try:
        import torch
    except ImportError:  # pragma: no cover
        return 0
    kinds = {x.dtype for x in xs if isinstance(x, torch.Tensor)}
    if len(kinds) > 1:
        raise TypeError("operands must share one type")
    return 1 if kinds == {torch.float16} else 0


def decode16(bits: int, in_f16: bool) -> float:
    """Exact value of a BF16 (in_f16 False) or FP16 bit pattern, from the C oracle."""
    return float(_load().oracle_decode16(int(bits) & 0xFFFF, int(bool(in_f16))))


def _as_f32(x) -> np.ndarray | None:
    if x is None:
        return None
    if isinstance(x, np.ndarray):
        return np.ascontiguousarray(x, dtype=np.float32)
    return np.ascontiguousarray(x.contiguous().numpy(), dtype=np.float32)


# --------------------------------------------------------------------------
# GEMM
# --------------------------------------------------------------------------
def gemm_full(A, B, alpha=1.0, beta=0.0, C=None, want_abs=True, in_f16=None):
    """Every entry of ``alpha * A.B + beta * C``.

    ``A`` is (M, K) K-contiguous, ``B`` is stored (N, K) K-contiguous, ``C`` is
    (M, N) float32 (read only when ``beta != 0``).  Returns ``(value, abs_sum)``
    as float64 (M, N) arrays, ``abs_sum[m, n] = sum_k |a(m,k) b(k,n)|``.
    """
    f16 = _is_f16(A, B) if in_f16 is None else int(bool(in_f16))
    a, b = _as_bits(A), _as_bits(B)
    M, K = a.shape
    N, K2 = b.shape
    if K2 != K:
        raise ValueError("inner dimensions differ")
    c = _as_f32(C) if beta != 0.0 else None
    if beta != 0.0 and (c is None or c.shape != (M, N)):
        raise ValueError("C must be (M, N) when beta != 0")
    out = np.empty((M, N), np.float64)
    ab = np.empty((M, N), np.float64) if want_abs else None
    _load().oracle_gemm_full(M, N, K, float(alpha), _ptr(a), K, _ptr(b), K,
                             float(beta), _ptr(c), N, _ptr(out), _ptr(ab), f16)
    return out, ab


def gemm_entries(A, B, rows, cols, alpha=1.0, beta=0.0, C=None, in_f16=None):
    """Entries ``(rows[i], cols[i])`` of ``alpha * A.B + beta * C``.

    Same storage as :func:`gemm_full`; returns ``(value, abs_sum)`` 1-D arrays.
    """
    f16 = _is_f16(A, B) if in_f16 is None else int(bool(in_f16))
    a, b = _as_bits(A), _as_bits(B)
    M, K = a.shape
    N, K2 = b.shape
    if K2 != K:
        raise ValueError("inner dimensions differ")
    r = np.ascontiguousarray(rows, dtype=np.int64)
    c_ = np.ascontiguousarray(cols, dtype=np.int64)
    if r.shape != c_.shape:
        raise ValueError("rows and cols differ in length")
    if r.size and (r.min() < 0 or r.max() >= M or c_.min() < 0 or c_.max() >= N):
        raise IndexError("entry outside the result")
    cm = _as_f32(C) if beta != 0.0 else None
    out = np.empty(r.size, np.float64)
    ab = np.empty(r.size, np.float64)
    _load().oracle_gemm_entries(K, float(alpha), _ptr(a), K, _ptr(b), K,
                                float(beta), _ptr(cm), N, r.size, _ptr(r),
                                _ptr(c_), _ptr(out), _ptr(ab), f16)
    return out, ab


# --------------------------------------------------------------------------
# gate/up projection
# --------------------------------------------------------------------------
def silu(t: float) -> float:
    """``t / (1 + exp(-t))`` evaluated by the C oracle in double."""
    return float(_load().oracle_silu(float(t)))


def gate_up_entries(X, Wg, Wu, rows, cols):
    """Entries of ``Y = silu(X.Wg) * (X.Wu)``.

    ``X`` is (M, K) K-contiguous, ``Wg`` and ``Wu`` are stored (N, K)
    K-contiguous.  Returns a dict with float64 arrays ``y``, ``g``, ``u``,
    ``abs_g``, ``abs_u``.
    """
    x, wg, wu = _as_bits(X), _as_bits(Wg), _as_bits(Wu)
    M, K = x.shape
    N = wg.shape[0]
    if wg.shape != (N, K) or wu.shape != (N, K):
        raise ValueError("weights must both be (N, K)")
    r = np.ascontiguousarray(rows, dtype=np.int64)
    c_ = np.ascontiguousarray(cols, dtype=np.int64)
    if r.size and (r.min() < 0 or r.max() >= M or c_.min() < 0 or c_.max() >= N):
        raise IndexError("entry outside the result")
    res = {k: np.empty(r.size, np.float64) for k in ("y", "g", "u", "abs_g", "abs_u")}
    _load().oracle_gate_up_entries(K, _ptr(x), K, _ptr(wg), _ptr(wu), K,
                                   r.size, _ptr(r), _ptr(c_),
                                   _ptr(res["y"]), _ptr(res["g"]), _ptr(res["u"]),
                                   _ptr(res["abs_g"]), _ptr(res["abs_u"]))
    return res


# --------------------------------------------------------------------------
# row normalisation and the reductions along a row
# --------------------------------------------------------------------------
def _norm_input(X):
    """(array, kind) of a normalisation input: kind 0 FP32, 1 BF16, 2 FP16."""
    if isinstance(X, np.ndarray):
        if X.dtype == np.float32:
            return np.ascontiguousarray(X), 0
        raise TypeError("numpy inputs to rms_norm are float32")
    import torch
    if X.dtype == torch.float32:
        return np.ascontiguousarray(X.contiguous().numpy()), 0
    return _as_bits(X), (2 if X.dtype == torch.float16 else 1)


def rms_norm(X, G, eps: float, rows=None):
    """Rows of ``y = x * inv * g``, ``inv = 1/sqrt(sum_k x^2 / D + eps)``.

    ``X`` is (M, D) FP32, BF16 or FP16 (a torch tensor, or float32 numpy);
    ``G`` holds D FP32 gains.  Returns ``(y, inv)``: float64 arrays of shape
    (len(rows), D) and (len(rows),); all rows when ``rows`` is None.
    """
    x, kind = _norm_input(X)
    M, D = x.shape
    g = _as_f32(G).reshape(-1)
    if g.size != D:
        raise ValueError("G must hold D gains")
    r = np.arange(M, dtype=np.int64) if rows is None else \
        np.ascontiguousarray(rows, dtype=np.int64)
    if r.size and (r.min() < 0 or r.max() >= M):
        raise IndexError("row outside X")
    y = np.empty((r.size, D), np.float64)
    inv = np.empty(r.size, np.float64)
    _load().oracle_rms_norm_rows(D, _ptr(x), D, kind, _ptr(g), float(eps), r.size, _ptr(r),
                                 _ptr(y), _ptr(inv))
    return y, inv


def rmsnorm_gate_up_entries(X, G, eps: float, Wg, Wu, rows, cols):
    """Entries of ``silu(Xn.Wg) * (Xn.Wu)`` with ``Xn = rms_norm(X, G, eps)``
    kept in float64.  Same result dict as :func:`gate_up_entries`."""
    r = np.ascontiguousarray(rows, dtype=np.int64)
    c_ = np.ascontiguousarray(cols, dtype=np.int64)
    wg, wu = _as_bits(Wg), _as_bits(Wu)
    N, K = wg.shape
    if wu.shape != (N, K) or X.shape[1] != K:
        raise ValueError("weights must both be (N, K) with K = X's columns")
    if c_.size and (c_.min() < 0 or c_.max() >= N):
        raise IndexError("entry outside the result")
    uniq, xrows = np.unique(r, return_inverse=True)
    xn, _ = rms_norm(X, G, eps, uniq)
    xrows = np.ascontiguousarray(xrows, dtype=np.int64)
    res = {k: np.empty(r.size, np.float64) for k in ("y", "g", "u", "abs_g", "abs_u")}
    _load().oracle_gate_up_entries_f64(K, _ptr(xn), K, _ptr(wg), _ptr(wu), K,
                                       r.size, _ptr(xrows), _ptr(c_),
                                       _ptr(res["y"]), _ptr(res["g"]), _ptr(res["u"]),
                                       _ptr(res["abs_g"]), _ptr(res["abs_u"]))
    return res


def gemm_row_stats(A, B, rows, alpha=1.0, beta=0.0, C=None, in_f16=None):
    """Sum, maximum and minimum over n of ``alpha * A.B + beta * C`` for each
    row in ``rows`` (whole rows, from :func:`gemm_entries`).

    Returns a dict of float64 arrays over ``rows``: ``sum``, ``max``, ``min``,
    and for the tolerance ``abs_sum`` (the (len(rows), N) array of
    ``sum_k |a b|``), ``values`` (the (len(rows), N) results) and ``c``
    (the matching entries of C, or None).
    """
    r = np.ascontiguousarray(rows, dtype=np.int64)
    N = B.shape[0]
    rr = np.repeat(r, N)
    cc = np.tile(np.arange(N, dtype=np.int64), r.size)
    v, ab = gemm_entries(A, B, rr, cc, alpha=alpha, beta=beta, C=C, in_f16=in_f16)
    v = v.reshape(r.size, N)
    cm = None
    if beta != 0.0 and C is not None:
        cm = _as_f32(C)[r].astype(np.float64)
    return {"sum": v.sum(axis=1), "max": v.max(axis=1), "min": v.min(axis=1),
            "values": v, "abs_sum": ab.reshape(r.size, N), "c": cm}


# --------------------------------------------------------------------------
# attention
# --------------------------------------------------------------------------
def attention_rows(Q, K, V, scale: float, heads, rows):
    """Rows of ``O = softmax(scale * Q.K^T) . V`` per head.

    ``Q`` is (H, Nq, D), ``K`` and ``V`` are (H, Nk, D), BF16 (torch tensors or
    uint16 bits); ``heads[i]``, ``rows[i]`` name the query rows.  Returns a
    dict of float64 arrays: ``o`` and ``abs_o`` (len(rows), D) and ``smax``
    (len(rows),): ``abs_o = sum_j w_j |v_j|`` with the softmax weights w and
    ``smax = |scale| max_j sum_d |q_d k_jd|``, both for the tolerance.
    """
    q, k, v = _as_bits(Q), _as_bits(K), _as_bits(V)
    H, Nq, D = q.shape
    _, Nk, _ = k.shape
    if k.shape != (H, Nk, D) or v.shape != (H, Nk, D):
        raise ValueError("K and V must be (H, Nk, D) with Q's H and D")
    if Nk < 1:
        raise ValueError("attention needs at least one key")
    h = np.ascontiguousarray(heads, dtype=np.int64)
    r = np.ascontiguousarray(rows, dtype=np.int64)
    if h.shape != r.shape:
        raise ValueError("heads and rows differ in length")
    if r.size and (h.min() < 0 or h.max() >= H or r.min() < 0 or r.max() >= Nq):
        raise IndexError("query row outside Q")
    o = np.empty((r.size, D), np.float64)
    ab = np.empty((r.size, D), np.float64)
    smax = np.empty(r.size, np.float64)
    _load().oracle_attention_rows(Nq, Nk, D, float(scale), _ptr(q), _ptr(k), _ptr(v), r.size,
                                  _ptr(h), _ptr(r), _ptr(o), _ptr(ab), _ptr(smax))
    return {"o": o, "abs_o": ab, "smax": smax}


# --------------------------------------------------------------------------
# BF16 encoding
# --------------------------------------------------------------------------
def bf16_bits_to_f64(bits) -> np.ndarray:
    """Exact value of BF16 bit patterns (the upper half of a binary32)."""
    b = np.asarray(bits, dtype=np.uint16).astype(np.uint32) << np.uint32(16)
    with np.errstate(invalid="ignore"):
        return b.view(np.float32).astype(np.float64)


def round_to_bf16_bits(x) -> np.ndarray:
    """Round float64 values to the nearest BF16, ties to even; NaN -> 0x7FC0.

    BF16 keeps 8 significant bits and the binary32 exponent range: normal
    values have spacing ``2**(e-7)`` in the binade ``[2**e, 2**(e+1))`` and the
    subnormal spacing is ``2**-133``.  The value is divided by the spacing,
    rounded half-to-even to an integer (exact in float64), scaled back
    (exact) and re-encoded; results beyond the largest finite BF16 become
    infinities, as nearest-even rounding prescribes.
    """
    v = np.asarray(x, dtype=np.float64)
    out = np.zeros(v.shape, dtype=np.uint16)
    nan = np.isnan(v)
    fin = np.isfinite(v)
    with np.errstate(over="ignore", invalid="ignore", divide="ignore"):
        mag = np.abs(np.where(fin, v, 0.0))
        _, e = np.frexp(mag)               # mag = f * 2**e, f in [0.5, 1)
        e = e - 1                          # binade exponent: mag in [2**e, 2**(e+1))
        spacing_exp = np.maximum(e - 7, -133)
        q = np.ldexp(1.0, spacing_exp)
        r = np.rint(mag / q) * q           # rint is half-to-even
        r32 = r.astype(np.float32)         # exact: r has <= 8 significant bits
        bits = (r32.view(np.uint32) >> np.uint32(16)).astype(np.uint16)
    sign = np.where(np.signbit(v), np.uint16(0x8000), np.uint16(0))
    out = np.where(fin, bits | sign, out)
    out = np.where(np.isinf(v), np.uint16(0x7F80) | sign, out)
    out = np.where(nan, np.uint16(0x7FC0), out)
    return out.astype(np.uint16)


def f16_bits_to_f64(bits) -> np.ndarray:
    """Exact value of IEEE binary16 bit patterns (numpy's float16)."""
    return np.asarray(bits, dtype=np.uint16).view(np.float16).astype(np.float64)


def round_to_f16_bits(x) -> np.ndarray:
    """Round float64 values to the nearest IEEE binary16, ties to even
    (numpy's float64 -> float16 conversion, pinned in the tests)."""
    with np.errstate(over="ignore", invalid="ignore"):
        return np.asarray(x, dtype=np.float64).astype(np.float16).view(np.uint16)


def f16_half_ulp(mag) -> np.ndarray:
    """Half the binary16 spacing at magnitude ``mag``: ``2**(floor(log2 mag) - 11)``,
    never below half the subnormal spacing (``2**-25``)."""
    m = np.abs(np.asarray(mag, dtype=np.float64))
    _, e = np.frexp(m)
    e = np.where(m == 0.0, -1000, e)   # zero: only the subnormal floor applies
    return np.maximum(np.ldexp(1.0, e - 1 - 11), np.ldexp(1.0, -25))


def bf16_half_ulp(mag) -> np.ndarray:
    """Half the BF16 spacing at magnitude ``mag``: ``2**(floor(log2 mag) - 8)``,
    never below half the subnormal spacing (``2**-134``)."""
    m = np.abs(np.asarray(mag, dtype=np.float64))
    _, e = np.frexp(m)
    e = np.where(m == 0.0, -1000, e)   # zero: only the subnormal floor applies
    return np.maximum(np.ldexp(1.0, e - 1 - 8), np.ldexp(1.0, -134))


# --------------------------------------------------------------------------
# tolerances
# --------------------------------------------------------------------------
REL_ACC = 4e-3      # admissible FP32-accumulation error per unit of sum |a b|
SILU_LIPSCHITZ = 1.1  # max |silu'(t)| = 1.0998... (at t ~ 2.3994)


def gemm_tolerance(ref, abs_sum, alpha, beta, c=None, out_bf16=False, out_f16=False):
    """``4e-3 * (|alpha| sum|ab| + |beta| |c|)`` plus, for a 16-bit output, the
    half-ulp of that format at the largest magnitude the FP32 result can take."""
    tol = REL_ACC * abs(alpha) * np.asarray(abs_sum, np.float64)
    if beta != 0.0 and c is not None:
        tol = tol + REL_ACC * abs(beta) * np.abs(np.asarray(c, np.float64))
    if out_bf16:
        tol = tol + bf16_half_ulp(np.abs(ref) + tol)
    if out_f16:
        tol = tol + f16_half_ulp(np.abs(ref) + tol)
    return tol


def gate_up_tolerance(res, rel: float = None):
    """Propagate the accumulation bound through ``silu(g) * u``.

    With ``|g' - g| <= e_g`` and ``|u' - u| <= e_u``:
    ``|silu(g')u' - silu(g)u| <= L e_g (|u| + e_u) + |silu(g)| e_u``, ``L`` the
    Lipschitz constant of silu.  ``1e-5 |y|`` covers the FP32 epilogue
    arithmetic (exp, divide, multiply) and the BF16 half-ulp the final
    rounding.
    """
    rel = REL_ACC if rel is None else rel
    g, u, y = res["g"], res["u"], res["y"]
    e_g = rel * res["abs_g"]
    e_u = rel * res["abs_u"]
    sg = np.abs(g / (1.0 + np.exp(-np.clip(g, -700, 700))))
    tol = SILU_LIPSCHITZ * e_g * (np.abs(u) + e_u) + sg * e_u + 1e-5 * np.abs(y)
    return tol + bf16_half_ulp(np.abs(y) + tol)


U32 = 2.0 ** -24    # unit roundoff of binary32


def rms_norm_rel_error(D: int) -> float:
    """Relative error bound of ``x * inv * g`` computed in FP32 against the
    exact value, for a row of D elements.

    The sum of squares is formed by 32 lanes, each adding at most
    ``ceil(D/32) + 1`` non-negative terms in order, then combined in 5
    pairwise steps: relative error at most ``gamma_n``, ``n = ceil(D/32) + 6``,
    ``gamma_n = n u / (1 - n u)``.  Dividing by D, adding eps, the square root
    and the reciprocal each add one rounding (the root halves the error of its
    argument), and the two products two more:
    ``gamma_n / 2 + 6 u`` in all, which this bound rounds up by 1 %.
    (When two warps share a row, each lane adds at most ``ceil(D/64) + 1``
    terms, then 5 pairwise steps and one more addition: a shorter chain, so
    the same bound holds.)
    """
    n = -(-int(D) // 32) + 6
    gamma = n * U32 / (1.0 - n * U32)
    return 1.01 * (gamma / 2.0 + 6.0 * U32)


def rms_norm_tolerance(y_ref, D: int, out_bf16=False, out_f16=False):
    """``rms_norm_rel_error(D) |y|`` plus the half-ulp of a 16-bit output."""
    y = np.abs(np.asarray(y_ref, np.float64))
    tol = rms_norm_rel_error(D) * y
    if out_bf16:
        tol = tol + bf16_half_ulp(y + tol)
    if out_f16:
        tol = tol + f16_half_ulp(y + tol)
    return tol


def rmsnorm_gate_up_rel(D: int) -> float:
    """Relative accumulation factor of the gate/up projection of a BF16-rounded
    normalised activation.

    The tensor cores take BF16 operands, so the FP32 normalised value
    ``y (1 + e)``, ``|e| <= rms_norm_rel_error(D)``, is rounded to BF16 (half
    an ulp, at most ``2**-8`` relative) before the contraction: each operand
    is within ``d = 2**-8 + e (1 + 2**-8)`` of the exact one, relative.  The
    products' sum moves by at most ``d sum |xn w|``, and the FP32 accumulation
    of the perturbed products adds ``REL_ACC (1 + d) sum |xn w|``.
    """
    e = rms_norm_rel_error(D)
    d = 2.0 ** -8 + e * (1.0 + 2.0 ** -8)
    return REL_ACC * (1.0 + d) + d


def row_stats_tolerance(stats, alpha, beta):
    """Admissible errors of FP32 row sums, maxima and minima.

    Each entry ``v`` of the row is within ``t = gemm_tolerance(...)`` (no
    output rounding: the reductions see the FP32 values).  The maximum and
    the minimum move by at most ``max_n t``; the sum by ``sum_n t`` plus the
    FP32 summation of N terms in any order, ``gamma_N sum_n (|v| + t)``.
    """
    v = stats["values"]
    t = gemm_tolerance(v, stats["abs_sum"], alpha, beta, stats["c"])
    N = v.shape[1]
    gamma = N * U32 / (1.0 - N * U32)
    return {"sum": t.sum(axis=1) + gamma * (np.abs(v) + t).sum(axis=1),
            "max": t.max(axis=1), "min": t.max(axis=1)}


def fp32_sum_rel(n: int) -> float:
    """Relative error bound of an FP32 sum of n exact terms in any order,
    each addition rounding (or truncating) with error at most 2u:
    ``2 n u``."""
    return 2.0 * n * U32


def attention_tolerance(res, D: int, Nk: int, out_bf16=True):
    """Admissible |O_gpu - O_ref| for attention computed as a flash loop in FP32
    with BF16 probabilities.

    * Scores: each is an FP32 accumulation of D exact BF16 products, so it is
      within ``fp32_sum_rel(D) sum|q k|`` of the exact one.  The exponent
      argument is then formed in FP32 from the score: the product with
      scale * log2 e (itself rounded) and the subtraction of the running
      maximum add at most 8 units of roundoff relative to |scale * s|.  So
      the argument is within ``e = (fp32_sum_rel(D) + 8 u) * smax``.
    * Weights: exp and the running rescaling keep ratios between keys, so a
      score shift of at most e moves each normalised weight by a factor within
      ``exp(+-2e)``; the BF16 probabilities add 2^-8 (round to nearest with an
      8-bit significand, whatever the scale the probabilities are taken at),
      the exp evaluation 2^-20, the FP32 sum of the Nk probabilities
      ``fp32_sum_rel(Nk)``:
      ``eta = exp(2e)(1 + 2^-8)(1 + 2^-20)(1 + fp32_sum_rel(Nk)) - 1``.
    * Output: the FP32 products of weights and values over Nk keys
      (``fp32_sum_rel(Nk)``), the per-block rescaling (at most one rounding
      per 128-key block) and the final normalisation: the division, and the
      merge of the two partial sums over disjoint key sets (even and odd
      blocks) that the loop may keep -- two scalings by 2^(m_c - m) (an
      approximate exp2, within 2^-22 = 4 units), their sum and the scaled
      reciprocal, 12 units in all; all relative to
      ``abs_o = sum_j w_j |v_j|``.
    Plus the BF16 half-ulp of a BF16 output.
    """
    e = (fp32_sum_rel(D) + 8.0 * U32) * res["smax"][:, None]
    eta = np.exp(2.0 * e) * (1 + 2.0 ** -8) * (1 + 2.0 ** -20) * (1 + fp32_sum_rel(Nk)) - 1.0
    acc = fp32_sum_rel(Nk) + (Nk / 128.0 + 12.0) * U32
    tol = (eta + acc * (1.0 + eta)) * res["abs_o"]
    if out_bf16:
        tol = tol + bf16_half_ulp(np.abs(res["o"]) + tol)
    return tol
