"""ctypes binding of the C ABI in ``include/gemm_bf16.h``.

Argument marshalling only: every step of the computation runs in the CUDA
library.  Loading fails loudly when the library has not been built; there is
no fallback.
"""
from __future__ import annotations

import ctypes
import os
import threading

from . import build as _build

GEMM_OK = 0
GEMM_ERR_INVALID_ARG = 1
GEMM_ERR_ALIGNMENT = 2
GEMM_ERR_UNSUPPORTED = 3
GEMM_ERR_CUDA = 4
GEMM_ERR_TIMEOUT = 5

GEMM_OUT_F32 = 0
GEMM_OUT_BF16 = 1
GEMM_OUT_F16 = 2

GEMM_IN_BF16 = 0
GEMM_IN_F16 = 1

KERNEL_NAMES = {0: "none", 1: "tiled", 2: "skinny_splitk", 3: "scale", 4: "gate_up",
                5: "pair", 6: "pair_gate_up", 7: "small_m", 8: "skinny_gate_up"}

# Every symbol the header declares.
EXPORTED = (
    "gemm_bf16",
    "gemm_gate_up_silu",
    "gemm_status_string",
    "gemm_get_device_status",
    "gemm_prepare",
    "gemm_bf16_plan",
    "gemm_gate_up_plan",
    "gemm_selftest_wait_timeout",
    "gemm_selftest_pipeline_timeout",
    "gemm_bf16_skinny_noalloc",
    "gemm_batched",
    "gemm_batched_plan",
    "gemm_row_stats",
    "gemm_row_stats_plan",
    "gemm_rms_norm",
    "gemm_rmsnorm_gate_up_silu",
    "gemm_attention",
    "gemm_layout_smem_descriptor",
    "gemm_layout_instr_descriptor",
    "gemm_layout_swizzle128_offset",
    "gemm_layout_tmem_address",
)


class GemmPlan(ctypes.Structure):
    _fields_ = [
        ("kernel", ctypes.c_int),
        ("tile_m", ctypes.c_int),
        ("tile_n", ctypes.c_int),
        ("tile_k", ctypes.c_int),
        ("stages", ctypes.c_int),
        ("split_k", ctypes.c_int),
        ("tiles", ctypes.c_int64),
        ("grid", ctypes.c_int),
        ("smem_bytes", ctypes.c_int),
        ("launches", ctypes.c_int),
        ("stage_tx_bytes", ctypes.c_int64),
    ]

    def as_dict(self) -> dict:
        d = {name: getattr(self, name) for name, _ in self._fields_}
        d["kernel_name"] = KERNEL_NAMES.get(self.kernel, "?")
        return d


class GemmError(RuntimeError):
    def __init__(self, status: int, what: str = ""):
        self.status = status
        msg = status_string(status) if _lib is not None else str(status)
        super().__init__(f"{what}: {msg} (status {status})" if what else msg)


_lock = threading.Lock()
_lib = None

_i64 = ctypes.c_int64
_vp = ctypes.c_void_p
_f32 = ctypes.c_float
_int = ctypes.c_int


def library_path() -> str:
    return _build.LIB_PATH


def lib() -> ctypes.CDLL:
    """The loaded CUDA library; raises if it has not been built."""
    global _lib
    with _lock:
        if _lib is None:
            path = _build.LIB_PATH
            if not os.path.exists(path):
                raise RuntimeError(
                    f"CUDA library {path} is missing: build it with "
                    "`python -m dense_bf16_gemm_gb300.build` (there is no CPU fallback)")
            l = ctypes.CDLL(path)
            l.gemm_bf16.restype = _int
            l.gemm_bf16.argtypes = [_i64, _i64, _i64, _f32, _vp, _i64, _vp, _i64, _f32,
                                    _vp, _i64, _int, _vp]
            l.gemm_gate_up_silu.restype = _int
            l.gemm_gate_up_silu.argtypes = [_i64, _i64, _i64, _vp, _i64, _vp, _vp, _i64,
                                            _vp, _i64, _vp]
            l.gemm_status_string.restype = ctypes.c_char_p
            l.gemm_status_string.argtypes = [_int]
            l.gemm_get_device_status.restype = _int
            l.gemm_get_device_status.argtypes = [_vp, ctypes.POINTER(_int)]
            l.gemm_prepare.restype = _int
            l.gemm_prepare.argtypes = [_i64, _vp]
            l.gemm_bf16_plan.restype = _int
            l.gemm_bf16_plan.argtypes = [_i64, _i64, _i64, _int, _int, ctypes.POINTER(GemmPlan)]
            l.gemm_batched.restype = _int
            l.gemm_batched.argtypes = [_i64, _i64, _i64, _i64, _f32, _vp, _i64, _i64, _vp, _i64,
                                       _i64, _f32, _vp, _i64, _i64, _int, _int, _vp]
            l.gemm_batched_plan.restype = _int
            l.gemm_batched_plan.argtypes = [_i64, _i64, _i64, _i64, _int, _int, _int,
                                            ctypes.POINTER(GemmPlan)]
            l.gemm_bf16_skinny_noalloc.restype = _int
            l.gemm_bf16_skinny_noalloc.argtypes = [_i64, _i64, _i64, _f32, _vp, _i64, _vp, _i64,
                                                   _f32, _vp, _i64, _int, _vp]
            l.gemm_selftest_wait_timeout.restype = _int
            l.gemm_selftest_wait_timeout.argtypes = [_i64, _vp]
            l.gemm_selftest_pipeline_timeout.restype = _int
            l.gemm_selftest_pipeline_timeout.argtypes = [_i64, _i64, _i64, _vp, _i64, _vp, _i64,
                                                         _vp, _i64, _int, _vp]
            l.gemm_gate_up_plan.restype = _int
            l.gemm_gate_up_plan.argtypes = [_i64, _i64, _i64, _int, ctypes.POINTER(GemmPlan)]
            l.gemm_row_stats.restype = _int
            l.gemm_row_stats.argtypes = [_i64, _i64, _i64, _i64, _f32, _vp, _i64, _i64, _vp,
                                         _i64, _i64, _f32, _vp, _i64, _i64, _int, _int,
                                         _vp, _vp, _vp, _vp]
            l.gemm_row_stats_plan.restype = _int
            l.gemm_row_stats_plan.argtypes = [_i64, _i64, _i64, _i64, _int, _int, _int,
                                              ctypes.POINTER(GemmPlan)]
            l.gemm_rms_norm.restype = _int
            l.gemm_rms_norm.argtypes = [_i64, _i64, _vp, _i64, _int, _vp, _f32, _vp, _i64,
                                        _int, _vp]
            l.gemm_rmsnorm_gate_up_silu.restype = _int
            l.gemm_rmsnorm_gate_up_silu.argtypes = [_i64, _i64, _i64, _vp, _i64, _vp, _f32,
                                                    _vp, _vp, _i64, _vp, _i64, _vp, _i64, _vp]
            l.gemm_layout_smem_descriptor.restype = ctypes.c_uint64
            l.gemm_layout_smem_descriptor.argtypes = [ctypes.c_uint32, ctypes.c_uint32]
            l.gemm_layout_instr_descriptor.restype = ctypes.c_uint32
            l.gemm_layout_instr_descriptor.argtypes = [_int, _int, _int]
            l.gemm_layout_swizzle128_offset.restype = ctypes.c_uint32
            l.gemm_layout_swizzle128_offset.argtypes = [_int, _int]
            l.gemm_layout_tmem_address.restype = ctypes.c_uint32
            l.gemm_layout_tmem_address.argtypes = [ctypes.c_uint32, _int, _int]
            l.gemm_attention.restype = _int
            l.gemm_attention.argtypes = [_i64, _i64, _i64, _i64, _f32, _vp, _i64, _i64, _vp, _i64,
                                         _i64, _vp, _i64, _i64, _vp, _i64, _i64, _int, _vp]
            _lib = l
    return _lib


def status_string(status: int) -> str:
    return lib().gemm_status_string(int(status)).decode()


def gemm_bf16(M, N, K, alpha, A, lda, B, ldb, beta, C, ldc, out_dtype, stream) -> int:
    """Raw C call; pointers and the stream are integers (0 = NULL)."""
    return lib().gemm_bf16(M, N, K, alpha, A or None, lda, B or None, ldb, beta, C or None,
                           ldc, out_dtype, stream or None)


def gemm_bf16_skinny_noalloc(M, N, K, alpha, A, lda, B, ldb, beta, C, ldc, out_dtype,
                             stream) -> int:
    """gemm_bf16 for M <= 16 using the library's fixed scratch array instead of
    an allocated workspace (for callers that may not allocate)."""
    return lib().gemm_bf16_skinny_noalloc(M, N, K, alpha, A or None, lda, B or None, ldb, beta,
                                          C or None, ldc, out_dtype, stream or None)


def gemm_batched(batch, M, N, K, alpha, A, lda, stride_a, B, ldb, stride_b, beta, C, ldc,
                 stride_c, in_dtype, out_dtype, stream) -> int:
    return lib().gemm_batched(batch, M, N, K, alpha, A or None, lda, stride_a, B or None, ldb,
                              stride_b, beta, C or None, ldc, stride_c, in_dtype, out_dtype,
                              stream or None)


def gemm_batched_plan(batch, M, N, K, in_dtype=GEMM_IN_BF16, out_dtype=GEMM_OUT_BF16, num_sms=0):
    plan = GemmPlan()
    st = lib().gemm_batched_plan(batch, M, N, K, in_dtype, out_dtype, num_sms, ctypes.byref(plan))
    return st, plan


def gemm_gate_up_silu(M, N, K, X, ldx, Wg, Wu, ldw, Y, ldy, stream) -> int:
    return lib().gemm_gate_up_silu(M, N, K, X or None, ldx, Wg or None, Wu or None, ldw,
                                   Y or None, ldy, stream or None)


def gemm_get_device_status(stream=0):
    site = _int(0)
    st = lib().gemm_get_device_status(stream or None, ctypes.byref(site))
    return st, site.value


def gemm_prepare(max_n: int, stream=0) -> int:
    return lib().gemm_prepare(max_n, stream or None)


def gemm_selftest_wait_timeout(limit_ns: int, stream=0) -> int:
    return lib().gemm_selftest_wait_timeout(limit_ns, stream or None)


def gemm_selftest_pipeline_timeout(M, N, K, A, lda, B, ldb, C, ldc, stall_after,
                                   stream=0) -> int:
    """A, B, C: device addresses (ints) of BF16 matrices."""
    return lib().gemm_selftest_pipeline_timeout(M, N, K, A or None, lda, B or None, ldb,
                                                C or None, ldc, stall_after, stream or None)


def gemm_bf16_plan(M, N, K, out_dtype=GEMM_OUT_BF16, num_sms=0):
    plan = GemmPlan()
    st = lib().gemm_bf16_plan(M, N, K, out_dtype, num_sms, ctypes.byref(plan))
    return st, plan


def gemm_gate_up_plan(M, N, K, num_sms=0):
    plan = GemmPlan()
    st = lib().gemm_gate_up_plan(M, N, K, num_sms, ctypes.byref(plan))
    return st, plan


def gemm_row_stats(batch, M, N, K, alpha, A, lda, stride_a, B, ldb, stride_b, beta, C, ldc,
                   stride_c, in_dtype, out_dtype, row_sum, row_max, row_min, stream) -> int:
    return lib().gemm_row_stats(batch, M, N, K, alpha, A or None, lda, stride_a, B or None, ldb,
                                stride_b, beta, C or None, ldc, stride_c, in_dtype, out_dtype,
                                row_sum or None, row_max or None, row_min or None,
                                stream or None)


def gemm_row_stats_plan(batch, M, N, K, in_dtype=GEMM_IN_BF16, out_dtype=GEMM_OUT_BF16,
                        num_sms=0):
    plan = GemmPlan()
    st = lib().gemm_row_stats_plan(batch, M, N, K, in_dtype, out_dtype, num_sms,
                                   ctypes.byref(plan))
    return st, plan


def gemm_rms_norm(rows, D, X, ldx, x_dtype, G, eps, Y, ldy, y_dtype, stream) -> int:
    return lib().gemm_rms_norm(rows, D, X or None, ldx, x_dtype, G or None, eps, Y or None,
                               ldy, y_dtype, stream or None)


def gemm_rmsnorm_gate_up_silu(M, N, K, X, ldx, G, eps, Wg, Wu, ldw, Xn, ldxn, Y, ldy,
                              stream) -> int:
    return lib().gemm_rmsnorm_gate_up_silu(M, N, K, X or None, ldx, G or None, eps, Wg or None,
                                           Wu or None, ldw, Xn or None, ldxn, Y or None, ldy,
                                           stream or None)


def gemm_attention(heads, Nq, Nk, D, scale, Q, ldq, sq, K, ldk, sk, V, ldv, sv, O, ldo, so,
                   out_dtype, stream) -> int:
    return lib().gemm_attention(heads, Nq, Nk, D, scale, Q or None, ldq, sq, K or None, ldk, sk,
                                V or None, ldv, sv, O or None, ldo, so, out_dtype, stream or None)
