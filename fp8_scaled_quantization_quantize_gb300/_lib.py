"""ctypes declarations of libfp8q.so's C ABI (include/fp8q.h)."""
from __future__ import annotations

import ctypes
import os

HERE = os.path.dirname(os.path.abspath(__file__))
LIB_PATH = os.path.join(HERE, "libfp8q.so")

# fp8q_status
OK, ERR_ARG, ERR_SHAPE, ERR_ALIGN, ERR_DTYPE, ERR_UNSUPPORTED, ERR_CUDA, ERR_TIMEOUT, WARN_NONFINITE = range(9)
# fp8q_format
E4M3, E5M2 = 0, 1
# fp8q_recipe_kind
PERTENSOR_CURRENT, PERTENSOR_DELAYED, BLOCK_1x128, BLOCK_128x128, MXFP8_1x32, PERCHANNEL_CURRENT, BLOCK_GENERIC = range(7)

EXPORTS = ("fp8q_version", "fp8q_status_str", "fp8q_scale_bytes", "fp8q_quantize", "fp8q_delayed_create",
           "fp8q_delayed_update", "fp8q_delayed_get", "fp8q_delayed_set", "fp8q_delayed_history_len",
           "fp8q_delayed_destroy", "fp8q_scaled_gemm", "fp8q_device_errors", "fp8q_cast_f32_bits", "fp8q_selftest_division",
           "fp8q_gemm_set_variant", "fp8q_scaled_gemm_mxq", "fp8q_quantize_multi", "fp8q_quantize_rows",
           "fp8q_set_wait_limit", "fp8q_stall_next", "fp8q_scaled_gemm_q")
MULTI_MAX = 16  # FP8Q_MULTI_MAX


class Recipe(ctypes.Structure):
    _fields_ = [("kind", ctypes.c_int), ("fmt", ctypes.c_int), ("want_rowwise", ctypes.c_int),
                ("want_colwise", ctypes.c_int), ("block_rows", ctypes.c_int), ("block_cols", ctypes.c_int)]


class Tensor(ctypes.Structure):
    _fields_ = [("data_row", ctypes.c_void_p), ("data_col", ctypes.c_void_p), ("scale_row", ctypes.c_void_p),
                ("scale_col", ctypes.c_void_p), ("amax", ctypes.c_void_p), ("scale", ctypes.c_void_p),
                ("scale_inv", ctypes.c_void_p), ("counters", ctypes.c_void_p), ("rows", ctypes.c_int64),
                ("cols", ctypes.c_int64), ("fmt", ctypes.c_int), ("kind", ctypes.c_int),
                ("block_rows", ctypes.c_int), ("block_cols", ctypes.c_int)]


class QuantizeJob(ctypes.Structure):
    _fields_ = [("recipe", Recipe), ("x", ctypes.c_void_p), ("rows", ctypes.c_int64), ("cols", ctypes.c_int64),
                ("state", ctypes.c_void_p), ("out", ctypes.POINTER(Tensor))]


class Fp8qError(RuntimeError):
    def __init__(self, status: int, what: str):
        self.status = status
        super().__init__(f"{what}: {status_str(status)} ({status})")


_lib = None


def load(path: str = LIB_PATH):
    """Loads libfp8q.so; raises if it has not been built (there is no fallback)."""
    global _lib
    if _lib is not None:
        return _lib
    if not os.path.exists(path):
        raise ImportError(f"libfp8q.so not built at {path}: run "
                          "`python -m fp8_scaled_quantization_quantize_gb300.build` (needs nvcc)")
    L = ctypes.CDLL(path)
    P, i64, i32, u32, u64 = ctypes.c_void_p, ctypes.c_int64, ctypes.c_int, ctypes.c_uint32, ctypes.c_uint64
    L.fp8q_version.restype = i32
    L.fp8q_version.argtypes = []
    L.fp8q_status_str.restype = ctypes.c_char_p
    L.fp8q_status_str.argtypes = [i32]
    L.fp8q_scale_bytes.restype = i32
    L.fp8q_scale_bytes.argtypes = [ctypes.POINTER(Recipe), i64, i64, ctypes.POINTER(ctypes.c_size_t),
                                   ctypes.POINTER(ctypes.c_size_t)]
    L.fp8q_quantize.restype = i32
    L.fp8q_quantize.argtypes = [ctypes.POINTER(Recipe), P, i64, i64, P, ctypes.POINTER(Tensor), P]
    L.fp8q_quantize_rows.restype = i32
    L.fp8q_quantize_rows.argtypes = [ctypes.POINTER(Recipe), P, i64, i64, i64, i64, ctypes.POINTER(Tensor), P]
    L.fp8q_quantize_multi.restype = i32
    L.fp8q_quantize_multi.argtypes = [ctypes.POINTER(QuantizeJob), i32, P]
    L.fp8q_delayed_create.restype = i32
    L.fp8q_delayed_create.argtypes = [i32, i32, i32, ctypes.POINTER(P)]
    L.fp8q_delayed_update.restype = i32
    L.fp8q_delayed_update.argtypes = [P, P, P, P]
    L.fp8q_delayed_get.restype = i32
    L.fp8q_delayed_get.argtypes = [P, P, ctypes.POINTER(i32), ctypes.POINTER(ctypes.c_float),
                                   ctypes.POINTER(ctypes.c_float)]
    L.fp8q_delayed_set.restype = i32
    L.fp8q_delayed_set.argtypes = [P, P, i32, ctypes.c_float, ctypes.c_float]
    L.fp8q_delayed_history_len.restype = i32
    L.fp8q_delayed_history_len.argtypes = [P]
    L.fp8q_delayed_destroy.restype = None
    L.fp8q_delayed_destroy.argtypes = [P]
    L.fp8q_scaled_gemm.restype = i32
    L.fp8q_scaled_gemm.argtypes = [ctypes.POINTER(Tensor), i32, ctypes.POINTER(Tensor), i32, P, i32, i64, i64,
                                   i64, P]
    L.fp8q_device_errors.restype = i32
    L.fp8q_device_errors.argtypes = [ctypes.POINTER(ctypes.c_uint), P]
    L.fp8q_scaled_gemm_mxq.restype = i32
    L.fp8q_scaled_gemm_mxq.argtypes = [ctypes.POINTER(Tensor), i32, ctypes.POINTER(Tensor), i32, P, i32,
                                       ctypes.POINTER(Tensor), i64, i64, i64, P]
    L.fp8q_scaled_gemm_q.restype = i32
    L.fp8q_scaled_gemm_q.argtypes = [ctypes.POINTER(Tensor), i32, ctypes.POINTER(Tensor), i32, P, i32, i32,
                                     ctypes.POINTER(Tensor), i64, i64, i64, P]
    L.fp8q_gemm_set_variant.restype = i32
    L.fp8q_gemm_set_variant.argtypes = [i32]
    L.fp8q_selftest_division.restype = i32
    L.fp8q_selftest_division.argtypes = [P, i64, i32, P, P]
    L.fp8q_set_wait_limit.restype = i32
    L.fp8q_set_wait_limit.argtypes = [u64]
    L.fp8q_stall_next.restype = i32
    L.fp8q_stall_next.argtypes = [i32]
    L.fp8q_cast_f32_bits.restype = i32
    L.fp8q_cast_f32_bits.argtypes = [u32, u64, i32, P, P]
    _lib = L
    return L


def status_str(status: int) -> str:
    try:
        return load().fp8q_status_str(status).decode()
    except ImportError:
        return "unknown"


def check(status: int, what: str):
    if status != OK:
        raise Fp8qError(status, what)
