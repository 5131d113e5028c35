"""Thin PyTorch binding of libfp8q: argument marshalling only.

torch provides device memory and the current CUDA stream; every step of the
quantize / GEMM path runs in the library's kernels (include/fp8q.h).  There
is no fallback: without the built library every call raises.
"""
from __future__ import annotations

import ctypes
from dataclasses import dataclass

import torch

from . import _lib as L
from ._lib import (BLOCK_1x128, BLOCK_128x128, BLOCK_GENERIC, E4M3, E5M2, MXFP8_1x32, PERCHANNEL_CURRENT,  # noqa: F401
                   PERTENSOR_CURRENT, PERTENSOR_DELAYED, Fp8qError)


def _stream(stream) -> int:
    if stream is None:
        return torch.cuda.current_stream().cuda_stream
    if isinstance(stream, torch.cuda.Stream):
        return stream.cuda_stream
    return int(stream)


def _ptr(t):
    return None if t is None else ctypes.c_void_p(t.data_ptr())


# The library takes plain pointers and cannot see a buffer's size or where it
# lives: a tensor of another shape than the buffers it pairs with, or one in
# host memory, would reach the kernels as an out-of-range or host address.
# These checks stop that here.

def _check_device(t: torch.Tensor, ref: torch.Tensor, name: str):
    if not t.is_cuda or t.device != ref.device:
        raise ValueError(f"{name} must be on the CUDA device of the buffers it pairs with ({ref.device})")
    _check_current(t.device, name)


def _check_current(dev: torch.device, name: str):
    """The library launches on the current CUDA device: buffers of another
    device would reach its kernels as foreign addresses."""
    cur = torch.cuda.current_device()
    if dev.index is not None and dev.index != cur:
        raise ValueError(f"{name} is on {dev} but cuda:{cur} is the current device; "
                         f"call inside `with torch.cuda.device({dev.index}):`")


def _check_input(x: torch.Tensor, qt: QTensor, name: str = "x", any_rows: bool = False):
    """x is contiguous 2-D bf16 of qt's shape (any row count with any_rows:
    a block of qt's rows) on qt's CUDA device."""
    if x.dtype != torch.bfloat16 or x.dim() != 2 or not x.is_contiguous():
        raise ValueError(f"{name} must be a contiguous 2-D bf16 tensor")
    want = (x.shape[0] if any_rows else qt.rows, qt.cols)
    if tuple(x.shape) != want:
        raise ValueError(f"{name} has shape {tuple(x.shape)}; the output buffers hold {(qt.rows, qt.cols)}")
    _check_device(x, qt.counters, name)


def scale_bytes(kind: int, rows: int, cols: int, rowwise: bool, colwise: bool, block=(0, 0)):
    """Bytes of the scale buffers (fp8q_scale_bytes); block = (rows, cols) of a
    BLOCK_GENERIC recipe's blocks."""
    rb, cb = ctypes.c_size_t(0), ctypes.c_size_t(0)
    rc = L.Recipe(kind, E4M3, int(rowwise), int(colwise), *block)
    L.check(L.load().fp8q_scale_bytes(ctypes.byref(rc), rows, cols, ctypes.byref(rb), ctypes.byref(cb)),
            "fp8q_scale_bytes")
    return rb.value, cb.value


@dataclass
class QTensor:
    """Device buffers of one quantized tensor (see fp8q_tensor)."""
    kind: int
    fmt: int
    rows: int
    cols: int
    data_row: torch.Tensor | None
    data_col: torch.Tensor | None
    scale_row: torch.Tensor | None   # raw bytes (uint8)
    scale_col: torch.Tensor | None
    amax: torch.Tensor               # fp32[1]
    scale: torch.Tensor              # fp32[1]
    scale_inv: torch.Tensor          # fp32[1]
    counters: torch.Tensor           # int64[3]: sat_row, sat_col, nonfinite
    block: tuple = (0, 0)            # BLOCK_GENERIC: (block rows, block cols)

    def c_struct(self) -> L.Tensor:
        return L.Tensor(_ptr(self.data_row), _ptr(self.data_col), _ptr(self.scale_row), _ptr(self.scale_col),
                        _ptr(self.amax), _ptr(self.scale), _ptr(self.scale_inv), _ptr(self.counters),
                        self.rows, self.cols, self.fmt, self.kind, *self.block)

    def recipe(self) -> L.Recipe:
        return L.Recipe(self.kind, self.fmt, int(self.rowwise), int(self.colwise), *self.block)

    @property
    def rowwise(self) -> bool:
        return self.data_row is not None

    @property
    def colwise(self) -> bool:
        return self.data_col is not None


def row_block(qt: QTensor, r0: int, r1: int) -> QTensor:
    """Rows [r0, r1) of a quantized tensor's row-wise copy as a QTensor of its
    own (views of qt's buffers, nothing copied): a GEMM operand for a block of
    output columns, e.g. one shard of a weight.  r0 and r1 are multiples of
    128 (r1 may be qt.rows).  Per-tensor, 128x128, MXFP8 and per-channel
    copies: their scales of a 128-row block are contiguous; a 1x128 copy's
    are K-block-major, so it raises."""
    if qt.data_row is None:
        raise ValueError("row_block needs the row-wise copy")
    if not (0 <= r0 < r1 <= qt.rows) or r0 % 128 or (r1 % 128 and r1 != qt.rows):
        raise ValueError("row block bounds must be multiples of 128 inside the tensor")
    C = qt.cols
    sr = None
    if qt.kind == BLOCK_128x128:
        per = -(-C // 128) * 4                       # bytes of one 128-row block of scales
        sr = qt.scale_row[(r0 // 128) * per:(-(-r1 // 128)) * per]
    elif qt.kind == MXFP8_1x32:
        per = -(-C // 128) * 512
        sr = qt.scale_row[(r0 // 128) * per:(-(-r1 // 128)) * per]
    elif qt.kind == PERCHANNEL_CURRENT:
        sr = qt.scale_row[r0 * 4:(-(-r1 // 128)) * 128 * 4]
    elif qt.kind not in (PERTENSOR_CURRENT, PERTENSOR_DELAYED):
        raise ValueError("row_block: the 1x128 scale layout is not row-contiguous")
    if qt.kind == BLOCK_GENERIC:
        raise ValueError("row_block: generic block scales are not taken apart by rows")
    return QTensor(qt.kind, qt.fmt, r1 - r0, C, qt.data_row[r0:r1], None, sr, None,
                   qt.amax, qt.scale, qt.scale_inv, qt.counters)


def alloc(kind: int, fmt: int, rows: int, cols: int, rowwise: bool = True, colwise: bool = False,
          device="cuda", block=(0, 0)) -> QTensor:
    """Device buffers for one quantize call; block = (rows, cols) of the
    blocks of a BLOCK_GENERIC recipe (1 x b or b x b, b in 32, 64, 128, 256)."""
    block = tuple(int(v) for v in block) if kind == BLOCK_GENERIC else (0, 0)
    rb, cb = scale_bytes(kind, rows, cols, rowwise, colwise, block)
    u8 = dict(dtype=torch.uint8, device=device)
    f32 = dict(dtype=torch.float32, device=device)
    return QTensor(kind, fmt, rows, cols,
                   torch.empty((rows, cols), **u8) if rowwise else None,
                   torch.empty((cols, rows), **u8) if colwise else None,
                   torch.empty(max(rb, 16), **u8) if rowwise and rb else None,
                   torch.empty(max(cb, 16), **u8) if colwise and cb else None,
                   torch.zeros(1, **f32), torch.ones(1, **f32), torch.ones(1, **f32),
                   torch.zeros(3, dtype=torch.int64, device=device), block)


class DelayedState:
    """Library-owned per-tensor delayed-scaling state (amax history)."""

    def __init__(self, history_len: int = 16, fmt: int = E4M3, margin: int = 0):
        h = ctypes.c_void_p(0)
        L.check(L.load().fp8q_delayed_create(history_len, fmt, margin, ctypes.byref(h)), "fp8q_delayed_create")
        self.handle = h
        self.history_len, self.fmt, self.margin = history_len, fmt, margin

    def update(self, amax: torch.Tensor, nonfinite: torch.Tensor | None = None, stream=None):
        if amax.dtype != torch.float32 or amax.numel() < 1 or not amax.is_cuda:
            raise ValueError("amax must be a CUDA fp32 tensor")
        _check_current(amax.device, "amax")
        if nonfinite is not None and (nonfinite.dtype != torch.int64 or nonfinite.numel() < 1
                                      or nonfinite.device != amax.device):
            raise ValueError("nonfinite must be an int64 tensor on amax's device")
        L.check(L.load().fp8q_delayed_update(self.handle, _ptr(amax), _ptr(nonfinite), _stream(stream)),
                "fp8q_delayed_update")

    def get(self):
        """(history fp32 list, head, scale, scale_inv); synchronises."""
        hist = (ctypes.c_float * self.history_len)()
        head, s, si = ctypes.c_int(0), ctypes.c_float(0), ctypes.c_float(0)
        L.check(L.load().fp8q_delayed_get(self.handle, hist, ctypes.byref(head), ctypes.byref(s), ctypes.byref(si)),
                "fp8q_delayed_get")
        return list(hist), head.value, s.value, si.value

    def set(self, hist, head: int, scale: float, scale_inv: float):
        arr = (ctypes.c_float * self.history_len)(*hist)
        L.check(L.load().fp8q_delayed_set(self.handle, arr, head, scale, scale_inv), "fp8q_delayed_set")

    def close(self):
        if getattr(self, "handle", None):
            L.load().fp8q_delayed_destroy(self.handle)
            self.handle = None

    def __del__(self):
        try:
            self.close()
        except Exception:
            pass


def quantize_into(x: torch.Tensor, qt: QTensor, state: DelayedState | None = None, stream=None) -> QTensor:
    """Quantizes bf16 x [rows, cols] into preallocated qt (same kind / fmt / copies)."""
    _check_input(x, qt)
    rc = qt.recipe()
    ct = qt.c_struct()
    L.check(L.load().fp8q_quantize(ctypes.byref(rc), _ptr(x), x.shape[0], x.shape[1],
                                   state.handle if state is not None else None, ctypes.byref(ct), _stream(stream)),
            "fp8q_quantize")
    return qt


def quantize_rows_into(x_block: torch.Tensor, qt: QTensor, row0: int, stream=None) -> QTensor:
    """Quantizes rows row0 .. row0 + len(x_block) - 1 of the tensor whose
    buffers qt holds (fp8q_quantize_rows); qt.counters are added to."""
    _check_input(x_block, qt, "x_block", any_rows=True)
    rc = qt.recipe()
    ct = qt.c_struct()
    L.check(L.load().fp8q_quantize_rows(ctypes.byref(rc), _ptr(x_block), row0, x_block.shape[0], qt.rows,
                                        x_block.shape[1], ctypes.byref(ct), _stream(stream)), "fp8q_quantize_rows")
    return qt


def quantize_multi(jobs, stream=None):
    """Quantizes several tensors in one call (fp8q_quantize_multi): jobs is a
    sequence of (x, qt) or (x, qt, state) with qt preallocated as for
    quantize_into; the outputs equal those of quantize_into on each."""
    jobs = list(jobs)
    arr = (L.QuantizeJob * max(len(jobs), 1))()
    keep = []
    for i, job in enumerate(jobs):
        x, qt = job[0], job[1]
        state = job[2] if len(job) > 2 else None
        _check_input(x, qt, f"x of job {i}")
        ct = qt.c_struct()
        keep.append(ct)
        arr[i].recipe = qt.recipe()
        arr[i].x = x.data_ptr()
        arr[i].rows, arr[i].cols = x.shape[0], x.shape[1]
        arr[i].state = state.handle if state is not None else None
        arr[i].out = ctypes.pointer(ct)
    L.check(L.load().fp8q_quantize_multi(arr, len(jobs), _stream(stream)), "fp8q_quantize_multi")
    return [job[1] for job in jobs]


def quantize(x: torch.Tensor, kind: int, fmt: int = E4M3, rowwise: bool = True, colwise: bool = False,
             state: DelayedState | None = None, stream=None, block=(0, 0)) -> QTensor:
    qt = alloc(kind, fmt, x.shape[0], x.shape[1], rowwise, colwise, device=x.device, block=block)
    return quantize_into(x, qt, state, stream)


def _check_operands(A: QTensor, a_use_col: bool, B: QTensor, b_use_col: bool) -> torch.Tensor:
    """The chosen copies' data on one CUDA device (a missing copy is left to
    the library, which rejects it); returns a tensor on that device."""
    ref = A.counters
    for name, qt, use_col in (("A", A, a_use_col), ("B", B, b_use_col)):
        data = qt.data_col if use_col else qt.data_row
        _check_device(data if data is not None else qt.counters, ref, f"{name}'s buffers")
    return ref


def scaled_gemm(A: QTensor, a_use_col: bool, B: QTensor, b_use_col: bool, out_dtype=torch.bfloat16,
                out: torch.Tensor | None = None, stream=None) -> torch.Tensor:
    """D = A_q . B_q^T (fp32 accumulate) with the recipes' scales applied."""
    M = A.cols if a_use_col else A.rows
    K = A.rows if a_use_col else A.cols
    N = B.cols if b_use_col else B.rows
    ref = _check_operands(A, a_use_col, B, b_use_col)
    if out is None:
        out = torch.empty((M, N), dtype=out_dtype, device=ref.device)
    if out.dtype not in (torch.bfloat16, torch.float32) or tuple(out.shape) != (M, N) or not out.is_contiguous():
        raise ValueError(f"out must be a contiguous bf16 or fp32 tensor of shape {(M, N)}")
    _check_device(out, ref, "out")
    od = {torch.bfloat16: 0, torch.float32: 1}[out.dtype]
    ca, cb = A.c_struct(), B.c_struct()
    L.check(L.load().fp8q_scaled_gemm(ctypes.byref(ca), int(a_use_col), ctypes.byref(cb), int(b_use_col), _ptr(out),
                                      od, M, N, K, _stream(stream)), "fp8q_scaled_gemm")
    return out


def scaled_gemm_q(A: QTensor, a_use_col: bool, B: QTensor, b_use_col: bool, kind: int = MXFP8_1x32,
                  fmt: int = E4M3, want_d: bool = True, out: QTensor | None = None,
                  d_out: torch.Tensor | None = None, stream=None, colwise: bool = False):
    """The GEMM with its bf16 output also quantized in the epilogue
    (fp8q_scaled_gemm_q), kind MXFP8_1x32 or BLOCK_1x128: the row-wise copy,
    and with colwise (or an `out` holding a column copy) the column-wise copy
    too (blocks along M; M % 16 == 0).  Returns (D bf16 or None, QTensor)."""
    M = A.cols if a_use_col else A.rows
    K = A.rows if a_use_col else A.cols
    N = B.cols if b_use_col else B.rows
    dev = _check_operands(A, a_use_col, B, b_use_col).device
    if kind not in (MXFP8_1x32, BLOCK_1x128):
        raise ValueError("kind must be MXFP8_1x32 or BLOCK_1x128")
    if out is None:
        out = alloc(kind, fmt, M, N, True, colwise, dev)
    if (out.rows, out.cols) != (M, N) or out.data_row is None or out.scale_row is None or out.kind != kind:
        raise ValueError(f"out must hold a row-wise copy of kind {kind} and shape {(M, N)}")
    rb, cb = scale_bytes(kind, M, N, True, out.data_col is not None)
    if out.scale_row.numel() < rb:
        raise ValueError("out.scale_row is smaller than the recipe's scale bytes")
    if out.data_col is not None:
        if tuple(out.data_col.shape) != (N, M) or out.scale_col is None or out.scale_col.numel() < cb:
            raise ValueError(f"out's column copy must be [{N}, {M}] with its scale bytes")
        if M % 16:
            raise ValueError("a column-wise copy needs M % 16 == 0")
        _check_device(out.data_col, out.counters, "out's buffers")
        _check_device(out.scale_col, out.counters, "out's buffers")
    _check_device(out.data_row, out.counters, "out's buffers")
    _check_device(out.counters, A.counters, "out's buffers")
    if want_d and d_out is None:
        d_out = torch.empty((M, N), dtype=torch.bfloat16, device=dev)
    if want_d:
        if d_out.dtype != torch.bfloat16 or tuple(d_out.shape) != (M, N) or not d_out.is_contiguous():
            raise ValueError(f"d_out must be a contiguous bf16 tensor of shape {(M, N)}")
        _check_device(d_out, A.counters, "d_out")
    ca, cb, cq = A.c_struct(), B.c_struct(), out.c_struct()
    L.check(L.load().fp8q_scaled_gemm_q(ctypes.byref(ca), int(a_use_col), ctypes.byref(cb), int(b_use_col),
                                        _ptr(d_out) if want_d else None, kind, fmt, ctypes.byref(cq), M, N, K,
                                        _stream(stream)), "fp8q_scaled_gemm_q")
    return (d_out if want_d else None), out


def scaled_gemm_mxq(A: QTensor, a_use_col: bool, B: QTensor, b_use_col: bool, fmt: int = E4M3,
                    want_d: bool = True, out: QTensor | None = None, d_out: torch.Tensor | None = None,
                    stream=None, colwise: bool = False):
    """The GEMM with its bf16 output also quantized MXFP8 1x32 in the epilogue
    (fp8q_scaled_gemm_mxq), row-wise and optionally column-wise: returns
    (D bf16 or None, QTensor)."""
    return scaled_gemm_q(A, a_use_col, B, b_use_col, MXFP8_1x32, fmt, want_d, out, d_out, stream, colwise)


def gemm_set_variant(variant: int):
    """0 automatic, 1 one SM per tile, 2 SM pairs (see fp8q_gemm_set_variant)."""
    L.check(L.load().fp8q_gemm_set_variant(int(variant)), "fp8q_gemm_set_variant")


def cast_f32_bits(start: int, count: int, fmt: int, out: torch.Tensor, stream=None) -> torch.Tensor:
    if out.dtype != torch.uint8 or not out.is_cuda or out.numel() < count or not out.is_contiguous():
        raise ValueError("out must be a contiguous CUDA uint8 tensor of at least count elements")
    _check_current(out.device, "out")
    L.check(L.load().fp8q_cast_f32_bits(start, count, fmt, _ptr(out), _stream(stream)), "fp8q_cast_f32_bits")
    return out


def selftest_division(d: torch.Tensor, fmt: int, stream=None):
    """(FP8 code mismatches, fp32 mismatches) of the blockwise division shortcut
    against IEEE division over every finite bf16 x and every divisor in d."""
    if d.dtype != torch.float32 or not d.is_cuda or not d.is_contiguous():
        raise ValueError("d must be a contiguous CUDA fp32 tensor")
    _check_current(d.device, "d")
    out = torch.zeros(2, dtype=torch.int64, device=d.device)
    L.check(L.load().fp8q_selftest_division(_ptr(d), d.numel(), fmt, _ptr(out), _stream(stream)),
            "fp8q_selftest_division")
    torch.cuda.synchronize()
    return int(out[0].item()), int(out[1].item())


def device_errors(stream=None) -> int:
    """Reads and clears the device error words (fp8q_device_errors): bit 0 a
    GEMM wait timed out, bit 1 a quantize wait timed out; 0 when none did."""
    v = ctypes.c_uint(0)
    st = L.load().fp8q_device_errors(ctypes.byref(v), _stream(stream))
    if st not in (L.OK, L.ERR_TIMEOUT):
        L.check(st, "fp8q_device_errors")
    return v.value


def set_wait_limit(ns: int):
    """Limit of every bounded device wait for later launches, in ns (0: the
    default, one second); see fp8q_set_wait_limit."""
    L.check(L.load().fp8q_set_wait_limit(int(ns)), "fp8q_set_wait_limit")


def stall_next(n: int):
    """The next n quantize-tile / GEMM launches run with no loads, so their
    waits run out (a test of the failure path; fp8q_stall_next)."""
    L.check(L.load().fp8q_stall_next(int(n)), "fp8q_stall_next")
