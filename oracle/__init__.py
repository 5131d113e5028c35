"""fp8q oracle: ctypes wrapper over the plain C restatement in fp8q_oracle.c.

TEST INFRASTRUCTURE ONLY.  Only ``tests/``, ``__graft_entry__.smoke()`` and
the cpu_baseline / reference legs of ``bench.py`` may import this package.
The product library never calls it; the two share no code.

The recipes follow the four web pages on FP8 training:
  * "2025 FP8 quantized-training guide", sec. 1.1 (E4M3 / E5M2 layouts),
    sec. 2.1 (per-tensor delayed and current scaling), sec. 2.2 (blockwise
    1x128 / 128x128), sec. 2.3 (MXFP8 1x32 with E8M0 scales), sec. 3.1
    (fprop / dgrad / wgrad GEMMs on quantized inputs);
  * "mastering FP8 LLM training 1.5x speedup", scaling strategies 1-4;
  * bjdmk.com.cn/news/5220490, sec. 3.3 (DelayedScaling margin / interval).

Per-channel current scaling ("mastering FP8 LLM training 1.5x speedup",
Figure 1 and its discussion: one scaling factor per channel, i.e. per row or
column, between per-tensor and 2D blocks in granularity) is read as the
per-tensor current rule applied to each row of x (row-wise copy) and to each
column of x (column-wise copy), so that a copy's factor is constant along the
contraction dimension of the GEMM it feeds.  Its stored dequantization factor
is RN(1 / s), the per-tensor recipe's scale_inv, one per row of the copy.

The column-wise copy is the quantized transpose: for per-tensor and 128x128
tiles it is the byte transpose of the row-wise copy (same scales, transposed
for tiles); for 1x128 and 1x32 blocks it is a re-quantization of x^T with the
blocks running along the rows of x (the contraction dimension of wgrad).
"""
from __future__ import annotations

import ctypes
import os
import subprocess

import numpy as np

_HERE = os.path.dirname(os.path.abspath(__file__))
_SRC = os.path.join(_HERE, "fp8q_oracle.c")
_LIB = os.path.join(_HERE, "liboracle.so")

E4M3, E5M2 = 0, 1
FMAX = {E4M3: 448.0, E5M2: 57344.0}

# recipe kinds (the oracle's own numbering)
PERTENSOR_CURRENT, PERTENSOR_DELAYED, BLOCK_1x128, BLOCK_128x128, MXFP8_1x32, PERCHANNEL_CURRENT, BLOCK_GENERIC = range(7)
KIND_MULT, KIND_DIV, KIND_POW2 = 0, 1, 2


def build(force: bool = False) -> str:
    """Compiles the oracle with gcc (no FMA contraction) if it is stale."""
    if force or not os.path.exists(_LIB) or os.path.getmtime(_LIB) < os.path.getmtime(_SRC):
        tmp = _LIB + f".tmp{os.getpid()}"
        subprocess.check_call(["gcc", "-O2", "-std=c11", "-ffp-contract=off", "-fno-fast-math", "-fopenmp",
                               "-fPIC", "-shared", _SRC, "-o", tmp, "-lm"])
        os.replace(tmp, _LIB)
    return _LIB


_lib = None


def lib():
    global _lib
    if _lib is None:
        build()
        L = ctypes.CDLL(_LIB)
        P = ctypes.c_void_p
        i64, u64, i32, f32 = ctypes.c_int64, ctypes.c_uint64, ctypes.c_int, ctypes.c_float
        L.orc_fp8_decode.restype = ctypes.c_double
        L.orc_fp8_decode.argtypes = [ctypes.c_uint8, i32]
        L.orc_fp8_encode.restype = ctypes.c_uint8
        L.orc_fp8_encode.argtypes = [f32, i32]
        L.orc_fp8_encode_bits_range.argtypes = [ctypes.c_uint32, u64, i32, P]
        L.orc_fp8_encode_array.argtypes = [P, i64, i32, P]
        L.orc_bf16_to_f32.restype = f32
        L.orc_bf16_to_f32.argtypes = [ctypes.c_uint16]
        L.orc_pertensor_scale.restype = f32
        L.orc_pertensor_scale.argtypes = [f32, i32]
        L.orc_block_scale.restype = f32
        L.orc_block_scale.argtypes = [f32, i32]
        L.orc_mx_exponent.restype = i32
        L.orc_mx_exponent.argtypes = [f32, i32]
        L.orc_quant_blocks.argtypes = [P, i64, i64, i64, i64, i32, i32, P, P, P, P, P, P]
        L.orc_cast_scaled.argtypes = [P, i64, f32, i32, P, P, P, P]
        L.orc_amax_sat.argtypes = [P, i64, f32, i32, P, P, P]
        L.orc_delayed_sizeof.restype = i32
        L.orc_delayed_init.restype = i32
        L.orc_delayed_init.argtypes = [P, i32, i32, i32]
        L.orc_delayed_update.argtypes = [P, f32, u64]
        L.orc_pack_mx.argtypes = [P, i64, i64, P]
        L.orc_pack_block1x128.argtypes = [P, i64, i64, P]
        L.orc_gemm_points.argtypes = [P, i32, P, i64, i64, i64, P, i32, P, i64, i64, i64,
                                      i64, i64, i64, P, P, i64, P]
        L.orc_set_threads.restype = i32
        L.orc_set_threads.argtypes = [i32]
        L.orc_f64_to_bf16.restype = ctypes.c_uint16
        L.orc_f64_to_bf16.argtypes = [ctypes.c_double]
        _lib = L
    return _lib


def set_threads(n: int = 0) -> int:
    """Host threads the oracle's loops use (0: leave as is); returns the count
    in force.  Results do not depend on it (see the C file's header)."""
    return int(lib().orc_set_threads(int(n)))


def _p(a: np.ndarray):
    return a.ctypes.data_as(ctypes.c_void_p)


# ---------------------------------------------------------------- formats

def decode(codes, fmt: int) -> np.ndarray:
    """Exact value of each FP8 code (fp64)."""
    L = lib()
    codes = np.asarray(codes, dtype=np.uint8)
    table = np.array([L.orc_fp8_decode(c, fmt) for c in range(256)], dtype=np.float64)
    return table[codes]


def encode(values, fmt: int) -> np.ndarray:
    """Saturating RNE cast of fp32 values to FP8 codes."""
    v = np.ascontiguousarray(np.asarray(values, dtype=np.float32))
    out = np.empty(v.shape, dtype=np.uint8)
    lib().orc_fp8_encode_array(_p(v), v.size, fmt, _p(out))
    return out


def encode_bits_range(start: int, count: int, fmt: int) -> np.ndarray:
    out = np.empty(count, dtype=np.uint8)
    lib().orc_fp8_encode_bits_range(start, count, fmt, _p(out))
    return out


def bf16_to_f32(bits) -> np.ndarray:
    b = np.asarray(bits, dtype=np.uint16)
    return (b.astype(np.uint32) << 16).view(np.float32)


def f64_to_bf16(values) -> np.ndarray:
    """Round fp64 values to bf16 (RNE); returns the bf16 bits."""
    L = lib()
    v = np.asarray(values, dtype=np.float64)
    return np.array([L.orc_f64_to_bf16(float(x)) for x in v.ravel()], dtype=np.uint16).reshape(v.shape)


# ------------------------------------------------------------ scale rules

def pertensor_scale(amax: float, fmt: int) -> np.float32:
    return np.float32(lib().orc_pertensor_scale(amax, fmt))


def block_scale(amax: float, fmt: int) -> np.float32:
    return np.float32(lib().orc_block_scale(amax, fmt))


def mx_exponent(amax: float, fmt: int) -> int:
    return int(lib().orc_mx_exponent(amax, fmt))


# ------------------------------------------------------------- quantizers

def quant_blocks(x_bits: np.ndarray, br: int, bc: int, kind: int, fmt: int):
    """Block quantizer (see orc_quant_blocks).  Returns (q, scale, e8m0,
    amax, sat, nonfinite) with scale / e8m0 / amax shaped [nbr, nbc]."""
    x = np.ascontiguousarray(x_bits, dtype=np.uint16)
    R, C = x.shape
    nbr, nbc = -(-R // br), -(-C // bc)
    q = np.empty((R, C), dtype=np.uint8)
    sc = np.empty((nbr, nbc), dtype=np.float32)
    e8 = np.empty((nbr, nbc), dtype=np.uint8)
    am = np.empty((nbr, nbc), dtype=np.float32)
    sat = np.zeros(1, dtype=np.uint64)
    nf = np.zeros(1, dtype=np.uint64)
    lib().orc_quant_blocks(_p(x), R, C, br, bc, kind, fmt, _p(q), _p(sc), _p(e8), _p(am), _p(sat), _p(nf))
    return q, sc, e8, am, int(sat[0]), int(nf[0])


def cast_scaled(x_bits: np.ndarray, s: float, fmt: int):
    """q = encode(x * s) with a given multiplier; returns (q, amax, sat, nonfinite)."""
    x = np.ascontiguousarray(x_bits, dtype=np.uint16)
    q = np.empty(x.shape, dtype=np.uint8)
    am = np.zeros(1, dtype=np.float32)
    sat = np.zeros(1, dtype=np.uint64)
    nf = np.zeros(1, dtype=np.uint64)
    lib().orc_cast_scaled(_p(x), x.size, np.float32(s), fmt, _p(q), _p(am), _p(sat), _p(nf))
    return q, float(am[0]), int(sat[0]), int(nf[0])


def amax_sat(x_bits: np.ndarray, s: float, fmt: int):
    """(amax, sat, nonfinite) of a per-tensor cast with multiplier s, no codes."""
    x = np.ascontiguousarray(x_bits, dtype=np.uint16)
    am = np.zeros(1, dtype=np.float32)
    sat = np.zeros(1, dtype=np.uint64)
    nf = np.zeros(1, dtype=np.uint64)
    lib().orc_amax_sat(_p(x), x.size, np.float32(s), fmt, _p(am), _p(sat), _p(nf))
    return float(am[0]), int(sat[0]), int(nf[0])


class Delayed:
    """Per-tensor delayed-scaling state: amax ring of length H, head, scale."""

    def __init__(self, H: int = 16, fmt: int = E4M3, margin: int = 0):
        self._buf = np.zeros(lib().orc_delayed_sizeof(), dtype=np.uint8)
        if lib().orc_delayed_init(_p(self._buf), H, fmt, margin) != 0:
            raise ValueError("bad history length")
        self.H, self.fmt, self.margin = H, fmt, margin

    def _fields(self):
        hdr = self._buf[:24].view(np.int32)
        f = self._buf[:24].view(np.float32)
        hist = self._buf[24:24 + 4 * self.H].view(np.float32)
        return int(hdr[1]), float(f[4]), float(f[5]), hist.copy()

    @property
    def head(self) -> int:
        return self._fields()[0]

    @property
    def scale(self) -> np.float32:
        return np.float32(self._fields()[1])

    @property
    def scale_inv(self) -> np.float32:
        return np.float32(self._fields()[2])

    @property
    def hist(self) -> np.ndarray:
        return self._fields()[3]

    def update(self, amax: float, nonfinite: int = 0):
        lib().orc_delayed_update(_p(self._buf), np.float32(amax), int(nonfinite))


# ---------------------------------------------------------------- layouts

def pack_mx(codes: np.ndarray) -> np.ndarray:
    c = np.ascontiguousarray(codes, dtype=np.uint8)
    R, S = c.shape
    out = np.empty(-(-R // 128) * -(-S // 4) * 512, dtype=np.uint8)
    lib().orc_pack_mx(_p(c), R, S, _p(out))
    return out


def pack_block1x128(d: np.ndarray) -> np.ndarray:
    a = np.ascontiguousarray(d, dtype=np.float32)
    R, Kb = a.shape
    out = np.empty((Kb, -(-R // 128) * 128), dtype=np.float32)
    lib().orc_pack_block1x128(_p(a), R, Kb, _p(out))
    return out


def pad128(v: np.ndarray) -> np.ndarray:
    """A per-channel copy's factors as stored for the GEMM: fp32, one per row
    of the copy, padded to a multiple of 128 entries with 1.0, the factor the
    rule gives an all-zero row (amax 0 -> s = 1), as the 1x128 layout pads."""
    v = np.asarray(v, dtype=np.float32)
    out = np.ones(-(-v.size // 128) * 128, dtype=np.float32)
    out[:v.size] = v
    return out


# --------------------------------------------------------------- recipes

def quantize_generic(fmt: int, x_bits: np.ndarray, br: int, bc: int, rowwise: bool = True,
                     colwise: bool = False) -> dict:
    """Sub-channel blocks of user-set dimensions ("mastering FP8 LLM training
    1.5x speedup", scaling strategy 3), the blockwise rule of sec. 2.2 of the
    2025 guide on br x bc blocks (1 x b or b x b): the row copy quantizes x,
    the column copy quantizes x^T, each with br x bc blocks (for square blocks
    that is the transpose of the row copy).  scale_row / scale_col are the
    plain [ceil(R/br)][ceil(C/bc)] d of each copy; *_packed the library's
    layout (1 x b: K-block-major [ceil(C/b)][Rp], pads 1.0; b x b: plain)."""
    x = np.ascontiguousarray(x_bits, dtype=np.uint16)
    out: dict = {"sat_row": 0, "sat_col": 0, "nonfinite": 0}
    for which, on, m in (("row", rowwise, x), ("col", colwise, np.ascontiguousarray(x.T))):
        if not on:
            continue
        q, d, _, am, sat, nf = quant_blocks(m, br, bc, KIND_DIV, fmt)
        packed = pack_block1x128(d) if br == 1 else d
        out.update({"data_" + which: q, "scale_" + which: d, "scale_" + which + "_packed": packed,
                    "sat_" + which: sat, "nonfinite": nf})
    if br == bc:
        out["sat_col"] = 0  # the column copy of square blocks is the row copy's transpose: no count of its own
    return out


def quantize(kind: int, fmt: int, x_bits: np.ndarray, rowwise: bool = True, colwise: bool = False,
             state: Delayed | None = None) -> dict:
    """One quantize call of a recipe, returning what the product writes:

    data_row [R, C] / data_col [C, R] uint8 codes;
    scale_row / scale_col in the plain layout (per-tensor: scalar s;
    1x128: [R, C/128] / [C, R/128] fp32 d; 128x128: [R/128, C/128] / its
    transpose; MXFP8: [R, C/32] / [C, R/32] E8M0 codes) and, for 1x128 and
    MXFP8, *_packed in the GEMM layout; amax, scale, scale_inv (per-tensor);
    per-channel: scale_row [R] / scale_col [C] fp32 RN(1 / s), *_packed
    padded to 128 entries with 1.0, and mult_* (s) and amax_* per row / column;
    sat_row, sat_col, nonfinite counts.
    """
    x = np.ascontiguousarray(x_bits, dtype=np.uint16)
    R, C = x.shape
    out: dict = {}
    if kind in (PERTENSOR_CURRENT, PERTENSOR_DELAYED):
        if kind == PERTENSOR_CURRENT:
            q, sc, _, am, sat, nf = quant_blocks(x, R, C, KIND_MULT, fmt)
            s = np.float32(sc[0, 0]) if sc.size else np.float32(1.0)
            amax = float(am[0, 0]) if am.size else 0.0
        else:
            assert state is not None
            s = state.scale
            q, amax, sat, nf = cast_scaled(x, s, fmt)
        out.update(amax=np.float32(amax), scale=np.float32(s), scale_inv=np.float32(np.float32(1.0) / np.float32(s)),
                   sat_row=sat if rowwise else 0, sat_col=0, nonfinite=nf)
        if rowwise:
            out["data_row"] = q
        if colwise:
            out["data_col"] = np.ascontiguousarray(q.T)
        if kind == PERTENSOR_DELAYED:
            state.update(amax, nf)
        return out

    if kind == BLOCK_128x128:
        q, d, _, am, sat, nf = quant_blocks(x, 128, 128, KIND_DIV, fmt)
        out.update(nonfinite=nf, sat_row=sat if rowwise else 0, sat_col=0)
        if rowwise:
            out.update(data_row=q, scale_row=d)
        if colwise:
            out.update(data_col=np.ascontiguousarray(q.T), scale_col=np.ascontiguousarray(d.T))
        if not rowwise:
            out["sat_row"] = 0
        return out

    if kind == PERCHANNEL_CURRENT:
        # one block per row (row copy) / per column (column copy), multiply rule
        out.update(sat_row=0, sat_col=0, nonfinite=0)
        if R == 0 or C == 0:
            if rowwise:
                out.update(data_row=np.zeros((R, C), np.uint8), scale_row=np.ones(R, np.float32),
                           scale_row_packed=pad128(np.ones(R, np.float32)))
            if colwise:
                out.update(data_col=np.zeros((C, R), np.uint8), scale_col=np.ones(C, np.float32),
                           scale_col_packed=pad128(np.ones(C, np.float32)))
            return out
        if rowwise:
            q, sm, _, am, sat, nf = quant_blocks(x, 1, C, KIND_MULT, fmt)
            inv = (np.float32(1.0) / sm[:, 0]).astype(np.float32)
            out.update(data_row=q, scale_row=inv, scale_row_packed=pad128(inv), mult_row=sm[:, 0],
                       amax_row=am[:, 0], sat_row=sat, nonfinite=nf)
        if colwise:
            q, sm, _, am, sat, nf = quant_blocks(x, R, 1, KIND_MULT, fmt)
            inv = (np.float32(1.0) / sm[0, :]).astype(np.float32)
            out.update(data_col=np.ascontiguousarray(q.T), scale_col=inv, scale_col_packed=pad128(inv),
                       mult_col=sm[0, :], amax_col=am[0, :], sat_col=sat, nonfinite=nf)
        return out

    if kind == BLOCK_1x128:
        blk, k, pack = 128, KIND_DIV, pack_block1x128
    elif kind == MXFP8_1x32:
        blk, k, pack = 32, KIND_POW2, pack_mx
    else:
        raise ValueError(kind)
    nf = None
    out.update(sat_row=0, sat_col=0)
    if rowwise:
        q, d, e8, am, sat, nf = quant_blocks(x, 1, blk, k, fmt)
        srow = e8 if kind == MXFP8_1x32 else d
        out.update(data_row=q, scale_row=srow, scale_row_packed=pack(srow), sat_row=sat)
    if colwise:
        q, d, e8, am, sat, nf2 = quant_blocks(x, blk, 1, k, fmt)
        scol = np.ascontiguousarray((e8 if kind == MXFP8_1x32 else d).T)
        out.update(data_col=np.ascontiguousarray(q.T), scale_col=scol, scale_col_packed=pack(scol), sat_col=sat)
        nf = nf2 if nf is None else nf
    out["nonfinite"] = nf if nf is not None else 0
    return out


# ------------------------------------------------------------------ GEMM

def gemm_points(A: np.ndarray, fmtA: int, sA: np.ndarray, a_bm: int, a_bk: int,
                B: np.ndarray, fmtB: int, sB: np.ndarray, b_bn: int, b_bk: int,
                pm: np.ndarray, pn: np.ndarray) -> np.ndarray:
    """D[pm[i], pn[i]] of D = A . B^T in fp64 (see orc_gemm_points).  sA / sB
    are the dequantization scales in the plain layout [ceil(M/a_bm),
    ceil(K/a_bk)] (fp32); a per-tensor scale is a 1x1 array with a_bm = M,
    a_bk = K."""
    A = np.ascontiguousarray(A, dtype=np.uint8)
    B = np.ascontiguousarray(B, dtype=np.uint8)
    sA = np.ascontiguousarray(np.atleast_2d(sA), dtype=np.float32)
    sB = np.ascontiguousarray(np.atleast_2d(sB), dtype=np.float32)
    M, K = A.shape
    N, K2 = B.shape
    assert K == K2
    pm = np.ascontiguousarray(pm, dtype=np.int64)
    pn = np.ascontiguousarray(pn, dtype=np.int64)
    out = np.empty(pm.size, dtype=np.float64)
    lib().orc_gemm_points(_p(A), fmtA, _p(sA), a_bm, a_bk, sA.shape[1],
                          _p(B), fmtB, _p(sB), b_bn, b_bk, sB.shape[1],
                          M, N, K, _p(pm), _p(pn), pm.size, _p(out))
    return out


def gemm_full(A, fmtA, sA, a_bm, a_bk, B, fmtB, sB, b_bn, b_bk) -> np.ndarray:
    M, N = A.shape[0], B.shape[0]
    mm, nn = np.meshgrid(np.arange(M), np.arange(N), indexing="ij")
    return gemm_points(A, fmtA, sA, a_bm, a_bk, B, fmtB, sB, b_bn, b_bk, mm.ravel(), nn.ravel()).reshape(M, N)


def dequant_scales(kind: int, q: dict, which: str, rows: int, cols: int, block=(0, 0)):
    """(scale array, block rows, block cols) of a quantized copy for
    gemm_points: which = 'row' or 'col'; block = (br, bc) of a generic kind."""
    if kind == BLOCK_GENERIC:
        return q["scale_" + which], block[0], block[1]
    if kind in (PERTENSOR_CURRENT, PERTENSOR_DELAYED):
        return np.array([[q["scale_inv"]]], dtype=np.float32), rows, cols
    s = q["scale_" + which]
    if kind == BLOCK_128x128:
        return s, 128, 128
    if kind == BLOCK_1x128:
        return s, 1, 128
    if kind == MXFP8_1x32:
        return np.ldexp(np.float32(1.0), s.astype(np.int32) - 127).astype(np.float32), 1, 32
    if kind == PERCHANNEL_CURRENT:
        return np.ascontiguousarray(s.reshape(rows, 1)), 1, max(cols, 1)
    raise ValueError(kind)
