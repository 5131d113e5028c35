"""Quantization error of the recipes on the same data.

The pages compare scaling granularities by the error they leave ("2025 FP8
quantized-training guide", sec. 2.2: blockwise scaling lowers the
quantization error against per-tensor scaling on data with outliers;
"mastering FP8 LLM training 1.5x speedup", scaling strategies 2-4).  This
module restates that comparison on synthetic tensors: it dequantizes a
quantized row-wise copy with its own scales and reports the normwise relative
error ||dq(q) - x||_F / ||x||_F and the SQNR 10 log10(||x||^2 / ||dq(q) - x||^2)
over the finite elements of x.

Analysis only, not the quantize -> GEMM path: the dequantization here is plain
torch arithmetic on the library's outputs (codes decoded through torch's float8
dtypes, scales expanded from their documented layouts).
"""
from __future__ import annotations

import math

import torch

from ._lib import (BLOCK_1x128, BLOCK_128x128, BLOCK_GENERIC, E4M3, MXFP8_1x32, PERCHANNEL_CURRENT, PERTENSOR_CURRENT,
                   PERTENSOR_DELAYED)


def _cdiv(a: int, b: int) -> int:
    return -(-a // b)


def decode(codes: torch.Tensor, fmt: int) -> torch.Tensor:
    """fp32 values of uint8 FP8 codes (E4M3 or E5M2)."""
    dt = torch.float8_e4m3fn if fmt == E4M3 else torch.float8_e5m2
    return codes.contiguous().view(dt).float()


def row_scales(qt) -> torch.Tensor:
    """The dequantization factor of every element of the row-wise copy, fp32
    [rows][cols], expanded from the copy's scale layout."""
    R, C = qt.rows, qt.cols
    dev = qt.data_row.device
    if qt.kind in (PERTENSOR_CURRENT, PERTENSOR_DELAYED):
        return qt.scale_inv.to(dev).float().reshape(1, 1).expand(R, C)
    buf = qt.scale_row
    if qt.kind == PERCHANNEL_CURRENT:
        return buf.view(torch.float32)[:R].reshape(R, 1).expand(R, C)
    if qt.kind == BLOCK_128x128:
        s = buf.view(torch.float32)[: _cdiv(R, 128) * _cdiv(C, 128)].reshape(_cdiv(R, 128), _cdiv(C, 128))
        return s.repeat_interleave(128, 0)[:R].repeat_interleave(128, 1)[:, :C]
    if qt.kind == BLOCK_1x128 or (qt.kind == BLOCK_GENERIC and qt.block[0] == 1):
        b = 128 if qt.kind == BLOCK_1x128 else qt.block[1]
        Rp = _cdiv(R, 128) * 128
        s = buf.view(torch.float32)[: _cdiv(C, b) * Rp].reshape(_cdiv(C, b), Rp)[:, :R].t()
        return s.repeat_interleave(b, 1)[:, :C]
    if qt.kind == BLOCK_GENERIC:  # b x b blocks: [ceil(R/b)][ceil(C/b)]
        b = qt.block[1]
        s = buf.view(torch.float32)[: _cdiv(R, b) * _cdiv(C, b)].reshape(_cdiv(R, b), _cdiv(C, b))
        return s.repeat_interleave(b, 0)[:R].repeat_interleave(b, 1)[:, :C]
    if qt.kind == MXFP8_1x32:
        S, tiles_c = _cdiv(C, 32), _cdiv(C, 128)
        r = torch.arange(R, device=dev).reshape(R, 1)
        k = torch.arange(S, device=dev).reshape(1, S)
        off = ((r // 128) * tiles_c + k // 4) * 512 + (r % 32) * 16 + ((r % 128) // 32) * 4 + k % 4
        e = buf[off.reshape(-1)].reshape(R, S).to(torch.int32) - 127
        s = torch.ldexp(torch.ones_like(e, dtype=torch.float32), e)
        return s.repeat_interleave(32, 1)[:, :C]
    raise ValueError(qt.kind)


def dequantize_rowwise(qt) -> torch.Tensor:
    """dq(q) = decode(code) * dequantization factor, fp32 [rows][cols]."""
    return decode(qt.data_row, qt.fmt) * row_scales(qt)


def error(x: torch.Tensor, dq: torch.Tensor) -> dict:
    """Normwise relative error and SQNR of dq against x over x's finite
    elements, in fp64."""
    xf = x.double()
    keep = torch.isfinite(xf)
    d = torch.where(keep, dq.double() - xf, torch.zeros_like(xf))
    xs = torch.where(keep, xf, torch.zeros_like(xf))
    num = float((d * d).sum())
    den = float((xs * xs).sum())
    rel = math.sqrt(num / den) if den > 0 else 0.0
    sqnr = 10.0 * math.log10(den / num) if num > 0 else math.inf
    return {"rel_err": rel, "sqnr_db": sqnr}
