"""Seeded random sweep over the quantize and GEMM parameter space against the
oracle: shapes drawn with ragged edges (rows a multiple of 16 where a column
copy needs it, columns a multiple of 16), every recipe including the generic
block shapes, both formats, random copies and value mixes (outliers, zero
stripes, NaN / Inf, whole tensors scaled by 1e-30 to 1e30, ties of block
maxima).  Quantize outputs bit-exact; GEMMs of random shapes and recipes
within 2e-3 normwise on every output."""
import numpy as np
import pytest
import torch

import oracle as O
from fp8_scaled_quantization_quantize_gb300 import inputs
from tests._helpers import assert_quant_equal, bits_of, gpu_outputs

pytestmark = pytest.mark.gpu

KINDS = [O.PERTENSOR_CURRENT, O.BLOCK_1x128, O.BLOCK_128x128, O.MXFP8_1x32, O.PERCHANNEL_CURRENT, O.BLOCK_GENERIC]
BLOCKS = [(1, 32), (1, 64), (1, 128), (1, 256), (32, 32), (64, 64), (128, 128), (256, 256)]


def _values(rng, shape):
    """One of several value mixes, as bf16."""
    mix = rng.integers(0, 5)
    x = rng.standard_normal(shape, dtype=np.float32)
    if mix == 1:   # outlier elements
        idx = rng.choice(x.size, size=max(1, x.size // 100), replace=False)
        x.reshape(-1)[idx] *= np.float32(rng.choice([100.0, 1e4, 1e-30]))
    elif mix == 2:  # the whole tensor scaled by 1e-30 .. 1e30, a zero stripe
        x *= np.float32(10.0 ** rng.uniform(-30, 30))
        x[:, : min(5, shape[1])] = 0.0
    elif mix == 3:  # NaN / Inf sprinkled
        for v in (np.nan, np.inf, -np.inf):
            x.reshape(-1)[rng.integers(0, x.size)] = v
    elif mix == 4:  # constant blocks (ties of the block maximum)
        x = np.round(x * 4.0) / 4.0
    return inputs.to_bf16(x)


@pytest.mark.parametrize("case", range(240))
def test_quantize_random_cases(case):
    from fp8_scaled_quantization_quantize_gb300 import api
    rng = np.random.default_rng(1000 + case)
    kind = KINDS[case % len(KINDS)]
    fmt = O.E4M3 if rng.random() < 0.6 else O.E5M2
    rowwise, colwise = [(True, False), (False, True), (True, True)][rng.integers(0, 3)]
    R = int(rng.integers(1, 40)) * 16
    C = int(rng.integers(1, 70)) * 16
    x = _values(rng, (R, C))
    if kind == O.BLOCK_GENERIC:
        block = BLOCKS[rng.integers(0, len(BLOCKS))]
        qt = api.quantize(x.cuda(), kind, fmt, rowwise, colwise, block=block)
        ref = O.quantize_generic(fmt, bits_of(x), *block, rowwise, colwise)
    else:
        block = None
        qt = api.quantize(x.cuda(), kind, fmt, rowwise, colwise)
        ref = O.quantize(kind, fmt, bits_of(x), rowwise, colwise)
    assert_quant_equal(kind, gpu_outputs(qt), ref, rowwise, colwise,
                       f"case {case}: kind {kind} block {block} fmt {fmt} {R}x{C} copies {rowwise},{colwise}")
    assert api.device_errors() == 0


RECIPES = [(O.PERTENSOR_CURRENT, O.PERTENSOR_CURRENT, None), (O.BLOCK_1x128, O.BLOCK_128x128, None),
           (O.BLOCK_1x128, O.BLOCK_1x128, None), (O.MXFP8_1x32, O.MXFP8_1x32, None),
           (O.PERCHANNEL_CURRENT, O.PERCHANNEL_CURRENT, None), (O.BLOCK_GENERIC, O.BLOCK_GENERIC, 64)]


@pytest.mark.parametrize("case", range(120))
def test_gemm_random_cases(case):
    from fp8_scaled_quantization_quantize_gb300 import api
    rng = np.random.default_rng(2000 + case)
    ka, kb, gb = RECIPES[case % len(RECIPES)]
    M = int(rng.integers(1, 48)) * 16
    N = int(rng.integers(1, 48)) * 32
    K = int(rng.integers(1, 24)) * (64 if gb else 32)
    fa = O.E4M3 if rng.random() < 0.7 else O.E5M2
    a = inputs.to_bf16(rng.standard_normal((M, K), dtype=np.float32))
    b = inputs.to_bf16(rng.standard_normal((N, K), dtype=np.float32) * np.float32(0.02))
    blk_a = (1, gb) if gb else (0, 0)
    blk_b = (gb, gb) if gb else (0, 0)
    qa = api.quantize(a.cuda(), ka, fa, True, False, block=blk_a)
    qb = api.quantize(b.cuda(), kb, O.E4M3, True, False, block=blk_b)
    D = api.scaled_gemm(qa, False, qb, False)
    torch.cuda.synchronize()
    if gb:
        ra = O.quantize_generic(fa, bits_of(a), *blk_a, True, False)
        rb = O.quantize_generic(O.E4M3, bits_of(b), *blk_b, True, False)
    else:
        ra = O.quantize(ka, fa, bits_of(a), True, False)
        rb = O.quantize(kb, O.E4M3, bits_of(b), True, False)
    assert np.array_equal(qa.data_row.cpu().numpy(), ra["data_row"])
    assert np.array_equal(qb.data_row.cpu().numpy(), rb["data_row"])
    sa, abm, abk = O.dequant_scales(ka, ra, "row", M, K, block=blk_a)
    sb, bbn, bbk = O.dequant_scales(kb, rb, "row", N, K, block=blk_b)
    ref = O.gemm_full(ra["data_row"], fa, sa, abm, abk, rb["data_row"], O.E4M3, sb, bbn, bbk)
    got = D.float().cpu().numpy().astype(np.float64)
    rel = np.linalg.norm(got - ref) / max(np.linalg.norm(ref), 1e-300)
    assert np.all(np.isfinite(got)) and rel <= 2e-3, (case, ka, kb, gb, M, N, K, fa, rel)
    assert api.device_errors() == 0


FUSED_RECIPES = [(O.PERTENSOR_CURRENT, O.PERTENSOR_CURRENT), (O.BLOCK_1x128, O.BLOCK_128x128),
                 (O.BLOCK_1x128, O.BLOCK_1x128), (O.MXFP8_1x32, O.MXFP8_1x32), (O.PERCHANNEL_CURRENT, O.PERCHANNEL_CURRENT)]


@pytest.mark.parametrize("case", range(60))
def test_fused_output_quantize_random_cases(case):
    """The GEMM with the next layer's quantize in its epilogue on random
    shapes: the fused codes, scales and counters equal the oracle's quantize
    of the kernel's own bf16 D (MXFP8 1x32 or 1x128 output, either format,
    the column-wise copy as well in half of the cases)."""
    from fp8_scaled_quantization_quantize_gb300 import api
    rng = np.random.default_rng(3000 + case)
    ka, kb = FUSED_RECIPES[case % len(FUSED_RECIPES)]
    out_kind = O.MXFP8_1x32 if case % 2 else O.BLOCK_1x128
    fmt = O.E4M3 if rng.random() < 0.6 else O.E5M2
    M = int(rng.integers(1, 40)) * 16
    N = int(rng.integers(1, 40)) * 32
    K = int(rng.integers(1, 20)) * 32
    scale = np.float32(10.0 ** rng.uniform(-3, 3))
    a = inputs.to_bf16(rng.standard_normal((M, K), dtype=np.float32) * scale)
    b = inputs.to_bf16(rng.standard_normal((N, K), dtype=np.float32) * np.float32(0.02))
    qa = api.quantize(a.cuda(), ka, O.E4M3, True, False)
    qb = api.quantize(b.cuda(), kb, O.E4M3, True, False)
    col = (case // 2) % 2 == 1
    D, Dq = api.scaled_gemm_q(qa, False, qb, False, out_kind, fmt, want_d=True, colwise=col)
    torch.cuda.synchronize()
    ref = O.quantize(out_kind, fmt, inputs.bf16_bits(D.cpu()), True, col)
    assert_quant_equal(out_kind, gpu_outputs(Dq), ref, True, col,
                       f"case {case}: {ka}x{kb} out {out_kind} fmt {fmt} {M}x{N}x{K} col {col}")
    assert api.device_errors() == 0
