"""GEMM with the next quantize fused into its epilogue (fp8q_scaled_gemm_q,
fp8q_scaled_gemm_mxq).

The fused output must be exactly what the quantize step would make of the
GEMM's bf16 output: the oracle quantizes the kernel's own bf16 D with the
MXFP8 1x32 recipe ("2025 FP8 quantized-training guide", sec. 2.3) or the
1x128 recipe (sec. 2.2), and every code, scale byte (in the library's
layout) and counter must match.  D itself is the plain SM-pair GEMM's D bit
for bit, and without D the quantized output is the same.
"""
import numpy as np
import pytest
import torch

import oracle as O
from fp8_scaled_quantization_quantize_gb300 import inputs
from _helpers import assert_quant_equal, gpu_outputs

pytestmark = pytest.mark.gpu


def _api():
    from fp8_scaled_quantization_quantize_gb300 import api
    return api


# name, kind A, kind B, format A, format B
RECIPES = [
    ("pertensor", 0, 0, O.E4M3, O.E4M3),
    ("mxfp8", 4, 4, O.E4M3, O.E4M3),
    ("block_1x128_128x128", 2, 3, O.E4M3, O.E4M3),
    ("block_1x128_1x128", 2, 2, O.E4M3, O.E4M3),
    ("perchannel", 5, 5, O.E4M3, O.E4M3),
]


def _operands(api, kA, kB, fA, fB, M, N, K, seed):
    a = inputs.normal_bf16((M, K), seed)
    b = inputs.normal_bf16((N, K), seed + 1, 0.02)
    qa = api.quantize(a.cuda(), kA, fA, True, False)
    qb = api.quantize(b.cuda(), kB, fB, True, False)
    return qa, qb


OUT_KINDS = {"mxfp8": O.MXFP8_1x32, "1x128": O.BLOCK_1x128}


def _check_fused(api, qa, qb, fmt, ctx, kind=O.MXFP8_1x32):
    D, Dq = api.scaled_gemm_q(qa, False, qb, False, kind, fmt, want_d=True)
    torch.cuda.synchronize()
    got = gpu_outputs(Dq)
    ref = O.quantize(kind, fmt, inputs.bf16_bits(D.cpu()), True, False)
    assert_quant_equal(kind, got, ref, True, False, ctx)
    return D, Dq, got


SHAPES = [(256, 512, 256), (208, 288, 400), (384, 800, 528), (640, 1024, 1040), (208, 272, 400)]


@pytest.mark.parametrize("name,kA,kB,fA,fB", RECIPES, ids=[r[0] for r in RECIPES])
@pytest.mark.parametrize("M,N,K", SHAPES)
@pytest.mark.parametrize("fmt", [O.E4M3, O.E5M2])
@pytest.mark.parametrize("out_kind", list(OUT_KINDS))
def test_fused_output_quantize_matches_quantize_of_d(name, kA, kB, fA, fB, M, N, K, fmt, out_kind):
    kind = OUT_KINDS[out_kind]
    if kind == O.MXFP8_1x32 and N % 32:
        pytest.skip("the MXFP8 output takes N % 32 == 0")
    api = _api()
    qa, qb = _operands(api, kA, kB, fA, fB, M, N, K, 60 + M)
    D, Dq, got = _check_fused(api, qa, qb, fmt, f"{name} {M}x{N}x{K} fmt={fmt} out={out_kind}", kind)
    # D is the plain SM-pair GEMM's D
    api.gemm_set_variant(2)
    try:
        D2 = api.scaled_gemm(qa, False, qb, False)
        torch.cuda.synchronize()
    finally:
        api.gemm_set_variant(0)
    assert torch.equal(D.view(torch.int16), D2.view(torch.int16)), "fused D differs from the GEMM's D"
    # and without D the quantized output is the same
    none, Dq2 = api.scaled_gemm_q(qa, False, qb, False, kind, fmt, want_d=False)
    torch.cuda.synchronize()
    assert none is None
    got2 = gpu_outputs(Dq2)
    assert np.array_equal(got2["data_row"], got["data_row"])
    assert np.array_equal(got2["scale_row_bytes"], got["scale_row_bytes"])
    assert (got2["sat_row"], got2["nonfinite"]) == (got["sat_row"], got["nonfinite"])
    assert api.device_errors() == 0


@pytest.mark.parametrize("out_kind", list(OUT_KINDS))
def test_fused_output_counts_saturation(out_kind):
    """MXFP8 blocks whose scaled maximum lands in (448, 512) saturate: a
    typical N(0,1) product has many.  A 1x128 block saturates when d =
    RN(amax / 448) rounds below amax / 448, so its maximum divides to just
    above 448.  Both counts must equal the oracle's."""
    api = _api()
    qa, qb = _operands(api, 4, 4, O.E4M3, O.E4M3, 512, 1024, 512, 5)
    _, _, got = _check_fused(api, qa, qb, O.E4M3, "saturation", OUT_KINDS[out_kind])
    assert got["sat_row"] > 0


@pytest.mark.parametrize("out_kind", list(OUT_KINDS))
def test_fused_output_of_overflowing_d(out_kind):
    """A per-tensor GEMM whose fp32 result overflows: D is +-Inf in bf16, every
    element is counted as nonfinite and encodes to +-448 (satfinite), and the
    blocks' finite maximum is 0 (E8M0 127, 1x128 d = 1)."""
    api = _api()
    M, N, K = 256, 256, 128
    big = torch.full((M, K), 1e30, dtype=torch.bfloat16)
    qa = api.quantize(big.cuda(), 0, O.E4M3, True, False)
    qb = api.quantize(big[:N].clone().cuda(), 0, O.E4M3, True, False)
    D, Dq, got = _check_fused(api, qa, qb, O.E4M3, "overflow", OUT_KINDS[out_kind])
    assert torch.isinf(D.float()).all()
    assert got["nonfinite"] == M * N


def test_fused_1x128_output_of_d_with_nan_and_tiny_blocks():
    """1x128 output blocks holding NaN (a NaN operand row), and blocks whose
    maximum is tiny (d below the reciprocal shortcut's range, IEEE division):
    codes, scales and counters equal the oracle's quantize of D."""
    api = _api()
    M, N, K = 256, 384, 256
    a = inputs.normal_f32((M, K), 91)
    a[7, 3] = np.nan
    a[100:140, :] *= np.float32(2.0 ** -80)   # rows of D near 2^-76: d near 2^-84, the IEEE-division path
    b = inputs.normal_f32((N, K), 92)
    qa = api.quantize(inputs.to_bf16(a).cuda(), O.BLOCK_1x128, O.E4M3, True, False)
    qb = api.quantize(inputs.to_bf16(b).cuda(), O.BLOCK_128x128, O.E4M3, True, False)
    D, Dq, got = _check_fused(api, qa, qb, O.E4M3, "nan / tiny", O.BLOCK_1x128)
    assert got["nonfinite"] > 0


def test_fused_output_llama8b_fprop_sampled_rows():
    """The Llama-3-8B MLP fprop shape (MXFP8 X [8192x4096] . W^T [14336x4096]):
    the fused codes and scales of 64 sampled rows against the oracle's quantize
    of those rows of the kernel's D."""
    api = _api()
    X, W, _ = inputs.llama8b_mlp()
    qx = api.quantize(X.cuda(), 4, O.E4M3, True, False)
    qw = api.quantize(W.cuda(), 4, O.E4M3, True, False)
    D, Dq = api.scaled_gemm_mxq(qx, False, qw, False, O.E4M3, want_d=True)
    torch.cuda.synchronize()
    rows = np.sort(np.random.default_rng(3).choice(8192, 64, replace=False))
    Dr = D[torch.as_tensor(rows, device=D.device)].cpu()
    ref = O.quantize(O.MXFP8_1x32, O.E4M3, inputs.bf16_bits(Dr), True, False)
    assert np.array_equal(Dq.data_row[torch.as_tensor(rows, device=D.device)].cpu().numpy(), ref["data_row"])
    # scale bytes of the sampled rows from the packed tiles: row r, scale column k
    sb = Dq.scale_row.cpu().numpy()
    S = 14336 // 32
    tiles_c = 14336 // 128
    k = np.arange(S)[None, :]
    r = rows[:, None]
    off = ((r // 128) * tiles_c + k // 4) * 512 + (r % 32) * 16 + ((r % 128) // 32) * 4 + k % 4
    assert np.array_equal(sb[off], ref["scale_row"])
    assert api.device_errors() == 0


def test_fused_1x128_output_llama8b_up_proj_sampled_rows():
    """The blockwise Llama-3-8B up-projection (X 1x128 [4096x4096] . W^T
    128x128 [14336x4096]) with the next layer's 1x128 quantize of Y fused:
    64 sampled rows' codes and fp32 scales (K-block-major [112][4096]) against
    the oracle's quantize of those rows of the kernel's own bf16 Y."""
    api = _api()
    X, W = inputs.llama8b_up_proj()
    qx = api.quantize(X.cuda(), O.BLOCK_1x128, O.E4M3, True, False)
    qw = api.quantize(W.cuda(), O.BLOCK_128x128, O.E4M3, True, False)
    D, Dq = api.scaled_gemm_q(qx, False, qw, False, O.BLOCK_1x128, O.E4M3, want_d=True)
    torch.cuda.synchronize()
    rows = np.sort(np.random.default_rng(4).choice(4096, 64, replace=False))
    idx = torch.as_tensor(rows, device=D.device)
    ref = O.quantize(O.BLOCK_1x128, O.E4M3, inputs.bf16_bits(D[idx].cpu()), True, False)
    assert np.array_equal(Dq.data_row[idx].cpu().numpy(), ref["data_row"])
    sc = Dq.scale_row.cpu().numpy().view(np.float32).reshape(14336 // 128, 4096)
    assert np.array_equal(sc[:, rows].T, ref["scale_row"])
    assert api.device_errors() == 0


# ---------------------------------------------------------------- the column-wise copy too
# The next layer's wgrad reads the column-wise copy of this GEMM's output
# (blocks along M); with colwise the epilogue writes it as well, and the codes,
# scales and counters of both copies must equal the oracle's quantize of the
# kernel's own bf16 D with both copies.

def _check_fused_both(api, qa, qb, fmt, ctx, kind):
    D, Dq = api.scaled_gemm_q(qa, False, qb, False, kind, fmt, want_d=True, colwise=True)
    torch.cuda.synchronize()
    got = gpu_outputs(Dq)
    ref = O.quantize(kind, fmt, inputs.bf16_bits(D.cpu()), True, True)
    assert_quant_equal(kind, got, ref, True, True, ctx)
    return D, Dq, got


@pytest.mark.parametrize("name,kA,kB,fA,fB", RECIPES, ids=[r[0] for r in RECIPES])
@pytest.mark.parametrize("M,N,K", SHAPES)
@pytest.mark.parametrize("fmt", [O.E4M3, O.E5M2])
@pytest.mark.parametrize("out_kind", list(OUT_KINDS))
def test_fused_column_copy_matches_quantize_of_d(name, kA, kB, fA, fB, M, N, K, fmt, out_kind):
    kind = OUT_KINDS[out_kind]
    if kind == O.MXFP8_1x32 and N % 32:
        pytest.skip("the MXFP8 output takes N % 32 == 0")
    api = _api()
    qa, qb = _operands(api, kA, kB, fA, fB, M, N, K, 160 + M)
    D, Dq, got = _check_fused_both(api, qa, qb, fmt, f"{name} {M}x{N}x{K} fmt={fmt} out={out_kind} +col", kind)
    # the row copy is the one the row-only call writes
    _, Dr = api.scaled_gemm_q(qa, False, qb, False, kind, fmt, want_d=False)
    torch.cuda.synchronize()
    rb = api.scale_bytes(kind, M, N, True, False)[0]
    assert torch.equal(Dr.data_row, Dq.data_row) and torch.equal(Dr.scale_row[:rb], Dq.scale_row[:rb])
    assert api.device_errors() == 0


@pytest.mark.parametrize("out_kind", list(OUT_KINDS))
def test_fused_column_copy_counts_saturation(out_kind):
    """Column blocks saturate like row blocks (a block's scaled maximum above
    fmax): the column copy's count, counters[1], equals the oracle's."""
    api = _api()
    qa, qb = _operands(api, 4, 4, O.E4M3, O.E4M3, 512, 1024, 512, 15)
    _, _, got = _check_fused_both(api, qa, qb, O.E4M3, "column saturation", OUT_KINDS[out_kind])
    assert got["sat_col"] > 0


@pytest.mark.parametrize("out_kind", list(OUT_KINDS))
def test_fused_column_copy_of_overflowing_d(out_kind):
    """An overflowing per-tensor GEMM (D all +-Inf): both copies encode +-fmax,
    every block's finite maximum is 0."""
    api = _api()
    M, N, K = 256, 256, 128
    big = torch.full((M, K), 1e30, dtype=torch.bfloat16)
    qa = api.quantize(big.cuda(), 0, O.E4M3, True, False)
    qb = api.quantize(big[:N].clone().cuda(), 0, O.E4M3, True, False)
    D, Dq, got = _check_fused_both(api, qa, qb, O.E4M3, "overflow +col", OUT_KINDS[out_kind])
    assert got["nonfinite"] == M * N


@pytest.mark.parametrize("out_kind", list(OUT_KINDS))
def test_fused_column_copy_with_nan_and_tiny_blocks(out_kind):
    """Columns of D holding a NaN (from a NaN operand row) and rows of D near
    2^-76 (1x128 column blocks with d below the reciprocal shortcut's range
    mix with normal ones): both copies equal the oracle's quantize of D."""
    api = _api()
    M, N, K = 384, 384, 256
    a = inputs.normal_f32((M, K), 93)
    a[7, 3] = np.nan
    a[128:256, :] *= np.float32(2.0 ** -80)
    b = inputs.normal_f32((N, K), 94)
    qa = api.quantize(inputs.to_bf16(a).cuda(), O.BLOCK_1x128, O.E4M3, True, False)
    qb = api.quantize(inputs.to_bf16(b).cuda(), O.BLOCK_128x128, O.E4M3, True, False)
    D, Dq, got = _check_fused_both(api, qa, qb, O.E4M3, "nan / tiny +col", OUT_KINDS[out_kind])
    assert got["nonfinite"] > 0


@pytest.mark.parametrize("out_kind", list(OUT_KINDS))
def test_fused_column_copy_many_tiles_per_pair(out_kind):
    """More tiles than SM pairs (each pair's epilogue runs several tiles, so the
    1x128 exchange alternates its two buffers): both copies of a
    2048 x 4096 x 256 output equal the oracle's."""
    api = _api()
    qa, qb = _operands(api, 2, 3, O.E4M3, O.E4M3, 2048, 4096, 256, 21)
    _check_fused_both(api, qa, qb, O.E5M2, "many tiles +col", OUT_KINDS[out_kind])
    assert api.device_errors() == 0


def test_fused_column_copy_llama8b_fprop_sampled_columns():
    """The Llama-3-8B MLP fprop (MXFP8 X [8192x4096] . W^T [14336x4096]) with
    both copies of Y fused: 64 sampled columns of Y -- rows of the column copy
    -- against the oracle's quantize of those rows of Y^T (the column copy of
    Y is the row copy of Y^T), codes and E8M0 bytes."""
    api = _api()
    X, W, _ = inputs.llama8b_mlp()
    qx = api.quantize(X.cuda(), 4, O.E4M3, True, False)
    qw = api.quantize(W.cuda(), 4, O.E4M3, True, False)
    D, Dq = api.scaled_gemm_mxq(qx, False, qw, False, O.E4M3, want_d=True, colwise=True)
    torch.cuda.synchronize()
    cols = np.sort(np.random.default_rng(5).choice(14336, 64, replace=False))
    idx = torch.as_tensor(cols, device=D.device)
    ref = O.quantize(O.MXFP8_1x32, O.E4M3, inputs.bf16_bits(D.t()[idx].contiguous().cpu()), True, False)
    assert np.array_equal(Dq.data_col[idx].cpu().numpy(), ref["data_row"])
    sb = Dq.scale_col.cpu().numpy()
    S = 8192 // 32
    tiles_c = 8192 // 128
    k = np.arange(S)[None, :]
    r = cols[:, None]
    off = ((r // 128) * tiles_c + k // 4) * 512 + (r % 32) * 16 + ((r % 128) // 32) * 4 + k % 4
    assert np.array_equal(sb[off], ref["scale_row"])
    assert api.device_errors() == 0


def test_fused_1x128_column_copy_llama8b_up_proj_sampled_columns():
    """The blockwise Llama-3-8B up-projection with both 1x128 copies of Y
    fused: 64 sampled columns of Y against the oracle's quantize of those rows
    of Y^T: codes and the fp32 scales [32][14336] of those columns."""
    api = _api()
    X, W = inputs.llama8b_up_proj()
    qx = api.quantize(X.cuda(), O.BLOCK_1x128, O.E4M3, True, False)
    qw = api.quantize(W.cuda(), O.BLOCK_128x128, O.E4M3, True, False)
    D, Dq = api.scaled_gemm_q(qx, False, qw, False, O.BLOCK_1x128, O.E4M3, want_d=True, colwise=True)
    torch.cuda.synchronize()
    cols = np.sort(np.random.default_rng(6).choice(14336, 64, replace=False))
    idx = torch.as_tensor(cols, device=D.device)
    ref = O.quantize(O.BLOCK_1x128, O.E4M3, inputs.bf16_bits(D.t()[idx].contiguous().cpu()), True, False)
    assert np.array_equal(Dq.data_col[idx].cpu().numpy(), ref["data_row"])
    sc = Dq.scale_col.cpu().numpy().view(np.float32).reshape(4096 // 128, 14336)
    assert np.array_equal(sc[:, cols].T, ref["scale_row"])
    assert api.device_errors() == 0
