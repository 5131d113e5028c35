"""Scaled GEMM on generic sub-channel blocks ("mastering FP8 LLM training 1.5x
speedup", scaling strategy 3 and Figure 1's 1D1D / 1D2D arrangements): A
quantized with 1 x b blocks along K, B with 1 x b or b x b blocks, the
partial sums of every b-wide K block scaled by d_A * d_B and summed in fp32
(b = 32, 64, 128, 256).  Compared with the fp64 oracle of the same quantized
operands (normwise relative error <= 2e-3, fp32 output <= 1e-4) for fprop on
the row-wise copies and wgrad on the column-wise copies, at ragged shapes
(K not a multiple of b, partial tiles); generic 1 x 128 / 128 x 128 gives the
specialised recipes' GEMM bit for bit."""
import numpy as np
import pytest
import torch

import oracle as O
from fp8_scaled_quantization_quantize_gb300 import inputs
from tests._helpers import bits_of

pytestmark = pytest.mark.gpu


def _api():
    from fp8_scaled_quantization_quantize_gb300 import api
    return api


def _rel(got: torch.Tensor, ref: np.ndarray) -> float:
    g = got.float().cpu().numpy().astype(np.float64)
    return float(np.linalg.norm(g - ref) / np.linalg.norm(ref))


@pytest.mark.parametrize("b", [32, 64, 128, 256])
@pytest.mark.parametrize("square_b", [False, True], ids=["1d1d", "1d2d"])
@pytest.mark.parametrize("M,N,K", [(256, 512, 512), (208, 288, 400), (384, 800, 1040)])
@pytest.mark.parametrize("out", ["bf16", "fp32"])
def test_generic_block_fprop_matches_oracle(b, square_b, M, N, K, out):
    api = _api()
    a = inputs.with_outlier_columns(inputs.normal_f32((M, K), 500 + b), 0.02, 50.0, 7)
    bm = inputs.normal_f32((N, K), 501 + b, 0.02)
    xa, xb = inputs.to_bf16(a), inputs.to_bf16(bm)
    ab, bb = (1, b), ((b, b) if square_b else (1, b))
    qa = api.quantize(xa.cuda(), O.BLOCK_GENERIC, O.E4M3, True, False, block=ab)
    qb = api.quantize(xb.cuda(), O.BLOCK_GENERIC, O.E4M3, True, False, block=bb)
    D = api.scaled_gemm(qa, False, qb, False, torch.bfloat16 if out == "bf16" else torch.float32)
    torch.cuda.synchronize()
    ra = O.quantize_generic(O.E4M3, bits_of(xa), *ab, True, False)
    rb = O.quantize_generic(O.E4M3, bits_of(xb), *bb, True, False)
    ref = O.gemm_full(ra["data_row"], O.E4M3, ra["scale_row"], *ab, rb["data_row"], O.E4M3, rb["scale_row"], *bb)
    rel = _rel(D, ref)
    assert rel <= (2e-3 if out == "bf16" else 1e-4), rel
    assert api.device_errors() == 0


@pytest.mark.parametrize("b", [32, 64, 256])
def test_generic_block_wgrad_on_column_copies(b):
    """wgrad dW = dY^T . X on the column-wise copies (blocks of b along the
    token dimension), E5M2 dY and E4M3 X."""
    api = _api()
    T_, F_, H_ = 400, 288, 320
    dy = inputs.to_bf16(inputs.normal_f32((T_, F_), 610 + b, 1e-3))
    x = inputs.to_bf16(inputs.normal_f32((T_, H_), 611 + b))
    qdy = api.quantize(dy.cuda(), O.BLOCK_GENERIC, O.E5M2, False, True, block=(1, b))
    qx = api.quantize(x.cuda(), O.BLOCK_GENERIC, O.E4M3, False, True, block=(1, b))
    D = api.scaled_gemm(qdy, True, qx, True)
    torch.cuda.synchronize()
    rdy = O.quantize_generic(O.E5M2, bits_of(dy), 1, b, False, True)
    rx = O.quantize_generic(O.E4M3, bits_of(x), 1, b, False, True)
    ref = O.gemm_full(rdy["data_col"], O.E5M2, rdy["scale_col"], 1, b, rx["data_col"], O.E4M3, rx["scale_col"], 1, b)
    assert _rel(D, ref) <= 2e-3
    assert api.device_errors() == 0


def test_generic_128_blocks_equal_the_specialised_recipes():
    api = _api()
    a = inputs.normal_bf16((512, 768), 620)
    w = inputs.normal_bf16((640, 768), 621, 0.02)
    qa_g = api.quantize(a.cuda(), O.BLOCK_GENERIC, O.E4M3, True, False, block=(1, 128))
    qw_g = api.quantize(w.cuda(), O.BLOCK_GENERIC, O.E4M3, True, False, block=(128, 128))
    qa = api.quantize(a.cuda(), O.BLOCK_1x128, O.E4M3, True, False)
    qw = api.quantize(w.cuda(), O.BLOCK_128x128, O.E4M3, True, False)
    assert torch.equal(qa_g.data_row, qa.data_row) and torch.equal(qa_g.scale_row, qa.scale_row)
    assert torch.equal(qw_g.data_row, qw.data_row) and torch.equal(qw_g.scale_row, qw.scale_row)
    for variant in (1, 2):
        api.gemm_set_variant(variant)
        try:
            D1 = api.scaled_gemm(qa_g, False, qw_g, False)
            D2 = api.scaled_gemm(qa, False, qw, False)
            torch.cuda.synchronize()
        finally:
            api.gemm_set_variant(0)
        assert torch.equal(D1.view(torch.int16), D2.view(torch.int16))


def test_generic_gemm_rejects_mismatched_blocks():
    from fp8_scaled_quantization_quantize_gb300 import _lib as L
    api = _api()
    a = inputs.normal_bf16((256, 256), 630)
    qa = api.quantize(a.cuda(), O.BLOCK_GENERIC, O.E4M3, True, False, block=(1, 64))
    qb = api.quantize(a.cuda(), O.BLOCK_GENERIC, O.E4M3, True, False, block=(1, 32))
    qc = api.quantize(a.cuda(), O.BLOCK_GENERIC, O.E4M3, True, False, block=(64, 64))
    for A, B in ((qa, qb), (qc, qa)):   # different K blocks; 2D blocks on the A side
        with pytest.raises(L.Fp8qError) as e:
            api.scaled_gemm(A, False, B, False)
        assert e.value.status == L.ERR_DTYPE
    assert api.device_errors() == 0
