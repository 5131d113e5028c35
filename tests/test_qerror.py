"""The error study's arithmetic (qerror.py) pinned on the CPU: the error
formula on a hand example, and the row-wise dequantization of every scale
layout against the oracle's own decode and plain-layout scales."""
import math
import types

import numpy as np
import pytest
import torch

import oracle as O
from fp8_scaled_quantization_quantize_gb300 import inputs, qerror
from _helpers import expected_scale_bytes


def test_error_formula_hand_example():
    x = torch.tensor([3.0, 4.0, float("nan")])
    dq = torch.tensor([3.0, 4.5, 7.0])
    e = qerror.error(x, dq)
    # ||(0, 0.5)|| / ||(3, 4)|| = 0.1, SQNR = 10 log10(25 / 0.25) = 20 dB; NaN dropped
    assert e["rel_err"] == pytest.approx(0.1, abs=1e-15)
    assert e["sqnr_db"] == pytest.approx(20.0, abs=1e-12)


@pytest.mark.parametrize("kind", [0, 2, 3, 4, 5])
@pytest.mark.parametrize("fmt", [O.E4M3, O.E5M2])
def test_dequantize_layouts_match_the_oracle(kind, fmt):
    R, C = 200, 272
    x = inputs.to_bf16(inputs.with_outlier_elements(inputs.normal_f32((R, C), 11), 0.01, 100.0, 12))
    ref = O.quantize(kind, fmt, inputs.bf16_bits(x), True, False)
    sb = expected_scale_bytes(kind, ref, "row")
    qt = types.SimpleNamespace(
        kind=kind, fmt=fmt, rows=R, cols=C, data_row=torch.from_numpy(ref["data_row"]),
        scale_row=None if sb is None else torch.from_numpy(np.ascontiguousarray(sb)),
        scale_inv=torch.tensor([float(ref.get("scale_inv", 1.0))], dtype=torch.float32))
    got = qerror.dequantize_rowwise(qt).double().numpy()
    s, bm, bk = O.dequant_scales(kind, ref, "row", R, C)
    full = np.repeat(np.repeat(np.asarray(s, dtype=np.float64), bm, 0)[:R], bk, 1)[:, :C]
    want = O.decode(ref["data_row"], fmt) * full
    # one fp32 rounding of the product on the torch side
    assert np.allclose(got, want, rtol=2.0 ** -23, atol=0.0)
    e = qerror.error(x.float(), torch.from_numpy(want))
    assert 0.0 < e["rel_err"] < 0.1 and math.isfinite(e["sqnr_db"])


@pytest.mark.parametrize("block", [(1, 32), (1, 64), (1, 256), (32, 32), (64, 64), (256, 256)],
                         ids=["1x32", "1x64", "1x256", "32x32", "64x64", "256x256"])
def test_dequantize_generic_layouts_match_the_oracle(block):
    """The sub-channel block layouts (1 x b: [ceil(C/b)][R up to 128], b x b:
    [ceil(R/b)][ceil(C/b)]) expanded by qerror.py equal the oracle's plain
    block scales, on a shape with ragged edges."""
    R, C = 200, 272
    x = inputs.to_bf16(inputs.with_outlier_elements(inputs.normal_f32((R, C), 13), 0.01, 100.0, 14))
    ref = O.quantize_generic(O.E4M3, inputs.bf16_bits(x), *block, True, False)
    sb = expected_scale_bytes(O.BLOCK_GENERIC, ref, "row")
    qt = types.SimpleNamespace(kind=O.BLOCK_GENERIC, fmt=O.E4M3, rows=R, cols=C, block=block,
                               data_row=torch.from_numpy(ref["data_row"]),
                               scale_row=torch.from_numpy(np.ascontiguousarray(sb)), scale_inv=None)
    got = qerror.dequantize_rowwise(qt).double().numpy()
    s, bm, bk = O.dequant_scales(O.BLOCK_GENERIC, ref, "row", R, C, block=block)
    full = np.repeat(np.repeat(np.asarray(s, dtype=np.float64), bm, 0)[:R], bk, 1)[:, :C]
    want = O.decode(ref["data_row"], O.E4M3) * full
    assert np.allclose(got, want, rtol=2.0 ** -23, atol=0.0)
