"""The error study on the CUDA path's outputs: the same errors as on the
oracle's outputs (the codes and scales are bit-exact), and the direction the
pages report ("2025 FP8 quantized-training guide", sec. 2.2): on activations
with outlier channels, 1x128 blocks leave less error than one per-tensor
scale."""
import numpy as np
import pytest
import torch

import oracle as O
from fp8_scaled_quantization_quantize_gb300 import inputs, qerror

pytestmark = pytest.mark.gpu


def test_errors_on_gpu_outputs_equal_the_oracles_and_order_as_reported():
    from fp8_scaled_quantization_quantize_gb300 import api
    x = inputs.to_bf16(inputs.with_outlier_columns(inputs.normal_f32((1024, 4096), 0), 0.01, 100.0, 2))
    errs = {}
    for kind in (0, 2, 3, 4, 5):
        qt = api.quantize(x.cuda(), kind, O.E4M3, True, False)
        e_gpu = qerror.error(x.float().cuda(), qerror.dequantize_rowwise(qt))
        ref = O.quantize(kind, O.E4M3, inputs.bf16_bits(x), True, False)
        s, bm, bk = O.dequant_scales(kind, ref, "row", *x.shape)
        full = np.repeat(np.repeat(np.asarray(s, dtype=np.float64), bm, 0)[: x.shape[0]], bk, 1)[:, : x.shape[1]]
        want = (O.decode(ref["data_row"], O.E4M3) * full).astype(np.float32)
        e_ref = qerror.error(x.float(), torch.from_numpy(want))
        assert e_gpu["rel_err"] == pytest.approx(e_ref["rel_err"], rel=1e-12)
        errs[kind] = e_gpu["rel_err"]
    # 1x128 blocks along the outlier channels' rows isolate them; 128x128 tiles
    # and MXFP8 (whose power-of-two scale puts block maxima in [256, 512) and
    # saturates the top of that range) are reported by bench.py --mode qerror
    assert errs[2] < 0.5 * errs[0], errs


@pytest.mark.parametrize("block", [(1, 32), (1, 64), (1, 256), (32, 32), (64, 64), (256, 256)],
                         ids=["1x32", "1x64", "1x256", "32x32", "64x64", "256x256"])
def test_generic_block_errors_equal_the_oracles(block):
    """The sub-channel block shapes ("mastering FP8 LLM training 1.5x speedup",
    scaling strategy 3) in the error study: the errors of the GPU's codes and
    scales, dequantized through their documented layout, equal those of the
    oracle's quantization (dequantized by the oracle's own scale expansion);
    1 x b blocks leave less error than one per-tensor scale, and less than
    half of it for b <= 64 (with 1 % outlier channels most 256-wide blocks
    hold one, so their maximum is the outlier's, as per tensor)."""
    from fp8_scaled_quantization_quantize_gb300 import api
    x = inputs.to_bf16(inputs.with_outlier_columns(inputs.normal_f32((1024, 4096), 0), 0.01, 100.0, 2))
    qt = api.quantize(x.cuda(), O.BLOCK_GENERIC, O.E4M3, True, False, block=block)
    e_gpu = qerror.error(x.float().cuda(), qerror.dequantize_rowwise(qt))
    ref = O.quantize_generic(O.E4M3, inputs.bf16_bits(x), *block, True, False)
    s, bm, bk = O.dequant_scales(O.BLOCK_GENERIC, ref, "row", *x.shape, block=block)
    full = np.repeat(np.repeat(np.asarray(s, dtype=np.float64), bm, 0)[: x.shape[0]], bk, 1)[:, : x.shape[1]]
    want = (O.decode(ref["data_row"], O.E4M3) * full).astype(np.float32)
    e_ref = qerror.error(x.float(), torch.from_numpy(want))
    assert e_gpu["rel_err"] == pytest.approx(e_ref["rel_err"], rel=1e-12)
    if block[0] == 1:
        qp = api.quantize(x.cuda(), O.PERTENSOR_CURRENT, O.E4M3, True, False)
        e_pt = qerror.error(x.float().cuda(), qerror.dequantize_rowwise(qp))
        assert e_gpu["rel_err"] < (0.5 if block[1] <= 64 else 1.0) * e_pt["rel_err"], (e_gpu, e_pt)
