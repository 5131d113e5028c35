"""Parity of the generic sub-channel block recipe (BLOCK_GENERIC: 1 x b and
b x b blocks, b in {32, 64, 128, 256}; "mastering FP8 LLM training 1.5x
speedup", scaling strategy 3, with the 2025 guide's sec. 2.2 rule d = amax /
448 per block) with the oracle: every code byte of both copies, every scale
(in the library's layout) and every counter bit-exact, on seeded inputs with
outliers, zero stripes, subnormal-range values, block-maximum ties, NaN and
Inf, at sizes that span several tiles and blocks with ragged edges."""
import numpy as np
import pytest

import oracle as O
from fp8_scaled_quantization_quantize_gb300 import inputs
from tests._helpers import assert_quant_equal, bits_of, gpu_outputs
from tests.test_quantize_gpu import _mixed

pytestmark = pytest.mark.gpu

BLOCKS = [(1, 32), (1, 64), (1, 128), (1, 256), (32, 32), (64, 64), (128, 128), (256, 256)]
COPIES = [(True, False), (False, True), (True, True)]


def _api():
    from fp8_scaled_quantization_quantize_gb300 import api
    return api


def _check(x, block, fmt, rowwise, colwise, ctx):
    api = _api()
    qt = api.quantize(x.cuda(), O.BLOCK_GENERIC, fmt, rowwise, colwise, block=block)
    got = gpu_outputs(qt)
    ref = O.quantize_generic(fmt, bits_of(x), *block, rowwise, colwise)
    assert_quant_equal(O.BLOCK_GENERIC, got, ref, rowwise, colwise, ctx)
    return got, ref


@pytest.mark.parametrize("block", BLOCKS, ids=[f"{a}x{b}" for a, b in BLOCKS])
@pytest.mark.parametrize("shape", [(272, 400), (400, 1040), (512, 768)])
@pytest.mark.parametrize("fmt", [O.E4M3, O.E5M2])
@pytest.mark.parametrize("copies", COPIES, ids=["row", "col", "both"])
def test_generic_blocks_match_oracle(block, shape, fmt, copies):
    x = _mixed(shape, 300 + shape[0] + block[1])
    _check(x, block, fmt, *copies, f"{block} {shape} fmt={fmt} copies={copies}")


@pytest.mark.parametrize("block", BLOCKS, ids=[f"{a}x{b}" for a, b in BLOCKS])
def test_generic_blocks_special_values(block):
    """NaN of both signs, +-Inf, -0 and bf16 subnormals inside blocks: NaN / Inf
    are counted and left out of the block maxima, NaN keeps its sign, Inf
    saturates."""
    x = inputs.normal_f32((288, 528), 77)
    x[3, 5], x[70, 300], x[200, 17] = np.nan, -np.inf, np.inf
    x[100, :] = -0.0
    x[130:140, 64:96] = np.float32(3e-39)
    xb = inputs.to_bf16(x)
    bits = bits_of(xb).copy()
    bits[9, 9] = 0xFFC1   # a negative NaN with a payload
    import torch
    xb = torch.from_numpy(bits.view(np.int16)).view(torch.bfloat16)
    got, ref = _check(xb, block, O.E4M3, True, True, f"special {block}")
    assert got["nonfinite"] == 4


@pytest.mark.parametrize("block", [(1, 32), (1, 64), (1, 256), (32, 32), (64, 64), (256, 256)],
                         ids=["1x32", "1x64", "1x256", "32x32", "64x64", "256x256"])
def test_generic_blocks_full_size_sweep_tensor(block):
    """A 64 MiB sweep tensor (0.1 % of elements x1000) with every block shape
    that has no specialised kernel (one tile pass for 32 and 64, an amax pass
    first for 256), both copies, every byte."""
    x = inputs.sweep_tensor(64)
    _check(x, block, O.E4M3, True, True, f"sweep {block}")


def test_generic_blocks_invalid_shapes_are_refused():
    from fp8_scaled_quantization_quantize_gb300 import _lib as L
    api = _api()
    import torch
    x = torch.zeros((128, 128), dtype=torch.bfloat16, device="cuda")
    for block in ((2, 64), (64, 32), (1, 16), (512, 512), (1, 96)):
        with pytest.raises(L.Fp8qError) as e:
            api.quantize(x, O.BLOCK_GENERIC, O.E4M3, True, False, block=block)
        assert e.value.status == L.ERR_UNSUPPORTED
    assert api.device_errors() == 0


def test_generic_blocks_in_a_multi_call():
    """fp8q_quantize_multi with generic-block jobs of both kinds of pass (1 x 32
    and 64 x 64 in one tile pass, 1 x 256 and 256 x 256 after their amax pass)
    beside a 1 x 128 job, on streams of their own: every output equals the
    oracle's."""
    import torch
    api = _api()
    specs = [((1, 32), O.E4M3, (400, 1040), True, True),
             ((64, 64), O.E5M2, (336, 528), True, True),
             ((1, 256), O.E4M3, (272, 768), True, True),
             ((256, 256), O.E4M3, (528, 400), False, True)]
    xs = [_mixed(sh, 120 + i) for i, (_, _, sh, _, _) in enumerate(specs)]
    qts = [api.alloc(O.BLOCK_GENERIC, f, *sh, r, c, "cuda", block=b) for b, f, sh, r, c in specs]
    x1 = _mixed((400, 1040), 130)
    q1 = api.alloc(O.BLOCK_1x128, O.E4M3, 400, 1040, True, True, "cuda")
    jobs = [(x.cuda(), q) for x, q in zip(xs, qts)] + [(x1.cuda(), q1)]
    api.quantize_multi(jobs)
    torch.cuda.synchronize()
    for (b, f, sh, r, c), x, q in zip(specs, xs, qts):
        ref = O.quantize_generic(f, bits_of(x), *b, r, c)
        assert_quant_equal(O.BLOCK_GENERIC, gpu_outputs(q), ref, r, c, f"multi generic {b}")
    ref1 = O.quantize(O.BLOCK_1x128, O.E4M3, bits_of(x1), True, True)
    assert_quant_equal(O.BLOCK_1x128, gpu_outputs(q1), ref1, True, True, "multi 1x128")
    assert api.device_errors() == 0
