"""The blockwise recipes divide by d = amax / fmax ("2025 FP8 quantized-training
guide", sec. 2.2) through a correctly rounded reciprocal plus one FMA residual
correction.  This checks that shortcut against IEEE division over its whole
reachable domain and beyond: every finite bf16 x against every d = RN(a / fmax)
for every positive finite bf16 a (the only divisors a bf16 tensor can
produce), both formats, plus random fp32 divisors, for every pair whose
quotient is below 2^126 (quantization's quotients never exceed
fmax (1 + 2^-23), since it divides |x| <= amax by RN(amax / fmax)).  FP8
codes must agree for all of them, fp32 bits wherever the quotient is at
least 2^-24 (below that, where the residual of a tiny x can leave fp32's
normal range, every quotient encodes to an FP8 zero)."""
import numpy as np
import pytest
import torch

pytestmark = pytest.mark.gpu


@pytest.mark.parametrize("fmt,fmax", [(0, 448.0), (1, 57344.0)])
def test_division_shortcut_exhaustive(fmt, fmax):
    from fp8_scaled_quantization_quantize_gb300 import api
    a = (np.arange(1, 0x7F80, dtype=np.uint32) << 16).view(np.float32)    # positive finite bf16
    d = (a / np.float32(fmax)).astype(np.float32)
    d = d[d > 0]
    rng = np.random.default_rng(9)
    extra = np.exp2(rng.uniform(-80, 127, 20000)).astype(np.float32) * rng.uniform(1, 2, 20000).astype(np.float32)
    d = np.concatenate([d, extra[np.isfinite(extra)]])
    codes, bits = api.selftest_division(torch.from_numpy(d).cuda(), fmt)
    assert codes == 0 and bits == 0, (codes, bits)
