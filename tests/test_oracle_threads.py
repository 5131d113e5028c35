"""The oracle's OpenMP loops only split independent blocks, elements and GEMM
output points across host threads, and combine across threads only maxima
and counts: every output is the same on one thread and on several (so the
single-core timing leg and the all-core leg time the same computation)."""
import numpy as np

import oracle as O
from fp8_scaled_quantization_quantize_gb300 import inputs


def _same(a, b):
    """Equal bit for bit (arrays) or equal (scalars)."""
    if isinstance(a, np.ndarray):
        return a.shape == b.shape and a.dtype == b.dtype and a.tobytes() == b.tobytes()
    return a == b


def test_thread_count_does_not_change_results():
    x = inputs.with_outlier_elements(inputs.normal_f32((272, 400), 31), 0.01, 1000.0, 32)
    x[5, 7] = np.nan
    x[9, 100] = -np.inf
    bits = inputs.bf16_bits(inputs.to_bf16(x))
    prev = O.set_threads(0)
    try:
        runs = []
        for th in (1, 4):
            O.set_threads(th)
            outs = {k: O.quantize(k, O.E4M3, bits, True, True)
                    for k in (O.PERTENSOR_CURRENT, O.BLOCK_1x128, O.BLOCK_128x128, O.MXFP8_1x32,
                              O.PERCHANNEL_CURRENT)}
            q = outs[O.BLOCK_1x128]
            s, bm, bk = O.dequant_scales(O.BLOCK_1x128, q, "row", 272, 400)
            pm, pn = np.arange(272).repeat(3), np.tile([0, 199, 271], 272)
            g = O.gemm_points(q["data_row"], O.E4M3, s, bm, bk, q["data_row"], O.E4M3, s, bm, bk, pm, pn)
            c = O.cast_scaled(bits, np.float32(3.5), O.E5M2)
            a = O.amax_sat(bits, np.float32(3.5), O.E5M2)
            runs.append((outs, g, c, a))
        (o1, g1, c1, a1), (o4, g4, c4, a4) = runs
        for k in o1:
            assert o1[k].keys() == o4[k].keys()
            for key in o1[k]:
                assert _same(o1[k][key], o4[k][key]), (k, key)
        assert np.array_equal(g1.view(np.uint64), g4.view(np.uint64))
        assert np.array_equal(c1[0], c4[0]) and c1[1:] == c4[1:]
        assert a1 == a4
    finally:
        O.set_threads(prev)
