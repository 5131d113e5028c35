"""Per-tensor delayed scaling at a Llama-3-70B FFN layer (tokens 4096, hidden
8192, ffn 28672), hybrid formats (E4M3 for X and W, E5M2 for dY), history 16,
32 steps of a lognormal magnitude walk with a x50 spike at step 20
("2025 FP8 quantized-training guide", sec. 2.1 delayed scaling from an amax
history; the bjdmk.com.cn FP8 essay, sec. 3.3 DelayedScaling(margin=0,
interval=1)).

Every step, through the C ABI:
- X, W and dY quantized with both copies: every code byte of the row-wise and
  column-wise copies equals the oracle's; amax, scale, scale_inv, saturation
  and nonfinite counts and the delayed state (history, head, next scale)
  equal the oracle's state machine;
- the three GEMMs of the layer on those FP8 operands -- fprop Y = X W^T,
  dgrad dX = dY W (dY's row copy with W's column copy, E5M2 x E4M3) and
  wgrad dW = dY^T X (the two column copies) -- bf16 output, against the fp64
  oracle on the same quantized operands: rows {0, last, 6 seeded} x every
  column and every row x columns {0, last, 6 seeded} (254 seeded at the
  first step and at the spike's step 20: 256 rows and 256 columns),
  normwise relative error <= 2e-3 on each of the 3 x 32 GEMMs.

The oracle's codes come from the oracle alone: per step and tensor the
oracle encodes every one of the 65536 bf16 bit patterns at the step's scale
(the cast rule q = encode(fp32(x) * s) is the same function of x for every
element), and the tensor's codes are that table looked up at its bits.
"""
import numpy as np
import pytest
import torch

import oracle as O
from fp8_scaled_quantization_quantize_gb300 import inputs
from tests._helpers import bits_of, gpu_outputs

pytestmark = pytest.mark.gpu

TOKENS, HIDDEN, FFN = 4096, 8192, 28672
FMTS = (O.E4M3, O.E4M3, O.E5M2)      # X, W, dY
ALL_BITS = np.arange(65536, dtype=np.uint16)


def _samples(n: int, rng, k: int = 6) -> np.ndarray:
    """{0, n - 1} and k seeded indices in between."""
    return np.unique(np.concatenate([[0, n - 1], rng.choice(np.arange(1, n - 1), k, replace=False)]))


def _gemm_rel(D: torch.Tensor, A, fa, sa, B, fb, sb, rng, k: int = 6) -> float:
    """Normwise relative error of the GPU D = A . B^T (bf16) against the fp64
    oracle over the sampled rows x all columns and all rows x sampled columns."""
    M, N = D.shape
    rows, cols = _samples(M, rng, k), _samples(N, rng, k)
    pm = np.concatenate([np.repeat(rows, N), np.tile(np.arange(M), cols.size)])
    pn = np.concatenate([np.tile(np.arange(N), rows.size), np.repeat(cols, M)])
    K = A.shape[1]
    ref = O.gemm_points(A, fa, np.array([[sa]], np.float32), M, K, B, fb, np.array([[sb]], np.float32), N, K, pm, pn)
    got = np.concatenate([D[torch.from_numpy(rows).cuda()].float().cpu().numpy().ravel(),
                          D[:, torch.from_numpy(cols).cuda()].float().t().cpu().numpy().ravel()]).astype(np.float64)
    return float(np.linalg.norm(got - ref) / np.linalg.norm(ref))


def test_delayed_llama70b_32_steps_codes_and_gemms():
    from fp8_scaled_quantization_quantize_gb300 import api
    O.set_threads(0)
    mags = inputs.delayed_magnitudes(32)
    bases = inputs.llama70b_ffn_bases(TOKENS, HIDDEN, FFN)
    states = [api.DelayedState(16, f, 0) for f in FMTS]
    ostates = [O.Delayed(16, f, 0) for f in FMTS]
    rng = np.random.default_rng(70)
    Y = torch.empty((TOKENS, FFN), dtype=torch.bfloat16, device="cuda")
    dX = torch.empty((TOKENS, HIDDEN), dtype=torch.bfloat16, device="cuda")
    dW = torch.empty((FFN, HIDDEN), dtype=torch.bfloat16, device="cuda")
    worst = 0.0
    for t in range(32):
        xs = inputs.llama70b_ffn_step(t, bases, mags)
        qts, codes, sinv = [], [], []
        for i, x in enumerate(xs):
            ctx = f"step {t} tensor {i}"
            s = ostates[i].scale
            qt = api.quantize(x.cuda(), O.PERTENSOR_DELAYED, FMTS[i], True, True, state=states[i])
            got = gpu_outputs(qt)
            bits = bits_of(x)
            table = O.cast_scaled(ALL_BITS, s, FMTS[i])[0]
            q = table[bits]
            assert np.array_equal(got["data_row"], q), ctx
            assert np.array_equal(got["data_col"], q.T), ctx
            amax, sat, nf = O.amax_sat(bits, s, FMTS[i])
            assert got["scale"] == s and got["scale_inv"] == np.float32(np.float32(1) / s), ctx
            assert np.float32(got["amax"]) == np.float32(amax), ctx
            assert got["sat_row"] == sat and got["sat_col"] == 0 and got["nonfinite"] == nf, ctx
            codes.append(q)
            sinv.append(np.float32(np.float32(1) / s))
            ostates[i].update(amax, nf)
            hist, head, sc, _ = states[i].get()
            assert np.float32(sc) == ostates[i].scale and head == ostates[i].head, ctx
            assert np.array_equal(np.float32(hist), ostates[i].hist), ctx
            qts.append(qt)
        qx, qw, qdy = qts
        cx, cw, cdy = codes
        api.scaled_gemm(qx, False, qw, False, out=Y)         # fprop: X . W^T
        api.scaled_gemm(qdy, False, qw, True, out=dX)        # dgrad: dY . W
        api.scaled_gemm(qdy, True, qx, True, out=dW)         # wgrad: dY^T . X
        torch.cuda.synchronize()
        k = 254 if t in (0, 20) else 6
        rels = (_gemm_rel(Y, cx, FMTS[0], sinv[0], cw, FMTS[1], sinv[1], rng, k),
                _gemm_rel(dX, cdy, FMTS[2], sinv[2], np.ascontiguousarray(cw.T), FMTS[1], sinv[1], rng, k),
                _gemm_rel(dW, np.ascontiguousarray(cdy.T), FMTS[2], sinv[2], np.ascontiguousarray(cx.T), FMTS[0],
                          sinv[0], rng, k))
        for name, rel in zip(("fprop", "dgrad", "wgrad"), rels):
            assert rel <= 2e-3, f"step {t} {name}: normwise relative error {rel:.3e}"
        worst = max(worst, *rels)
        if t == 20:   # the spike pulls the next scales of X and W below 448
            assert any(ostates[i].scale < np.float32(448.0) for i in range(2))
    assert api.device_errors() == 0
    print(f"delayed Llama-3-70B: 32 steps, worst GEMM normwise relative error {worst:.3e}")
