"""Pins of the oracle's scaled GEMM: brute force on tiny inputs with exact
rational arithmetic (Python fractions, codes decoded by PyTorch's float8 dtypes,
not by the oracle), the operand-swap identity, and the bf16 rounding bound."""
from fractions import Fraction

import numpy as np
import pytest
import torch

import oracle as O

TORCH_DT = {O.E4M3: torch.float8_e4m3fn, O.E5M2: torch.float8_e5m2}


def _finite_codes(rng, shape, fmt, narrow=False):
    table = torch.arange(256, dtype=torch.int32).to(torch.uint8).view(TORCH_DT[fmt]).double().numpy()
    ok = np.isfinite(table)
    if narrow:          # magnitudes in [2^-3, 2^4): keeps exact sums within 53 bits
        ok &= (np.abs(table) >= 2.0 ** -3) & (np.abs(table) < 2.0 ** 4)
    ok = np.flatnonzero(ok)
    return ok[rng.integers(0, ok.size, size=shape)].astype(np.uint8), table


def _exact(A, tabA, sA, a_bm, a_bk, B, tabB, sB, b_bn, b_bk):
    M, K = A.shape
    N = B.shape[0]
    D = np.empty((M, N), dtype=object)
    for m in range(M):
        for n in range(N):
            acc = Fraction(0)
            for k in range(K):
                a = Fraction(float(tabA[A[m, k]])) * Fraction(float(sA[m // a_bm, k // a_bk]))
                b = Fraction(float(tabB[B[n, k]])) * Fraction(float(sB[n // b_bn, k // b_bk]))
                acc += a * b
            D[m, n] = acc
    return D


CASES = [
    # name, (a_bm, a_bk), (b_bn, b_bk): per-tensor, 1x128 x 128x128, 1x128 x 1x128, MX 1x32,
    # per-channel
    ("pertensor", None, None),
    ("block_1d2d", (1, 128), (128, 128)),
    ("block_1d1d", (1, 128), (1, 128)),
    ("mx", (1, 32), (1, 32)),
    ("perchannel", (1, 300), (1, 300)),     # one factor per row of A and of B
]


@pytest.mark.parametrize("name,ab,bb", CASES)
@pytest.mark.parametrize("pow2", [True, False])
def test_tiny_gemm_vs_exact_rationals(name, ab, bb, pow2):
    rng = np.random.default_rng([len(name), int(pow2), sum(map(ord, name))])
    M, N, K = 5, 131, 300                    # K spans partial 32- and 128-blocks
    fmtA, fmtB = (O.E4M3, O.E5M2) if name == "pertensor" else (O.E4M3, O.E4M3)
    A, tabA = _finite_codes(rng, (M, K), fmtA, narrow=pow2)
    B, tabB = _finite_codes(rng, (N, K), fmtB, narrow=pow2)
    a_bm, a_bk = ab if ab else (M, K)
    b_bn, b_bk = bb if bb else (N, K)
    sa_shape = (-(-M // a_bm), -(-K // a_bk))
    sb_shape = (-(-N // b_bn), -(-K // b_bk))
    if pow2:
        sA = np.ldexp(np.float32(1), rng.integers(-3, 4, sa_shape)).astype(np.float32)
        sB = np.ldexp(np.float32(1), rng.integers(-3, 4, sb_shape)).astype(np.float32)
    else:
        sA = rng.uniform(1e-3, 3, sa_shape).astype(np.float32)
        sB = rng.uniform(1e-3, 3, sb_shape).astype(np.float32)
    D = O.gemm_full(A, fmtA, sA, a_bm, a_bk, B, fmtB, sB, b_bn, b_bk)
    E = _exact(A, tabA, sA, a_bm, a_bk, B, tabB, sB, b_bn, b_bk)
    absum = np.array([[sum(abs(Fraction(float(tabA[A[m, k]])) * Fraction(float(tabB[B[n, k]])))
                           for k in range(0, K, 50)) for n in range(N)] for m in range(M)], dtype=object)
    for m in range(M):
        for n in range(N):
            if pow2:
                # power-of-two scales in 2^[-3, 3], codes in [2^-3, 2^4): every
                # product is a multiple of 2^-19 below 2^14, the sum of 300 stays
                # below 2^23, so fp64 holds every partial sum exactly
                assert Fraction(D[m, n]) == E[m, n], (m, n)
            else:
                err = abs(Fraction(D[m, n]) - E[m, n])
                assert err <= Fraction(2 ** -40) * (abs(E[m, n]) + 1 + absum[m, n] * 50)


def test_operand_swap_is_transpose():
    rng = np.random.default_rng(1)
    A, _ = _finite_codes(rng, (17, 96), O.E4M3)
    B, _ = _finite_codes(rng, (23, 96), O.E4M3)
    sA = rng.uniform(0.5, 2, (17, 3)).astype(np.float32)
    sB = rng.uniform(0.5, 2, (23, 3)).astype(np.float32)
    D1 = O.gemm_full(A, O.E4M3, sA, 1, 32, B, O.E4M3, sB, 1, 32)
    D2 = O.gemm_full(B, O.E4M3, sB, 1, 32, A, O.E4M3, sA, 1, 32)
    assert np.array_equal(D1, D2.T)


def test_bf16_output_rounding_is_within_normwise_bound():
    rng = np.random.default_rng(2)
    A, _ = _finite_codes(rng, (64, 256), O.E4M3)
    B, _ = _finite_codes(rng, (64, 256), O.E4M3)
    s = np.ones((1, 1), dtype=np.float32)
    D = O.gemm_full(A, O.E4M3, s, 64, 256, B, O.E4M3, s, 64, 256)
    Db = O.bf16_to_f32(O.f64_to_bf16(D)).astype(np.float64)
    rel = np.linalg.norm(Db - D) / np.linalg.norm(D)
    # round-to-nearest to 8 significant bits: relative error <= 2^-8 per element
    assert np.all(np.abs(Db - D) <= np.abs(D) * 2.0 ** -8)
    assert rel < 2e-3


def test_gemm_points_at_scattered_points():
    """The point-wise entry (what the full-size parity tests sample) at
    out-of-order and repeated output points, with 128x128 tiles on B and 1x128
    blocks on A at a ragged M, N, K: each point equals the exact rational sum
    of its own row of A and row of B."""
    rng = np.random.default_rng(31)
    M, N, K = 9, 260, 300
    A, tabA = _finite_codes(rng, (M, K), O.E4M3, narrow=True)
    B, tabB = _finite_codes(rng, (N, K), O.E4M3, narrow=True)
    sA = np.ldexp(np.float32(1), rng.integers(-3, 4, (M, 3))).astype(np.float32)
    sB = np.ldexp(np.float32(1), rng.integers(-3, 4, (3, 3))).astype(np.float32)
    pm = rng.integers(0, M, 200)
    pn = rng.integers(0, N, 200)
    pm[:3], pn[:3] = [M - 1, 0, M - 1], [N - 1, N - 1, N - 1]     # corners, one repeated
    got = O.gemm_points(A, O.E4M3, sA, 1, 128, B, O.E4M3, sB, 128, 128, pm, pn)
    for i, (m, n) in enumerate(zip(pm, pn)):
        acc = Fraction(0)
        for k in range(K):
            acc += (Fraction(float(tabA[A[m, k]])) * Fraction(float(sA[m, k // 128]))
                    * Fraction(float(tabB[B[n, k]])) * Fraction(float(sB[n // 128, k // 128])))
        assert Fraction(got[i]) == acc, (i, m, n)
