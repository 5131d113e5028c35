"""Pins of the oracle's recipes (per-tensor current / delayed, blockwise 1x128 /
128x128, MXFP8 1x32) against hand-worked blocks, closed forms, invariants and
independent restatements, plus its scale layouts."""
import os

import numpy as np
import pytest
import torch

import oracle as O
from fp8_scaled_quantization_quantize_gb300 import inputs

GOLD = os.path.join(os.path.dirname(__file__), "golden")


def _bits(x: np.ndarray) -> np.ndarray:
    return inputs.bf16_bits(torch.from_numpy(np.asarray(x, dtype=np.float32)).to(torch.bfloat16))


def _k32_table():
    tab = {}
    with open(os.path.join(GOLD, "block_k_times_32.txt")) as f:
        for line in f:
            if line.strip() and not line.startswith("#"):
                k, code = line.split()[:2]
                tab[int(k)] = int(code, 16)
    assert len(tab) == 15
    return tab


def _k32_expected(ks):
    tab = _k32_table()
    return np.array([tab[abs(k)] | (0x80 if k < 0 else 0) for k in ks], dtype=np.uint8)


def test_hand_block_1x128():
    ks = np.array([(i % 29) - 14 for i in range(128)])
    q, d, _, am, sat, nf = O.quant_blocks(_bits(ks[None, :]), 1, 128, O.KIND_DIV, O.E4M3)
    assert am[0, 0] == 14.0 and d[0, 0] == np.float32(2.0 ** -5)
    assert np.array_equal(q[0], _k32_expected(ks)) and sat == 0 and nf == 0


def test_hand_block_128x128():
    ks = np.array([[((r * 7 + c) % 29) - 14 for c in range(128)] for r in range(128)])
    q, d, _, am, sat, nf = O.quant_blocks(_bits(ks), 128, 128, O.KIND_DIV, O.E4M3)
    assert d.shape == (1, 1) and d[0, 0] == np.float32(2.0 ** -5)
    assert np.array_equal(q, _k32_expected(ks.ravel()).reshape(128, 128))


def test_hand_block_mx():
    ks = np.array([(i % 29) - 14 for i in range(32)])
    q, sc, e8, am, sat, nf = O.quant_blocks(_bits(ks[None, :]), 1, 32, O.KIND_POW2, O.E4M3)
    assert e8[0, 0] == 122 and sc[0, 0] == np.float32(2.0 ** -5)
    assert np.array_equal(q[0], _k32_expected(ks))


def test_hand_block_pertensor():
    ks = np.array([[((r + 3 * c) % 29) - 14 for c in range(40)] for r in range(9)])
    res = O.quantize(O.PERTENSOR_CURRENT, O.E4M3, _bits(ks), True, True)
    assert res["scale"] == np.float32(32.0) and res["scale_inv"] == np.float32(1 / 32)
    assert res["amax"] == 14.0
    exp = _k32_expected(ks.ravel()).reshape(ks.shape)
    assert np.array_equal(res["data_row"], exp)
    assert np.array_equal(res["data_col"], exp.T)


def _k4096_e5m2_expected(ks):
    tab = {}
    with open(os.path.join(GOLD, "block_k_times_4096_e5m2.txt")) as f:
        for line in f:
            if line.strip() and not line.startswith("#"):
                k, code = line.split()[:2]
                tab[int(k)] = int(code, 16)
    assert len(tab) == 15
    return np.array([tab[abs(k)] | (0x80 if k < 0 else 0) for k in ks], dtype=np.uint8)


def test_hand_block_e5m2_all_recipes():
    """The same block in E5M2: 1x128 and 128x128 (d = 2^-12), MX (E8M0 115)
    and per-tensor (s = 4096) all cast 4096 k, three of them ties."""
    ks = np.array([(i % 29) - 14 for i in range(128)])
    exp = _k4096_e5m2_expected(ks)
    for br, bc in ((1, 128), (128, 128)):
        q, d, _, am, sat, nf = O.quant_blocks(_bits(ks[None, :]), br, bc, O.KIND_DIV, O.E5M2)
        assert d[0, 0] == np.float32(2.0 ** -12) and am[0, 0] == 14.0
        assert np.array_equal(q[0], exp) and sat == 0 and nf == 0
    q, sc, e8, am, sat, nf = O.quant_blocks(_bits(ks[None, :]), 1, 32, O.KIND_POW2, O.E5M2)
    assert e8.shape == (1, 4) and np.all(e8 == 115) and np.array_equal(q[0], exp) and sat == 0
    res = O.quantize(O.PERTENSOR_CURRENT, O.E5M2, _bits(ks[None, :]), True, False)
    assert res["scale"] == np.float32(4096.0) and res["scale_inv"] == np.float32(2.0 ** -12)
    assert np.array_equal(res["data_row"][0], exp) and res["sat_row"] == 0


def test_hand_perchannel():
    """Rows k, 2k, k/2 of k = (c % 29) - 14: row maxima 14, 28, 7 give s = 32,
    16, 64 (RN(448 / amax), exact) and every row the codes of k x 32.  Column
    c holds k, 2k, k/2 with maximum 2|k|: s = 224 / |k| maps the rows to
    +-224, +-448, +-112 (E4M3 0x76, 0x7E, 0x6E); all-zero columns keep s = 1."""
    k = np.array([(c % 29) - 14 for c in range(48)], dtype=np.float64)
    x = np.stack([k, 2 * k, k / 2])
    res = O.quantize(O.PERCHANNEL_CURRENT, O.E4M3, _bits(x), True, True)
    assert list(res["mult_row"]) == [32.0, 16.0, 64.0]
    assert list(res["scale_row"]) == [np.float32(1 / 32), np.float32(1 / 16), np.float32(1 / 64)]
    exp = _k32_expected(k.astype(int))
    for r in range(3):
        assert np.array_equal(res["data_row"][r], exp)
    mag = {0: 0x76, 1: 0x7E, 2: 0x6E}
    for c in range(48):
        kc = int(k[c])
        if kc == 0:
            assert res["mult_col"][c] == 1.0 and not res["data_col"][c].any()
            continue
        assert res["mult_col"][c] == np.float32(448.0 / (2 * abs(kc)))
        sign = 0x80 if kc < 0 else 0
        assert list(res["data_col"][c]) == [mag[r] | sign for r in range(3)], c
    # saturated before the cast: where RN(224 / |k|) rounded up, 2|k| s lands
    # just above 448 (and still encodes to 448)
    s32 = np.float32(448.0) / np.float32(2 * np.abs(k[k != 0]))
    over = int(np.count_nonzero(np.float32(2 * np.abs(k[k != 0])) * s32 > np.float32(448.0)))
    assert res["sat_row"] == 0 and res["sat_col"] == over and res["nonfinite"] == 0
    assert res["scale_row_packed"].size == 128 and np.all(res["scale_row_packed"][3:] == 1.0)


def test_perchannel_rows_are_pertensor():
    """Each row of a per-channel copy is the per-tensor current quantization of
    that row alone: codes, multiplier, dequantization factor, saturation."""
    x = _rand_bits((37, 208), 11)
    x[5, 7] = 0x7F80                   # an Inf in one row: excluded from its amax, counted
    res = O.quantize(O.PERCHANNEL_CURRENT, O.E5M2, x, True, False)
    sat = 0
    for r in range(37):
        one = O.quantize(O.PERTENSOR_CURRENT, O.E5M2, x[r:r + 1], True, False)
        assert np.array_equal(res["data_row"][r], one["data_row"][0]), r
        assert res["mult_row"][r] == one["scale"] and res["scale_row"][r] == one["scale_inv"]
        assert res["amax_row"][r] == one["amax"]
        sat += one["sat_row"]
    assert res["sat_row"] == sat and res["nonfinite"] == 1


def test_e8m0_closed_form():
    fmts = {"e4m3": O.E4M3, "e5m2": O.E5M2}
    n = 0
    with open(os.path.join(GOLD, "e8m0_closed_form.txt")) as f:
        for line in f:
            if not line.strip() or line.startswith("#"):
                continue
            fmt, amax, e, code = line.split()[:4]
            a = np.float32(float.fromhex(amax))
            got = O.mx_exponent(a, fmts[fmt])
            assert got == int(e) and got + 127 == int(code), line
            n += 1
    assert n >= 10


def test_scale_rule_special_cases():
    # amax 0: neutral scales
    assert O.pertensor_scale(0.0, O.E4M3) == 1.0
    assert O.block_scale(0.0, O.E4M3) == 1.0
    assert O.mx_exponent(0.0, O.E4M3) == 0
    # tiny amax: 448 / 2^-133 overflows fp32 and clamps to FLT_MAX
    assert O.pertensor_scale(np.float32(2.0 ** -133), O.E4M3) == np.finfo(np.float32).max
    # d underflowing to 0 becomes the smallest subnormal 2^-149
    assert O.block_scale(np.float32(2.0 ** -149), O.E4M3) == np.float32(2.0 ** -149)
    # ordinary cases are single IEEE fp32 divisions
    assert O.pertensor_scale(np.float32(3.0), O.E4M3) == np.float32(448.0) / np.float32(3.0)
    assert O.block_scale(np.float32(3.0), O.E5M2) == np.float32(3.0) / np.float32(57344.0)


def _rand_bits(shape, seed, outliers=True):
    x = inputs.normal_f32(shape, seed)
    if outliers:
        x = inputs.with_outlier_elements(x, 0.01, 1000.0, seed + 1)
    return _bits(x)


# code of the largest finite magnitude: E4M3 0.1111.110 = 448, E5M2 0.11110.11 = 57344
FMAX_CODE = {O.E4M3: 0x7E, O.E5M2: 0x7B}


@pytest.mark.parametrize("fmt", [O.E4M3, O.E5M2])
@pytest.mark.parametrize("br,bc", [(1, 128), (128, 128), (1, 64), (64, 64), (32, 32), (1, 256), (256, 256)])
def test_blockwise_block_max_hits_fmax(br, bc, fmt):
    x = _rand_bits((300, 390), 1)
    q, d, _, am, sat, nf = O.quant_blocks(x, br, bc, O.KIND_DIV, fmt)
    xf = np.abs(O.bf16_to_f32(x))
    for bi in range(am.shape[0]):
        for bj in range(am.shape[1]):
            blk = xf[bi * br:(bi + 1) * br, bj * bc:(bj + 1) * bc]
            qb = q[bi * br:(bi + 1) * br, bj * bc:(bj + 1) * bc]
            assert am[bi, bj] == blk.max()
            assert np.all((qb[blk == blk.max()] & 0x7F) == FMAX_CODE[fmt])
            assert np.all((qb & 0x7F) <= FMAX_CODE[fmt])


@pytest.mark.parametrize("fmt,emax,top_lo", [(O.E4M3, 8, 0x78), (O.E5M2, 15, 0x78)])
def test_mx_scaled_block_max_in_top_binade(fmt, emax, top_lo):
    """e = floor(log2 amax) - emax puts the scaled block maximum in
    [2^(emax), 2^(emax + 1)): E4M3 [256, 512) (codes 0x78 = 256 .. 0x7E = 448,
    saturating above), E5M2 [32768, 65536) (0x78 = 32768 .. 0x7B = 57344)."""
    x = _rand_bits((64, 320), 2)
    q, sc, e8, am, sat, nf = O.quant_blocks(x, 1, 32, O.KIND_POW2, fmt)
    for r in range(64):
        for b in range(10):
            e = int(e8[r, b]) - 127
            scaled = float(am[r, b]) * 2.0 ** -e
            assert 2.0 ** emax <= scaled < 2.0 ** (emax + 1)
            top = (q[r, b * 32:(b + 1) * 32] & 0x7F).max()
            assert top_lo <= top <= FMAX_CODE[fmt]


@pytest.mark.parametrize("fmt", [O.E4M3, O.E5M2])
def test_pertensor_amax_maps_to_fmax(fmt):
    x = _rand_bits((200, 160), 3)
    res = O.quantize(O.PERTENSOR_CURRENT, fmt, x, True, False)
    xf = np.abs(O.bf16_to_f32(x))
    assert res["amax"] == xf.max()
    assert np.all((res["data_row"][xf == xf.max()] & 0x7F) == FMAX_CODE[fmt])


@pytest.mark.parametrize("kind", [O.BLOCK_1x128, O.MXFP8_1x32, O.PERCHANNEL_CURRENT])
def test_colwise_is_rowwise_of_transpose(kind):
    x = _rand_bits((200, 176), 4)
    res = O.quantize(kind, O.E4M3, x, True, True)
    tr = O.quantize(kind, O.E4M3, np.ascontiguousarray(x.T), True, False)
    assert np.array_equal(res["data_col"], tr["data_row"])
    assert np.array_equal(res["scale_col"], tr["scale_row"])
    assert res["sat_col"] == tr["sat_row"]


@pytest.mark.parametrize("br,bc,kind", [(1, 128, O.KIND_DIV), (128, 128, O.KIND_DIV), (1, 32, O.KIND_POW2),
                                        (32, 1, O.KIND_POW2), (128, 1, O.KIND_DIV), (1, 64, O.KIND_DIV),
                                        (64, 64, O.KIND_DIV), (256, 256, O.KIND_DIV)])
def test_ragged_edges_equal_zero_padding(br, bc, kind):
    """A partial edge block takes the elements present: zero padding to full
    blocks (zeros never change an amax) must give the same codes and scales."""
    x = _rand_bits((133, 272), 5)
    q, s, e8, am, *_ = O.quant_blocks(x, br, bc, kind, O.E4M3)
    R = -(-133 // br) * br
    C = -(-272 // bc) * bc
    xp = np.zeros((R, C), dtype=np.uint16)
    xp[:133, :272] = x
    qp, sp, e8p, amp, *_ = O.quant_blocks(xp, br, bc, kind, O.E4M3)
    assert np.array_equal(q, qp[:133, :272])
    assert np.array_equal(s, sp) and np.array_equal(am, amp)


@pytest.mark.parametrize("br,bc,kind", [(1, 128, O.KIND_DIV), (64, 64, O.KIND_DIV), (32, 128, O.KIND_DIV),
                                        (1, 32, O.KIND_POW2), (1, 256, O.KIND_MULT)])
def test_block_shape_transposes_with_the_matrix(br, bc, kind):
    """Generic sub-channel blocks: quantizing x^T with br x bc blocks gives the
    transpose of quantizing x with bc x br blocks (codes, scales, maxima), so
    no row / column index is swapped anywhere in the block loop."""
    x = _rand_bits((200, 330), 21)
    xt = np.ascontiguousarray(x.T)
    q, sc, _, am, sat, nf = O.quant_blocks(x, bc, br, kind, O.E4M3)
    qt, sct, _, amt, satt, nft = O.quant_blocks(xt, br, bc, kind, O.E4M3)
    assert np.array_equal(qt, q.T) and np.array_equal(sct, sc.T) and np.array_equal(amt, am.T)
    assert (satt, nft) == (sat, nf)


def test_nonfinite_inputs():
    x = _bits(np.array([[1.0, 0.0, np.inf, -np.inf, -2.0, 0.5] + [0.25] * 26], dtype=np.float32))
    x[0, 1] = 0x7FC0          # +NaN (torch's own float->bf16 cast yields 0xFFFF)
    for br, bc, kind in [(1, 32, O.KIND_POW2), (1, 128, O.KIND_DIV), (1, 32, O.KIND_MULT)]:
        q, s, e8, am, sat, nf = O.quant_blocks(x, br, bc, kind, O.E4M3)
        assert nf == 3 and am[0, 0] == 2.0
        assert q[0, 1] == 0x7F and q[0, 2] == 0x7E and q[0, 3] == 0xFE
    x[0, 1] = 0xFFC0          # -NaN keeps its sign
    q, *_ = O.quant_blocks(x, 1, 32, O.KIND_POW2, O.E4M3)
    assert q[0, 1] == 0xFF


def test_delayed_trace_golden():
    st = O.Delayed(16, O.E4M3, 0)
    n = 0
    with open(os.path.join(GOLD, "delayed_trace.txt")) as f:
        for line in f:
            if not line.strip() or line.startswith("#"):
                continue
            t, a, nan, s, code, nsat = line.split()[:6]
            a = float(a)
            row = np.zeros((1, 64), dtype=np.float32)
            row[0, 0], row[0, 1] = a, -a / 2
            if int(nan):
                row[0, 7] = np.nan
            assert st.scale == np.float32(float(s)), (t, st.scale)
            res = O.quantize(O.PERTENSOR_DELAYED, O.E4M3, _bits(row), True, False, state=st)
            assert res["scale"] == np.float32(float(s))
            assert res["data_row"][0, 0] == int(code, 16)
            assert res["sat_row"] == int(nsat) and res["nonfinite"] == int(nan)
            n += 1
    assert n == 32


def test_delayed_spike_leaves_after_history_length():
    st = O.Delayed(16, O.E4M3, 0)
    scales = []
    for t in range(40):
        scales.append(float(st.scale))
        st.update(100.0 if t == 3 else 1.0)
    # the spike recorded at step 3 governs the scales of steps 4 .. 19
    assert all(s == np.float32(4.48) for s in scales[4:20])
    assert all(s == 448.0 for s in scales[20:])
    assert np.all(np.diff(scales[4:20]) == 0)


def test_delayed_margin():
    """Margins worked by hand: E4M3, margin 1, amax 7: 448 / 7 = 64 exactly,
    times 2^-1 gives s = 32, and x = 7 scales to 224 = 1.75 * 2^7, the E4M3
    code 0 1110 110 = 0x76.  E5M2, margin 2, amax 7: 57344 / 7 = 8192 exactly,
    s = 2048 = 2^11, scale_inv = 2^-11."""
    st = O.Delayed(4, O.E4M3, 1)
    st.update(7.0)
    assert st.scale == 32.0 and st.scale_inv == 1.0 / 32.0
    q, amax, sat, nf = O.cast_scaled(np.array([0x40E0, 0xC0E0], dtype=np.uint16), st.scale, O.E4M3)  # +-7.0
    assert list(q) == [0x76, 0xF6] and amax == 7.0 and sat == 0 and nf == 0
    st5 = O.Delayed(4, O.E5M2, 2)
    st5.update(7.0)
    assert st5.scale == 2048.0 and st5.scale_inv == 2.0 ** -11


def test_delayed_margin_underflow_is_clamped():
    """A margin large enough to push s below the normal fp32 range (margin
    64 with history max 2^127: 448 / 2^127 * 2^-64 = 1.75 * 2^-183, below the
    smallest subnormal) raises s to the smallest normal, 2^-126, so scale_inv
    = 2^126 stays finite; a subnormal product (margin 20: 1.75 * 2^-139) is
    raised the same way, and margin 5 on amax 2^120 (s = 1.75 * 2^(8 - 120 - 5) = 1.75 * 2^-117, a
    normal number) is left alone."""
    for margin, amax, want in ((64, 2.0 ** 127, 2.0 ** -126), (20, 2.0 ** 127, 2.0 ** -126),
                               (5, 2.0 ** 120, 1.75 * 2.0 ** -117)):
        st = O.Delayed(16, O.E4M3, margin)
        st.update(amax)
        assert st.scale == np.float32(want), (margin, st.scale)
        assert np.isfinite(st.scale_inv) and st.scale_inv == np.float32(1.0 / want)


def test_pack_mx_positions_and_padding():
    R, S = 130, 6
    codes = np.arange(R * S, dtype=np.int64).reshape(R, S) % 251
    p = O.pack_mx(codes.astype(np.uint8))
    assert p.size == 2 * 2 * 512
    # row 33, scale column 2 -> tile 0, byte (33 % 32) * 16 + (33 // 32) * 4 + 2
    assert p[1 * 16 + 1 * 4 + 2] == codes[33, 2]
    # row 129, column 5 -> tile (1, 1) = 3, byte 1 * 16 + 0 * 4 + 1
    assert p[3 * 512 + 16 + 1] == codes[129, 5]
    # padding: columns 6, 7 and rows 130..255 hold 127
    assert p[0 * 512 + 1 * 512 + 0 * 16 + 0 * 4 + 2] == 127
    assert p[2 * 512 + 5 * 16] == 127
    # every code appears once in the packed buffer outside the padding
    assert (p != 127).sum() == (codes != 127).sum()


def test_pack_block1x128_positions():
    d = np.arange(3 * 5, dtype=np.float32).reshape(3, 5) + 2
    p = O.pack_block1x128(d)
    assert p.shape == (5, 128)
    assert p[4, 2] == d[2, 4] and p[0, 1] == d[1, 0]
    assert np.all(p[:, 3:] == 1.0)


def test_amax_sat_matches_cast_scaled():
    x = _rand_bits((64, 96), 8)
    x[3, 4] = 0x7F80      # +Inf
    x[5, 6] = 0xFFC1      # -NaN
    for s in (np.float32(3.0), np.float32(448.0 / 7.0), np.float32(1e4)):
        for fmt in (O.E4M3, O.E5M2):
            q, amax, sat, nf = O.cast_scaled(x, s, fmt)
            assert O.amax_sat(x, s, fmt) == (amax, sat, nf)


def test_generic_128_blocks_are_the_specialised_recipes():
    """The generic sub-channel recipe at 1 x 128 and 128 x 128 is exactly the
    guide's sec. 2.2 recipes (codes, packed scales, counters), and its square
    blocks' column copy is the transpose of the row copy."""
    x = _rand_bits((272, 400), 41)
    for (br, bc), kind in (((1, 128), O.BLOCK_1x128), ((128, 128), O.BLOCK_128x128)):
        g = O.quantize_generic(O.E4M3, x, br, bc, True, True)
        s = O.quantize(kind, O.E4M3, x, True, True)
        for key in ("data_row", "data_col", "sat_row", "sat_col", "nonfinite"):
            assert np.array_equal(g[key], s[key]), (kind, key)
        for which in ("row", "col"):
            sp = s.get("scale_" + which + "_packed", s["scale_" + which])
            assert np.array_equal(g["scale_" + which + "_packed"], sp), (kind, which)
    g = O.quantize_generic(O.E5M2, x, 64, 64, True, True)
    assert np.array_equal(g["data_col"], g["data_row"].T) and np.array_equal(g["scale_col"], g["scale_row"].T)
