"""Pins of the oracle's FP8 / bf16 format code against things other than itself:
hand-derived values, the closed forms of the formats, PyTorch's float8 dtypes
(named by the "2025 FP8 quantized-training guide", sec. 1.1), and brute-force
nearest-value search."""
import os

import numpy as np
import pytest
import torch

import oracle as O

GOLD = os.path.join(os.path.dirname(__file__), "golden")
FMT = {"e4m3": O.E4M3, "e5m2": O.E5M2}
TORCH_DT = {O.E4M3: torch.float8_e4m3fn, O.E5M2: torch.float8_e5m2}


def _parse_value(s: str) -> np.float32:
    if s in ("nan", "inf", "-inf"):
        return np.float32(float(s))
    return np.float32(float.fromhex(s))


def _torch_decode(fmt):
    codes = torch.arange(256, dtype=torch.int32).to(torch.uint8)
    return codes.view(TORCH_DT[fmt]).to(torch.float64).numpy()


@pytest.mark.parametrize("fmt", [O.E4M3, O.E5M2])
def test_decode_matches_torch_dtype(fmt):
    ours = O.decode(np.arange(256), fmt)
    ref = _torch_decode(fmt)
    assert np.array_equal(np.isnan(ours), np.isnan(ref))
    ok = ~np.isnan(ref)
    assert np.array_equal(ours[ok], ref[ok])


def test_decode_closed_forms():
    e4 = O.decode(np.arange(256), O.E4M3)
    e5 = O.decode(np.arange(256), O.E5M2)
    assert np.nanmax(e4) == 1.75 * 2 ** 8 == 448.0
    assert np.nanmax(e5[np.isfinite(e5)]) == 1.75 * 2 ** 15 == 57344.0
    assert e4[0x01] == 2.0 ** -9 and e5[0x01] == 2.0 ** -16
    assert e4[0x08] == 2.0 ** -6 and e5[0x04] == 2.0 ** -14
    # E4M3 (fn): only S.1111.111 is NaN, no infinities
    assert [c for c in range(256) if np.isnan(e4[c])] == [0x7F, 0xFF]
    assert not np.isinf(e4).any()
    # E5M2: S.11111.00 is Inf, S.11111.{01,10,11} NaN
    assert e5[0x7C] == np.inf and e5[0xFC] == -np.inf
    assert [c for c in range(256) if np.isnan(e5[c])] == [0x7D, 0x7E, 0x7F, 0xFD, 0xFE, 0xFF]
    # sign symmetry
    for t in (e4, e5):
        fin = np.isfinite(t[:128])
        assert np.array_equal(t[128:][fin], -t[:128][fin])


def test_encode_golden_cases():
    n = 0
    with open(os.path.join(GOLD, "fp8_encode_cases.txt")) as f:
        for line in f:
            if not line.strip() or line.startswith("#"):
                continue
            fmt, val, code = line.split()[:3]
            got = int(O.encode([_parse_value(val)], FMT[fmt])[0])
            assert got == int(code, 16), (line, hex(got))
            n += 1
    assert n >= 25


@pytest.mark.parametrize("fmt", [O.E4M3, O.E5M2])
def test_roundtrip_every_finite_code(fmt):
    vals = O.decode(np.arange(256), fmt)
    fin = np.isfinite(vals)
    codes = np.arange(256)[fin]
    back = O.encode(vals[fin].astype(np.float32), fmt)
    assert np.array_equal(back, codes.astype(np.uint8))


@pytest.mark.parametrize("fmt", [O.E4M3, O.E5M2])
def test_midpoints_round_to_even(fmt):
    vals = O.decode(np.arange(128), fmt)
    fin = [c for c in range(128) if np.isfinite(vals[c])]
    for c in fin[:-1]:
        lo, hi = vals[c], vals[c + 1]
        mid = np.float32((lo + hi) / 2)          # exact: few significant bits
        assert float(mid) == (lo + hi) / 2
        even = c if c % 2 == 0 else c + 1
        assert O.encode([mid], fmt)[0] == even
        assert O.encode([-mid], fmt)[0] == even | 0x80
        below = np.nextafter(mid, np.float32(0))
        above = np.nextafter(mid, np.float32(np.inf))
        assert O.encode([below], fmt)[0] == c
        assert O.encode([above], fmt)[0] == c + 1


@pytest.mark.parametrize("fmt", [O.E4M3, O.E5M2])
def test_encode_monotonic(fmt):
    rng = np.random.default_rng(11)
    v = np.sort(np.concatenate([
        rng.standard_normal(20000).astype(np.float32) * np.float32(10.0 ** rng.uniform(-8, 6, 20000)),
        np.linspace(-70000, 70000, 5001, dtype=np.float32)]))
    d = O.decode(O.encode(v, fmt), fmt)
    assert np.all(np.diff(d) >= 0)


@pytest.mark.parametrize("fmt", [O.E4M3, O.E5M2])
def test_encode_matches_torch_in_range(fmt):
    rng = np.random.default_rng(5)
    fmax = O.FMAX[fmt]
    v = (rng.uniform(-1, 1, 200000) * fmax).astype(np.float32)
    v = np.concatenate([v, (rng.standard_normal(100000) * 2.0 ** rng.integers(-20, 4, 100000)).astype(np.float32)])
    v = v[np.abs(v) < fmax]
    ref = torch.from_numpy(v).to(TORCH_DT[fmt]).view(torch.uint8).numpy()
    assert np.array_equal(O.encode(v, fmt), ref)


@pytest.mark.parametrize("fmt", [O.E4M3, O.E5M2])
def test_encode_bruteforce_nearest(fmt):
    """Nearest finite code by scanning all codes (torch-decoded), ties to the
    even code, magnitudes beyond the largest finite value clamped to it."""
    table = _torch_decode(fmt)
    pos = [(table[c], c) for c in range(128) if np.isfinite(table[c])]
    pv = np.array([p[0] for p in pos])
    rng = np.random.default_rng(7)
    v = np.concatenate([rng.standard_normal(3000) * 2.0 ** rng.integers(-20, 18, 3000),
                        rng.uniform(-70000, 70000, 1000)]).astype(np.float32)
    got = O.encode(v, fmt)
    for x, g in zip(v, got):
        a = min(abs(float(x)), pv.max())
        dist = np.abs(pv - a)
        best = np.flatnonzero(dist == dist.min())
        codes = [pos[i][1] for i in best]
        code = [c for c in codes if c % 2 == 0][0] if len(codes) > 1 else codes[0]
        if np.signbit(x):
            code |= 0x80
        assert g == code, (x, hex(g), hex(code))


def test_bf16_decode_matches_torch():
    bits = np.arange(0, 1 << 16, dtype=np.uint32).astype(np.uint16)
    ours = O.bf16_to_f32(bits)
    ref = torch.from_numpy(bits.view(np.int16)).view(torch.bfloat16).float().numpy()
    assert np.array_equal(ours.view(np.uint32), ref.view(np.uint32))


def test_f64_to_bf16():
    rng = np.random.default_rng(3)
    v = rng.standard_normal(5000).astype(np.float32).astype(np.float64)
    ref = torch.from_numpy(v.astype(np.float32)).to(torch.bfloat16).view(torch.int16).numpy().view(np.uint16)
    assert np.array_equal(O.f64_to_bf16(v), ref)
    # A double just above a bf16 midpoint: 1 + 2^-8 + 2^-40 rounds up to 1 + 2^-7
    # (a first rounding to fp32 would land on the midpoint and round to even 1.0).
    assert O.f64_to_bf16([1 + 2 ** -8 + 2 ** -40])[0] == 0x3F81
    assert O.f64_to_bf16([1 + 2 ** -8])[0] == 0x3F80
    assert O.f64_to_bf16([3.5e38])[0] == 0x7F80
    assert O.f64_to_bf16([-0.0])[0] == 0x8000


def _pattern_windows(fmt):
    """Windows of 2^17 consecutive fp32 bit patterns (both signs) around the
    places a cast can go wrong: fp32 subnormals and zero, the format's
    smallest subnormal, 1.0, its largest finite value, and Inf / NaN."""
    fmax = O.FMAX[fmt]
    smallest = 2.0 ** -9 if fmt == O.E4M3 else 2.0 ** -16
    centres = [0, int(np.float32(smallest).view(np.uint32)), int(np.float32(1.0).view(np.uint32)),
               int(np.float32(fmax).view(np.uint32)), 0x7F800000]
    half = 1 << 16
    out = []
    for c in centres:
        lo = max(0, c - half)
        hi = min(0x80000000, c + half)
        out += [(lo, hi - lo), (0x80000000 + lo, hi - lo)]
    return out


@pytest.mark.parametrize("fmt", [O.E4M3, O.E5M2])
def test_encode_bits_range_over_fp32_patterns(fmt):
    """The encoder over a range of fp32 bit patterns (the expected side of
    the exhaustive GPU cast check): PyTorch's float8 cast below the largest
    finite value, saturation to it at and above (Inf included), and the
    format's NaN code (S.1111.111 / S.11111.11) for NaN."""
    fmax = O.FMAX[fmt]
    fmax_code = 0x7E if fmt == O.E4M3 else 0x7B
    for start, count in _pattern_windows(fmt):
        bits = np.arange(start, start + count, dtype=np.uint64).astype(np.uint32)
        v = bits.view(np.float32)
        got = O.encode_bits_range(start, count, fmt)
        sign = (bits >> 31).astype(np.uint8) << 7
        nan = np.isnan(v)
        big = ~nan & ((bits & 0x7FFFFFFF) >= np.float32(fmax).view(np.uint32))   # |v| >= fmax, by bits
        small = ~nan & ~big
        assert np.all(got[nan] & 0x7F == 0x7F)
        assert np.array_equal(got[big], fmax_code | sign[big])
        ref = torch.from_numpy(v[small].copy()).to(TORCH_DT[fmt]).view(torch.uint8).numpy()
        assert np.array_equal(got[small], ref), hex(start)
