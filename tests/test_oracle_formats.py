"""Pins of the oracle's FP8 encode/decode against things other than itself.

* hand-derived code points and rounding cases (tests/golden, derived from the
  1-4-3 / 1-5-2 bit layouts of the guide's "format choice E4M3 and E5M2");
* all 256 codes of each format round-trip bit-exactly (decode, then encode);
* two independent library implementations of the same formats (ml_dtypes and
  torch's float8 casts), exhaustively over every bf16 input times a set of scales;
* brute-force nearest-value search with exact rational arithmetic.
"""
import math
from fractions import Fraction

import numpy as np
import pytest
import torch

import oracle
from conftest import golden_rows

FMT = {"e4m3": oracle.E4M3, "e5m2": oracle.E5M2}


def f32(x):
    return np.float32(x)


def bits32(v):
    return int(np.array([v], np.float32).view(np.uint32)[0])


def test_decode_golden_codes():
    rows = golden_rows("fp8_codes.txt")
    assert len(rows) >= 30
    for fmt, code, value, *_ in rows:
        got = oracle.decode(np.array([int(code, 16)], np.uint8), FMT[fmt])[0]
        if value == "nan":
            assert np.isnan(got), (fmt, code)
        elif value in ("inf", "-inf"):
            assert got == float(value), (fmt, code)
        else:
            assert got == float(value), (fmt, code, got, value)
            assert math.copysign(1.0, got) == math.copysign(1.0, float(value)), (fmt, code)


def test_maxima_are_the_stated_ones():
    assert oracle.decode(np.array([0x7E], np.uint8), oracle.E4M3)[0] == 448.0
    assert oracle.decode(np.array([0x7B], np.uint8), oracle.E5M2)[0] == 57344.0
    assert oracle.fmax(oracle.E4M3) == 448.0
    assert oracle.fmax(oracle.E5M2) == 57344.0
    for fmt in (oracle.E4M3, oracle.E5M2):
        vals = oracle.decode(np.arange(256, dtype=np.uint8), fmt)
        finite = vals[np.isfinite(vals)]
        assert finite.max() == oracle.fmax(fmt)
        assert finite.min() == -oracle.fmax(fmt)


@pytest.mark.parametrize("fmt", [oracle.E4M3, oracle.E5M2])
def test_all_256_codes_round_trip(fmt):
    codes = np.arange(256, dtype=np.uint8)
    vals = oracle.decode(codes, fmt)
    np.testing.assert_array_equal(oracle.encode(vals, fmt, saturate=False), codes)
    # the saturating cast differs only where it must: +-inf (E5M2) become +-max
    back = oracle.encode(vals, fmt, saturate=True)
    inf = np.isinf(vals)
    np.testing.assert_array_equal(back[~inf], codes[~inf])
    assert np.all(back[inf] & 0x7F == 0x7B)


@pytest.mark.parametrize("fmt", [oracle.E4M3, oracle.E5M2])
def test_codes_are_monotone_and_layout_counts(fmt):
    vals = oracle.decode(np.arange(256, dtype=np.uint8), fmt).astype(np.float64)
    pos = vals[:128]
    fin = pos[np.isfinite(pos)]
    # positive codes increase strictly in value up to the largest finite one
    assert np.all(np.diff(fin) > 0)
    n_nan = int(np.isnan(vals).sum())
    n_inf = int(np.isinf(vals).sum())
    if fmt == oracle.E4M3:
        assert (n_nan, n_inf) == (2, 0)
        # 4 exponent bits: 15 binades of normals + subnormals, 8 values per binade
        assert len(fin) == 127
    else:
        assert (n_nan, n_inf) == (6, 2)
        assert len(fin) == 124


def test_rounding_golden_cases():
    rows = golden_rows("fp8_rounding.txt")
    assert len(rows) >= 30
    for fmt, value, sat, expected, *_ in rows:
        got = oracle.encode(np.array([float(value)], np.float32), FMT[fmt], saturate=bool(int(sat)))[0]
        assert got == int(expected, 16), (fmt, value, sat, hex(got), expected)


def _exact_nearest_code(v, fmt, saturate):
    """Brute force over all finite codes with exact rationals (ties -> even code)."""
    codes = np.arange(256, dtype=np.uint8)
    vals = oracle.decode(codes, fmt)
    if math.isnan(v):
        return None
    neg = math.copysign(1.0, v) < 0
    a = abs(v)
    fmax = oracle.fmax(fmt)
    if a > fmax and saturate:
        return (0x80 if neg else 0) | (0x7E if fmt == oracle.E4M3 else 0x7B)
    fa = Fraction(a) if math.isfinite(a) else None
    best, best_d = None, None
    cands = [(int(c), Fraction(float(vals[c]))) for c in range(128) if np.isfinite(vals[c])]
    # the value one step past the largest finite code (overflow threshold)
    # (its code is the one after the largest finite code: 0x7F, odd, for E4M3 -- NaN;
    # 0x7C, even, for E5M2 -- infinity -- which decides the tie at the threshold)
    over_code = 0x7F if fmt == oracle.E4M3 else 0x7C
    cands.append((over_code, Fraction(480) if fmt == oracle.E4M3 else Fraction(65536)))
    if fa is None:
        best = over_code
    else:
        for c, cv in cands:
            d = abs(fa - cv)
            if best_d is None or d < best_d or (d == best_d and (c & 1) == 0 and (best & 1) == 1):
                best, best_d = c, d
    return (0x80 if neg else 0) | best


@pytest.mark.parametrize("fmt", [oracle.E4M3, oracle.E5M2])
def test_encode_matches_exact_brute_force(fmt):
    rng = np.random.default_rng(7)
    # values spread over every binade of the format plus overflow and underflow regions
    exps = rng.integers(-20, 18, size=3000)
    v = (rng.uniform(1.0, 2.0, size=3000) * np.exp2(exps)).astype(np.float32)
    v[::2] *= -1
    # add every exact midpoint between neighbouring finite codes (the tie cases)
    vals = oracle.decode(np.arange(128, dtype=np.uint8), fmt).astype(np.float64)
    fin = vals[np.isfinite(vals)]
    mids = ((fin[1:] + fin[:-1]) / 2).astype(np.float32)
    v = np.concatenate([v, mids, -mids, np.array([np.inf, -np.inf, 0.0, -0.0], np.float32)])
    for sat in (False, True):
        got = oracle.encode(v, fmt, saturate=sat)
        for x, g in zip(v.tolist(), got.tolist()):
            assert g == _exact_nearest_code(x, fmt, sat), (fmt, sat, x, hex(g))


def _all_bf16_as_f32():
    b = np.arange(65536, dtype=np.uint32) << 16
    x = b.view(np.float32)
    return x[~np.isnan(x)]


@pytest.mark.parametrize("fmt", [oracle.E4M3, oracle.E5M2])
def test_exhaustive_bf16_against_ml_dtypes(fmt):
    ml_dtypes = pytest.importorskip("ml_dtypes")
    target = ml_dtypes.float8_e4m3fn if fmt == oracle.E4M3 else ml_dtypes.float8_e5m2
    x = _all_bf16_as_f32()
    fmax = oracle.fmax(fmt)
    for scale in (1.0, 0.125, 128.0, 448.0 / 3.7, 57344.0 / 11.0, 2.0 ** -100, 3.0e30):
        p = (x * np.float32(scale)).astype(np.float32)     # binary32 product, RN
        # plain cast: ml_dtypes rounds to nearest-even with NaN/inf on overflow
        ref = p.astype(target).view(np.uint8)
        got = oracle.encode(p, fmt, saturate=False)
        np.testing.assert_array_equal(got, ref, err_msg=f"scale={scale}")
        # saturating cast: the same, with magnitudes above the largest finite value clamped
        clamped = np.clip(p, -fmax, fmax).astype(np.float32)
        ref_sat = clamped.astype(target).view(np.uint8)
        got_sat = oracle.encode(p, fmt, saturate=True)
        np.testing.assert_array_equal(got_sat, ref_sat, err_msg=f"sat scale={scale}")


@pytest.mark.parametrize("fmt", [oracle.E4M3, oracle.E5M2])
def test_exhaustive_bf16_against_torch_float8(fmt):
    tdt = torch.float8_e4m3fn if fmt == oracle.E4M3 else torch.float8_e5m2
    x = _all_bf16_as_f32()
    fmax = oracle.fmax(fmt)
    for scale in (1.0, 0.5, 96.0, 448.0 / 5.25):
        p = (x * np.float32(scale)).astype(np.float32)
        clamped = np.clip(p, -fmax, fmax).astype(np.float32)   # in range: no overflow rule involved
        ref = torch.from_numpy(clamped).to(tdt).view(torch.uint8).numpy()
        got = oracle.encode(p, fmt, saturate=True)
        np.testing.assert_array_equal(got, ref, err_msg=f"scale={scale}")


def test_decode_against_ml_dtypes_all_codes():
    ml_dtypes = pytest.importorskip("ml_dtypes")
    codes = np.arange(256, dtype=np.uint8)
    for fmt, t in ((oracle.E4M3, ml_dtypes.float8_e4m3fn), (oracle.E5M2, ml_dtypes.float8_e5m2)):
        ref = codes.view(t).astype(np.float32)
        got = oracle.decode(codes, fmt)
        np.testing.assert_array_equal(np.isnan(got), np.isnan(ref))
        ok = ~np.isnan(ref)
        np.testing.assert_array_equal(got[ok], ref[ok])
        np.testing.assert_array_equal(np.signbit(got[ok]), np.signbit(ref[ok]))
