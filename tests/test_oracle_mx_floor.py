"""Pins of the oracle's floor-rule MX exponent (the documented alternate of the guide's
"MXFP8 scaling" section, behind its own recipe; the ceil rule stays the default).

e = floor(log2 amax) - emax (emax 8 for E4M3, 15 for E5M2): hand-derived values
(tests/golden/mx_exponent_floor.txt), the closed-form bracket 2^(e+emax) <= amax <
2^(e+emax+1) on random and boundary amaxes, its relation to the ceil rule (equal unless
amax's significand exceeds 1.75), and the quantized block against a library computation
(exact power-of-two scaling, then a saturating round-to-nearest-even cast)."""
import numpy as np
import pytest

import oracle
from conftest import golden_rows

FMT = {"e4m3": oracle.E4M3, "e5m2": oracle.E5M2}
EMAX = {oracle.E4M3: 8, oracle.E5M2: 15}
FMAX = {oracle.E4M3: 448.0, oracle.E5M2: 57344.0}


def test_hand_derived_floor_exponents():
    rows = golden_rows("mx_exponent_floor.txt")
    assert len(rows) >= 14
    for fmt_name, amax, e, *_ in rows:
        assert oracle.mx_exponent_floor(np.float32(float(amax)), FMT[fmt_name]) == int(e), (fmt_name, amax)


@pytest.mark.parametrize("fmt", [oracle.E4M3, oracle.E5M2])
def test_floor_bracket_and_relation_to_the_ceil_rule(fmt):
    rng = np.random.default_rng(5)
    vals = np.concatenate([np.exp2(rng.uniform(-120, 120, 4000)).astype(np.float32),
                           np.exp2(np.arange(-120, 121)).astype(np.float32),
                           np.nextafter(np.exp2(np.arange(-120, 121)).astype(np.float32), np.float32(0))])
    for a in vals:
        e = oracle.mx_exponent_floor(a, fmt)
        lo, hi = np.ldexp(1.0, e + EMAX[fmt]), np.ldexp(1.0, e + EMAX[fmt] + 1)
        if -127 < e < 127:
            assert lo <= float(a) < hi, (a, e)
        m = float(a) / np.ldexp(1.0, int(np.floor(np.log2(float(a)))))   # significand in [1, 2)
        ec = oracle.mx_exponent(a, fmt)
        if -127 < e < 127 and -127 < ec < 127:
            assert ec == (e + 1 if m > 1.75 else e), (a, e, ec)


@pytest.mark.parametrize("fmt", [oracle.E4M3, oracle.E5M2])
def test_floor_blocks_match_a_library_computation(fmt):
    ml_dtypes = pytest.importorskip("ml_dtypes")
    lib = {oracle.E4M3: ml_dtypes.float8_e4m3fn, oracle.E5M2: ml_dtypes.float8_e5m2}[fmt]
    rng = np.random.default_rng(8)
    x = (rng.standard_normal((64, 256)) * np.exp2(rng.integers(-6, 7, (64, 1)))).astype(np.float32)
    x[3, 32:64] *= np.float32(1.9) / np.max(np.abs(x[3, 32:64]))   # a block whose max saturates after scaling
    q, s = oracle.quantize_rowwise_f32(x, oracle.KIND_MX_FLOOR, fmt)
    h = np.ascontiguousarray(x).view(np.uint32)
    xb = ((h.astype(np.uint64) + 0x7FFF + ((h >> 16) & 1)) >> 16).astype(np.uint16)   # bf16 copy
    qb, sb = oracle.quantize_rowwise(xb, oracle.KIND_MX_FLOOR, fmt)
    xbf = (xb.astype(np.uint32) << 16).view(np.float32)
    m = np.float32(FMAX[fmt])
    for src, qq, ss in ((x, q, s), (xbf, qb, sb)):
        for r in range(0, 64, 3):
            for b in range(8):
                blk = src[r, 32 * b:32 * b + 32]
                amax = float(np.max(np.abs(blk)))
                e = int(np.floor(np.log2(amax))) - EMAX[fmt] if amax > 0 else 0
                e = max(-127, min(127, e))
                assert ss[r, b] == e + 127
                p = blk * np.float32(np.ldexp(1.0, -e))
                assert np.array_equal(qq[r, 32 * b:32 * b + 32], np.clip(p, -m, m).astype(lib).view(np.uint8))
    # the saturating block: its largest element lands on +-FMAX
    assert np.max(q[3, 32:64] & 0x7F) == (0x7E if fmt == oracle.E4M3 else 0x7B)
