"""Pins of the oracle's FP8 -> BF16 dequantization (fp8_oracle.c: orc_round_bf16,
orc_dequantize_bf16) against what the mathematics fixes: brute-force nearest
bfloat16 (ties to even, gradual underflow, overflow at max + half an ulp), an
independent library conversion on binary32 inputs, and exact power-of-two cases."""
import numpy as np
import pytest
import torch

import oracle


def _bf16_table():
    """All finite non-negative bfloat16 values (bit patterns 0x0000..0x7F7F) as float64."""
    bits = np.arange(0, 0x7F80, dtype=np.uint32)
    return bits.astype(np.uint16), (bits << 16).view(np.float32).astype(np.float64)


def brute_nearest_bf16(v: float) -> int:
    bits, vals = _TABLE
    if np.isnan(v):
        return 0x7FC0 | (0x8000 if np.signbit(v) else 0)
    sign = 0x8000 if np.signbit(v) else 0
    a = abs(v)
    top = vals[-1]
    half_ulp_top = (vals[-1] - vals[-2]) / 2
    if a >= top + half_ulp_top:
        return sign | 0x7F80
    i = int(np.searchsorted(vals, a))
    cands = [j for j in (i - 1, i) if 0 <= j < len(vals)]
    d = [abs(vals[j] - a) for j in cands]
    best = min(d)
    ties = [cands[k] for k in range(len(cands)) if d[k] == best]
    pick = ties[0] if len(ties) == 1 else [j for j in ties if bits[j] % 2 == 0][0]
    return sign | int(bits[pick])


_TABLE = _bf16_table()


def tricky_values():
    rng = np.random.default_rng(7)
    out = []
    bits, vals = _TABLE
    # exact midpoints and their neighbours across the whole range (incl. subnormals)
    idx = np.concatenate([np.arange(0, 300), rng.integers(0, len(vals) - 1, 400), np.arange(len(vals) - 300, len(vals) - 1)])
    for i in idx:
        m = (vals[i] + vals[i + 1]) / 2
        out += [m, np.nextafter(m, 0), np.nextafter(m, np.inf)]
    # products with 28-bit significands (FP8 code x binary32 multiplier) over all exponents
    sig = rng.integers(1 << 27, 1 << 28, 600).astype(np.float64)
    ex = rng.integers(-165, 100, 600)
    out += list(np.ldexp(sig, ex))
    # overflow boundary and specials
    top, half = vals[-1], (vals[-1] - vals[-2]) / 2
    out += [top, top + half, np.nextafter(top + half, 0), 2.0 ** 128, 0.0, -0.0, np.inf, -np.inf]
    out = np.array(out, np.float64)
    return np.concatenate([out, -out[: len(out) // 3]])


def test_round_bf16_is_brute_force_nearest_even():
    v = tricky_values()
    got = oracle.round_bf16(v)
    for x, g in zip(v, got):
        assert int(g) == brute_nearest_bf16(float(x)), (x, hex(int(g)))


def test_round_bf16_matches_library_on_binary32_inputs():
    # a binary32 -> bfloat16 conversion (round to nearest even) from another implementation
    rng = np.random.default_rng(8)
    f = np.concatenate([(rng.standard_normal(20000) * 10.0 ** rng.integers(-40, 38, 20000)).astype(np.float32),
                        rng.integers(0, 1 << 32, 20000, dtype=np.uint64).astype(np.uint32).view(np.float32)])
    f = f[np.isfinite(f)]
    lib = torch.from_numpy(f.copy()).to(torch.bfloat16).view(torch.int16).numpy().view(np.uint16)
    assert np.array_equal(oracle.round_bf16(f.astype(np.float64)), lib)


@pytest.mark.parametrize("fmt", [oracle.E4M3, oracle.E5M2])
@pytest.mark.parametrize("k", [-20, 0, 13])
def test_dequantize_bf16_power_of_two_scale_is_exact(fmt, k):
    # every FP8 value times 2^k is a bfloat16 (at most 4 significant bits)
    codes = np.arange(256, dtype=np.uint8).reshape(2, 128)
    s = np.array([2.0 ** k], np.float32)
    got = oracle.dequantize_bf16(codes, oracle.KIND_TENSOR, fmt, s)
    dec = oracle.decode(codes, fmt).astype(np.float64) * 2.0 ** k
    fin = np.isfinite(dec)
    exp_bits = (dec[fin].astype(np.float32).view(np.uint32) >> 16).astype(np.uint16)
    assert np.array_equal(got[fin], exp_bits)
    assert np.all((got[~fin] & 0x7F80) == 0x7F80)     # inf / NaN codes stay non-finite


def test_dequantize_bf16_recipes_and_mx_nan_byte():
    rng = np.random.default_rng(9)
    q = rng.integers(0, 256, (256, 256), dtype=np.uint8)
    q[(q & 0x7F) == 0x7F] = 0x10                      # no E4M3 NaN codes here
    s1 = (rng.random((256, 2)) * 3 + 0.1).astype(np.float32)
    got = oracle.dequantize_bf16(q, oracle.KIND_1x128, oracle.E4M3, s1)
    # element (r, c) uses the multiplier of its 1 x 128 block, rounded once
    r, c = 77, 200
    ref = oracle.round_bf16(np.array([float(oracle.decode(q[r:r + 1, c:c + 1], oracle.E4M3)[0, 0]) * float(s1[r, 1])]))
    assert got[r, c] == ref[0]
    e = rng.integers(100, 150, (256, 8)).astype(np.uint8)
    e[3, 2] = 255
    got = oracle.dequantize_bf16(q, oracle.KIND_MX, oracle.E4M3, e)
    assert np.all((got[3, 64:96] & 0x7FFF) > 0x7F80)  # the E8M0 NaN byte gives NaN
    assert np.all((np.delete(got, 3, axis=0) & 0x7F80) != 0x7F80)
