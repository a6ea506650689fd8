"""Pins of the oracle's binary32-input quantizers (the FP32 master copy of a weight
quantized directly; search-result page, mixed-precision dataflow paragraph).

The element rule, block amaxes, scale rule and layouts are the BF16 quantizers';
only the input type differs.  Pinned by: the reduction to the (pinned) BF16
quantizers on inputs that are bfloat16 values, hand-derived codes of inputs whose
bfloat16 rounding would land on an FP8 midpoint (tests/golden/fp8_f32_inputs.txt),
and a library computation (numpy binary32 division and products, ml_dtypes'
round-to-nearest-even casts) on general binary32 inputs."""
import numpy as np
import pytest

import oracle
from conftest import golden_rows

ml_dtypes = pytest.importorskip("ml_dtypes")

FMT = {"e4m3": oracle.E4M3, "e5m2": oracle.E5M2}
KINDS = [oracle.KIND_TENSOR, oracle.KIND_1x128, oracle.KIND_128x128, oracle.KIND_MX]
LIB_FP8 = {oracle.E4M3: ml_dtypes.float8_e4m3fn, oracle.E5M2: ml_dtypes.float8_e5m2}
FMAX = {oracle.E4M3: 448.0, oracle.E5M2: 57344.0}


def to_bf16_bits(x):
    b = np.ascontiguousarray(x, np.float32).view(np.uint32).astype(np.uint64)
    return ((b + 0x7FFF + ((b >> 16) & 1)) >> 16).astype(np.uint16)


def bf16_to_f32(h):
    return (h.astype(np.uint32) << 16).view(np.float32)


def general_f32(shape, seed):
    """Binary32 values with every mantissa bit in use, a spread of magnitudes and a few
    exact zeros and outliers."""
    rng = np.random.default_rng(seed)
    x = (rng.standard_normal(shape) * np.exp2(rng.integers(-6, 7, shape))).astype(np.float32)
    x.reshape(-1)[rng.integers(0, x.size, 7)] = 0.0
    x.reshape(-1)[rng.integers(0, x.size, 3)] *= np.float32(1000.0)
    return x


@pytest.mark.parametrize("kind", KINDS)
@pytest.mark.parametrize("fmt", [oracle.E4M3, oracle.E5M2])
def test_reduces_to_the_bf16_quantizer_on_bf16_values(kind, fmt):
    h = to_bf16_bits(general_f32((256, 384), 1 + kind))
    x = bf16_to_f32(h)
    scale = None
    if kind == oracle.KIND_TENSOR:
        scale, _ = oracle.tensor_scale(oracle.amax(h), fmt)
    for f32_fn, bf_fn in ((oracle.quantize_rowwise_f32, oracle.quantize_rowwise),
                          (oracle.quantize_colwise_f32, oracle.quantize_colwise)):
        q32, s32 = f32_fn(x, kind, fmt, scale)
        qbf, sbf = bf_fn(h, kind, fmt, scale)
        assert np.array_equal(q32, qbf)
        assert np.array_equal(np.asarray(s32).view(np.uint8), np.asarray(sbf).view(np.uint8))


def test_hand_derived_codes_of_binary32_inputs():
    rows = golden_rows("fp8_f32_inputs.txt")
    assert len(rows) >= 8
    for fmt_name, bits, _, expected, *_ in rows:
        x = np.array([[int(bits, 16)]], np.uint32).view(np.float32)
        q, s = oracle.quantize_rowwise_f32(x, oracle.KIND_TENSOR, FMT[fmt_name], np.float32(1.0))
        assert q[0, 0] == int(expected, 16), (fmt_name, bits, hex(q[0, 0]))
        assert s[0] == np.float32(1.0)


def lib_scale(amax, fmt):
    """scale = FMAX / amax in binary32 (numpy), amax 0 or non-finite -> 1, inf -> FLT_MAX."""
    if not amax > 0 or not np.isfinite(amax):
        return np.float32(1.0)
    with np.errstate(over="ignore"):
        s = np.float32(FMAX[fmt]) / np.float32(amax)
    return np.float32(np.finfo(np.float32).max) if np.isinf(s) else s


def lib_cast(p, fmt):
    """Saturating round-to-nearest-even cast of binary32 products (ml_dtypes' cast of the
    products clipped to +-max: the clip moves only values beyond max, which round to max)."""
    m = np.float32(FMAX[fmt])
    return np.clip(p, -m, m).astype(LIB_FP8[fmt]).view(np.uint8)


def lib_mx_exponent(amax, fmt):
    if not amax > 0 or not np.isfinite(amax):
        return 0
    e = -127
    while e < 127 and float(amax) > np.ldexp(FMAX[fmt], e):
        e += 1
    return e


@pytest.mark.parametrize("fmt", [oracle.E4M3, oracle.E5M2])
def test_blockwise_and_mx_match_a_library_computation(fmt):
    x = general_f32((256, 256), 7)
    # 1 x 128
    q, s = oracle.quantize_rowwise_f32(x, oracle.KIND_1x128, fmt)
    for r in range(x.shape[0]):
        for b in range(2):
            blk = x[r, 128 * b:128 * b + 128]
            sc = lib_scale(np.max(np.abs(blk)), fmt)
            assert np.array_equal(q[r, 128 * b:128 * b + 128], lib_cast(blk * sc, fmt)), (r, b)
            assert s[r, b] == np.float32(1.0) / sc
    # 128 x 128
    q, s = oracle.quantize_rowwise_f32(x, oracle.KIND_128x128, fmt)
    for br in range(2):
        for bc in range(2):
            blk = x[128 * br:128 * br + 128, 128 * bc:128 * bc + 128]
            sc = lib_scale(np.max(np.abs(blk)), fmt)
            assert np.array_equal(q[128 * br:128 * br + 128, 128 * bc:128 * bc + 128], lib_cast(blk * sc, fmt))
            assert s[br, bc] == np.float32(1.0) / sc
    # MX 1 x 32: exact power-of-two scaling
    q, s = oracle.quantize_rowwise_f32(x, oracle.KIND_MX, fmt)
    for r in range(0, x.shape[0], 7):
        for b in range(8):
            blk = x[r, 32 * b:32 * b + 32]
            e = lib_mx_exponent(np.max(np.abs(blk)), fmt)
            assert s[r, b] == e + 127
            assert np.array_equal(q[r, 32 * b:32 * b + 32], lib_cast(blk * np.float32(np.ldexp(1.0, -e)), fmt))


@pytest.mark.parametrize("fmt", [oracle.E4M3, oracle.E5M2])
def test_per_tensor_matches_a_library_computation_and_the_column_copy_is_the_transpose(fmt):
    x = general_f32((130, 70), 9)
    sc = lib_scale(np.max(np.abs(x)), fmt)
    q, s = oracle.quantize_rowwise_f32(x, oracle.KIND_TENSOR, fmt, sc)
    assert np.array_equal(q, lib_cast(x * sc, fmt))
    qc, _ = oracle.quantize_colwise_f32(x, oracle.KIND_TENSOR, fmt, sc)
    assert np.array_equal(qc, q.T)
