"""GPU parity of fp8_dequantize (FP8 -> BF16) against the oracle, bit for bit
(NaN outputs: NaN-ness).  The FP8 codes and multipliers are the oracle's own
(quantized from seeded inputs, or constructed), uploaded to the device."""
import numpy as np
import pytest
import torch

import oracle
import scaled_quantize_gemm_amax_gb300 as fq
from scaled_quantize_gemm_amax_gb300 import workloads as wl
from gpu_util import R, F, KIND, assert_status_ok, bits16, host, require_gpu

pytestmark = pytest.mark.gpu


@pytest.fixture(scope="module", autouse=True)
def _gpu():
    require_gpu()


def dev(a):
    return torch.from_numpy(np.ascontiguousarray(a)).cuda()


def run_gpu(q, recipe, fmt, s):
    y = fq.dequantize(dev(q), recipe, fmt, dev(s))
    torch.cuda.synchronize()
    assert_status_ok()
    return host(y.view(torch.int16)).view(np.uint16)


def assert_bf16_equal(got, ref, what):
    nan_g = (got & 0x7F80) == 0x7F80
    nan_g &= (got & 0x007F) != 0
    nan_r = ((ref & 0x7F80) == 0x7F80) & ((ref & 0x007F) != 0)
    assert np.array_equal(nan_g, nan_r), f"{what}: NaN positions differ"
    bad = np.argwhere((got != ref) & ~nan_r)
    if bad.size:
        i = tuple(bad[0])
        raise AssertionError(f"{what}: {len(bad)} differ; first at {i}: got {got[i]:#06x} ref {ref[i]:#06x}")


@pytest.mark.parametrize("recipe", [R.TENSOR, R.BLOCK_1x128, R.BLOCK_128x128, R.MX_1x32, R.MX_1x32_TILED])
@pytest.mark.parametrize("fmt", [F.E4M3, F.E5M2])
def test_dequantize_round_trip_copies(recipe, fmt):
    # the oracle's row- and column-wise copies of a seeded matrix (with outlier columns)
    x = wl.normal_bf16((384, 256), 70, 1.0, "cpu")
    x[:, 5] *= 300.0
    xh = bits16(x)
    kind = KIND[recipe]
    scale = None
    if recipe == R.TENSOR:
        scale, _ = oracle.tensor_scale(oracle.amax(xh), int(fmt))
    for name, (q, s) in (("row", oracle.quantize_rowwise(xh, kind, int(fmt), scale)),
                         ("col", oracle.quantize_colwise(xh, kind, int(fmt), scale))):
        ref = oracle.dequantize_bf16(q, kind, int(fmt), s)
        s_dev = oracle.mx_to_tiled(s) if recipe == R.MX_1x32_TILED else s
        assert_bf16_equal(run_gpu(q, recipe, fmt, s_dev), ref, f"{recipe.name} {name}")


@pytest.mark.parametrize("fmt", [F.E4M3, F.E5M2])
@pytest.mark.parametrize("scale", [1.7, 2.0 ** -20, 2.0 ** -100, 2.0 ** -101, 2.0 ** -130, 3.0 * 2.0 ** -149,
                                   2.0 ** 100, 2.0 ** 101, 2.0 ** 120, 0.0])
def test_dequantize_every_code_every_range(fmt, scale):
    # all 256 codes (NaN / inf included) under multipliers that keep the products normal,
    # push them into the subnormal range, or past the bfloat16 maximum
    q = np.tile(np.arange(256, dtype=np.uint8), 8).reshape(16, 128)
    s = np.array([scale], np.float32)
    ref = oracle.dequantize_bf16(q, oracle.KIND_TENSOR, int(fmt), s)
    assert_bf16_equal(run_gpu(q, R.TENSOR, fmt, s), ref, f"scale {scale}")


def test_dequantize_mx_extreme_exponents_and_nan_byte():
    rng = np.random.default_rng(71)
    q = rng.integers(0, 256, (256, 256), dtype=np.uint8)
    e = rng.integers(0, 256, (256, 8), dtype=np.uint8)       # every E8M0 byte, 0 (2^-127) .. 255 (NaN)
    e[0, :] = [0, 1, 26, 27, 227, 228, 254, 255]
    for fmt in (F.E4M3, F.E5M2):
        ref = oracle.dequantize_bf16(q, oracle.KIND_MX, int(fmt), e)
        assert_bf16_equal(run_gpu(q, R.MX_1x32, fmt, e), ref, f"MX row-major {fmt.name}")
        assert_bf16_equal(run_gpu(q, R.MX_1x32_TILED, fmt, oracle.mx_to_tiled(e)), ref, f"MX tiled {fmt.name}")


@pytest.mark.parametrize("shape", [(1, 1), (37, 53), (3, 16), (5, 1000)])
def test_dequantize_per_tensor_any_shape(shape):
    rng = np.random.default_rng(72)
    q = rng.integers(0, 256, shape, dtype=np.uint8)
    s = np.array([0.37], np.float32)
    ref = oracle.dequantize_bf16(q, oracle.KIND_TENSOR, oracle.E4M3, s)
    assert_bf16_equal(run_gpu(q, R.TENSOR, F.E4M3, s), ref, str(shape))


def test_dequantize_blockwise_4096_full():
    # the blockwise workload's activation size, every element compared
    x = wl.normal_bf16((4096, 4096), 73, 1.0, "cpu")
    xh = bits16(x)
    q, s = oracle.quantize_rowwise(xh, oracle.KIND_1x128, oracle.E4M3)
    ref = oracle.dequantize_bf16(q, oracle.KIND_1x128, oracle.E4M3, s)
    assert_bf16_equal(run_gpu(q, R.BLOCK_1x128, F.E4M3, s), ref, "4096^2 1x128")
