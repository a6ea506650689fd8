"""GPU parity of amax, scale and quantize / cast-transpose against the oracle:
bit-exact FP8 bytes, scales and amax for every recipe and format, at sizes that
span several tiles and ragged edges, at the benchmark sizes, and at edge cases
(empty, all-zero, tiny values, saturation, NaN)."""
import numpy as np
import pytest
import torch

import oracle
import scaled_quantize_gemm_amax_gb300 as fq
from scaled_quantize_gemm_amax_gb300 import workloads as wl
from gpu_util import R, F, KIND, assert_bytes_equal, assert_status_ok, bits16, check_cast, f32bits, host, \
    require_gpu

pytestmark = pytest.mark.gpu

ALL_RECIPES = [R.TENSOR, R.BLOCK_1x128, R.BLOCK_128x128, R.MX_1x32, R.MX_1x32_TILED]


@pytest.fixture(scope="module", autouse=True)
def _gpu():
    require_gpu()


def _x(shape, seed, sigma=1.0, outliers=True):
    x = wl.normal_bf16(shape, seed, sigma, device="cuda")
    if outliers:
        wl.with_outlier_elements(x, seed, frac=0.002, factor=100.0)
    return x


@pytest.mark.parametrize("recipe", ALL_RECIPES)
@pytest.mark.parametrize("fmt", [F.E4M3, F.E5M2])
def test_cast_transpose_multi_tile(recipe, fmt):
    check_cast(_x((384, 512), 100 + int(recipe)), recipe, fmt)


@pytest.mark.parametrize("recipe", ALL_RECIPES)
def test_row_only_and_col_only(recipe):
    x = _x((256, 384), 200 + int(recipe))
    check_cast(x, recipe, F.E4M3, row=True, col=False)
    check_cast(x, recipe, F.E4M3, row=False, col=True)


@pytest.mark.parametrize("shape", [(144, 272), (16, 16), (1000, 48), (130, 2048)])
def test_per_tensor_ragged_tiles(shape):
    # multiples of 16: the TMA path with partial tiles
    check_cast(_x(shape, 300), R.TENSOR, F.E4M3)


@pytest.mark.parametrize("shape", [(33, 47), (1, 1), (7, 300), (129, 130)])
def test_per_tensor_any_shape(shape):
    # not multiples of 16: the plain path
    check_cast(_x(shape, 301, outliers=False), R.TENSOR, F.E5M2)


def test_block_recipes_with_ragged_free_dimension():
    # 1x128 row-wise only with rows not a multiple of 128; MX plain layout with 160 rows
    check_cast(_x((200, 256), 302), R.BLOCK_1x128, F.E4M3, row=True, col=False)
    check_cast(_x((160, 256), 303), R.MX_1x32, F.E4M3)
    check_cast(_x((96, 160), 304), R.MX_1x32, F.E5M2)
    # column tiles hanging over C by 1 and 3 blocks of 32 (no bytes past the last block)
    check_cast(_x((256, 416), 305), R.MX_1x32, F.E4M3)
    check_cast(_x((128, 352), 306), R.MX_1x32, F.E4M3, row=True, col=False)


def test_blockwise_config_full_size():
    # the 4096 x 4096 blockwise workload: X (1x128, row + col) and W (128x128)
    x, w = wl.cfg2_blockwise("cuda")
    check_cast(x, R.BLOCK_1x128, F.E4M3)
    check_cast(w, R.BLOCK_128x128, F.E4M3)


def test_mx_config_full_size():
    x, w = wl.cfg3_mx("up", "cuda")            # 8192 x 4096 and 11008 x 4096
    check_cast(x, R.MX_1x32_TILED, F.E4M3)
    check_cast(w, R.MX_1x32_TILED, F.E4M3, col=False)


def test_sweep_largest_size_sampled_tiles():
    # 32768 x 32768 (2 GiB bf16): compare a seeded sample of 128x128 tiles of every
    # output; per-tensor uses the exact full-tensor amax from the oracle.
    x = wl.cfg5_sweep(32768, "cuda")
    rng = np.random.default_rng(5)
    tiles = [(0, 0), (255, 255)] + [tuple(t) for t in rng.integers(0, 256, (6, 2))]
    xh_full_amax = oracle.amax(bits16(x))
    for recipe in (R.TENSOR, R.BLOCK_1x128, R.BLOCK_128x128, R.MX_1x32):
        scale_np = scale_t = None
        if recipe == R.TENSOR:
            scale_np, _ = oracle.tensor_scale(xh_full_amax, 0)
            scale_t = torch.tensor([scale_np], dtype=torch.float32, device="cuda")
        amax_t = torch.zeros(1, dtype=torch.float32, device="cuda")
        qr, sr, qc, sc = fq.cast_transpose(x, recipe, F.E4M3, scale_t, amax_t)
        torch.cuda.synchronize()
        assert_status_ok()
        assert f32bits(host(amax_t))[0] == f32bits(xh_full_amax)
        for (ti, tj) in tiles:
            rs, cs = slice(ti * 128, ti * 128 + 128), slice(tj * 128, tj * 128 + 128)
            xt = bits16(x[rs, cs])
            kind = KIND[recipe]
            q_ref, s_ref = oracle.quantize_rowwise(xt, kind, 0, scale_np)
            assert_bytes_equal(host(qr[rs, cs]), q_ref, f"q_row tile {ti},{tj}")
            qc_ref, sc_ref = oracle.quantize_colwise(xt, kind, 0, scale_np)
            assert_bytes_equal(host(qc[cs, rs]), qc_ref, f"q_col tile {ti},{tj}")
            if recipe == R.BLOCK_1x128:
                assert_bytes_equal(f32bits(host(sr[rs, tj])), f32bits(s_ref[:, 0]), "s_row")
                assert_bytes_equal(f32bits(host(sc[cs, ti])), f32bits(sc_ref[:, 0]), "s_col")
            elif recipe == R.BLOCK_128x128:
                assert f32bits(host(sr[ti, tj])) == f32bits(s_ref[0, 0])
                assert f32bits(host(sc[tj, ti])) == f32bits(sc_ref[0, 0])
            elif recipe == R.MX_1x32:
                assert_bytes_equal(host(sr[rs, 4 * tj:4 * tj + 4]), s_ref, "s_row")
                assert_bytes_equal(host(sc[cs, 4 * ti:4 * ti + 4]), sc_ref, "s_col")
        del qr, sr, qc, sc


def test_amax_kernel_and_compute_scale_chain():
    # per-tensor current scaling end to end on the device: amax -> scale -> cast
    for fmt in (F.E4M3, F.E5M2):
        for shape, seed in (((256, 256), 1), ((1, 7), 2), ((1000, 1003), 3), ((4096, 4096), 4)):
            x = _x(shape, 400 + seed)
            xh = bits16(x)
            amax = torch.empty(1, dtype=torch.float32, device="cuda")
            scale = torch.empty(1, dtype=torch.float32, device="cuda")
            sinv = torch.empty(1, dtype=torch.float32, device="cuda")
            fq.fp8_amax(x, amax)
            fq.fp8_compute_scale(amax, fmt, scale, sinv)
            q = torch.empty(shape, dtype=torch.uint8, device="cuda")
            fq.fp8_quantize(x, R.TENSOR, fmt, scale, None, q, None)
            torch.cuda.synchronize()
            assert_status_ok()
            a_ref = oracle.amax(xh)
            s_ref, si_ref = oracle.tensor_scale(a_ref, int(fmt))
            assert f32bits(host(amax))[0] == f32bits(a_ref)
            assert f32bits(host(scale))[0] == f32bits(s_ref)
            assert f32bits(host(sinv))[0] == f32bits(si_ref)
            q_ref, _ = oracle.quantize_rowwise(xh, oracle.KIND_TENSOR, int(fmt), s_ref)
            assert_bytes_equal(host(q), q_ref, "q")


def test_compute_scale_edge_values():
    # IEEE division on many amax values, including 0, inf, NaN, subnormals, FLT_MAX
    rng = np.random.default_rng(9)
    vals = np.concatenate([
        np.abs(rng.standard_normal(64)).astype(np.float32) * np.exp2(rng.integers(-140, 120, 64)).astype(np.float32),
        np.array([0.0, np.inf, np.nan, 1e-45, 1.4e-40, 3.4028235e38, 448.0, 57344.0, 3.5], np.float32)])
    amax = torch.empty(1, dtype=torch.float32, device="cuda")
    scale = torch.empty(1, dtype=torch.float32, device="cuda")
    sinv = torch.empty(1, dtype=torch.float32, device="cuda")
    for fmt in (F.E4M3, F.E5M2):
        for v in vals:
            amax.fill_(float(v))
            fq.fp8_compute_scale(amax, fmt, scale, sinv)
            s_ref, si_ref = oracle.tensor_scale(v, int(fmt))
            assert f32bits(host(scale))[0] == f32bits(s_ref), (fmt, v)
            assert f32bits(host(sinv))[0] == f32bits(si_ref), (fmt, v)
    assert_status_ok()


def test_empty_and_all_zero_inputs():
    amax = torch.full((1,), 7.0, dtype=torch.float32, device="cuda")
    x0 = torch.empty((0, 128), dtype=torch.bfloat16, device="cuda")
    fq.fp8_amax(x0, amax)
    torch.cuda.synchronize()
    assert host(amax)[0] == 0.0
    q = torch.empty((0, 128), dtype=torch.uint8, device="cuda")
    s = torch.empty((0, 1), dtype=torch.float32, device="cuda")
    fq.fp8_quantize(x0, R.BLOCK_1x128, F.E4M3, None, amax, q, s)
    z = torch.zeros((256, 256), dtype=torch.bfloat16, device="cuda")
    for recipe in ALL_RECIPES:
        scale_np = np.float32(1.0) if recipe == R.TENSOR else None
        check_cast(z, recipe, F.E4M3, scale_np=scale_np)


def test_tiny_values_signed_zero_and_saturation():
    # tiny magnitudes round to +-0 with the sign kept; a stale (too large) scale saturates
    x = _x((256, 256), 500, sigma=1e-3, outliers=False)
    x[0, :8] = torch.tensor([1e-38, -1e-38, 1e-30, -1e-30, -0.0, 0.0, 2e-39, -2e-39], dtype=torch.bfloat16)
    for fmt in (F.E4M3, F.E5M2):
        check_cast(x, R.TENSOR, fmt, scale_np=np.float32(1.0))
        check_cast(x, R.TENSOR, fmt, scale_np=np.float32(3.0e5))      # saturates most elements
        check_cast(x, R.TENSOR, fmt, scale_np=np.float32(3.4028235e38))
        for recipe in (R.BLOCK_1x128, R.BLOCK_128x128, R.MX_1x32):
            check_cast(x, recipe, fmt)


def test_nan_inputs_stay_nan_and_are_ignored_by_amax():
    x = _x((128, 256), 600, outliers=False)
    x[3, 5] = float("nan")
    x[77, 200] = float("nan")
    xh = bits16(x)
    amax = torch.empty(1, dtype=torch.float32, device="cuda")
    fq.fp8_amax(x, amax)
    torch.cuda.synchronize()
    assert f32bits(host(amax))[0] == f32bits(oracle.amax(xh))
    qr, sr, qc, sc = fq.cast_transpose(x, R.BLOCK_1x128, F.E4M3)
    torch.cuda.synchronize()
    q_ref, s_ref = oracle.quantize_rowwise(xh, oracle.KIND_1x128, 0)
    got = host(qr)
    nan_ref = (q_ref & 0x7F) == 0x7F
    assert np.array_equal((got & 0x7F) == 0x7F, nan_ref)
    assert_bytes_equal(got[~nan_ref], q_ref[~nan_ref], "non-NaN bytes")
    assert_bytes_equal(f32bits(host(sr)), f32bits(s_ref), "scales (NaN ignored by block amax)")
