"""GPU parity of the binary32-input cast (fp8_cast_transpose_f32) and amax
(fp8_amax_f32) against the oracle's binary32 quantizers, bit for bit: FP8 bytes of
both copies, every block scale (FP32 multipliers and E8M0 bytes) and amax_out.  The
inputs are general binary32 values (every mantissa bit in use), so a kernel that read
them through bfloat16 would differ."""
import numpy as np
import pytest
import torch

import oracle
import scaled_quantize_gemm_amax_gb300 as fq
from gpu_util import (R, F, KIND, MX_RECIPES, Guarded, assert_bytes_equal, assert_status_ok, f32bits, host,
                      oracle_scales_like, require_gpu)

pytestmark = pytest.mark.gpu


@pytest.fixture(scope="module", autouse=True)
def _gpu():
    require_gpu()


def f32_input(shape, seed, sigma=1.0, outliers=True):
    g = torch.Generator(device="cuda")
    g.manual_seed(seed)
    x = torch.randn(shape, generator=g, device="cuda") * sigma
    x *= torch.exp2(torch.randint(-4, 5, shape, generator=g, device="cuda").float())
    if outliers:
        flat = x.view(-1)
        idx = torch.randint(0, flat.numel(), (max(1, flat.numel() // 1000),), generator=g, device="cuda")
        flat[idx] *= 1000.0
    return x


def _check_scales(recipe, got, ref, what):
    if recipe in MX_RECIPES:
        assert_bytes_equal(got, ref, what)
    else:
        assert_bytes_equal(f32bits(got), f32bits(ref), what)


def check_cast_f32(x, recipe, fmt, row=True, col=True, guard=False):
    xh = host(x).astype(np.float32)
    rows, cols = xh.shape
    kind = KIND[recipe]
    scale_np = scale_t = None
    if recipe == R.TENSOR:
        scale_np, _ = oracle.tensor_scale(oracle.amax_f32(xh), int(fmt))
        scale_t = torch.tensor([scale_np], dtype=torch.float32, device="cuda")
    shp_r, dt_r = fq.scale_shape(recipe, rows, cols)
    shp_c, dt_c = fq.scale_shape(recipe, cols, rows)
    mk = (lambda shp, dt: Guarded(shp, dt)) if guard else (lambda shp, dt: None)
    bufs = {}
    outs = {}
    for name, shp, dt, want in (("q_row", (rows, cols), torch.uint8, row), ("s_row", shp_r, dt_r, row),
                                ("q_col", (cols, rows), torch.uint8, col), ("s_col", shp_c, dt_c, col),
                                ("amax", (1,), torch.float32, True)):
        if not want:
            outs[name] = None
            continue
        g = mk(shp, dt)
        if g is not None:
            bufs[name] = g
            outs[name] = g.t
        else:
            outs[name] = torch.full(shp, 0x5A if dt == torch.uint8 else 7.0, dtype=dt, device="cuda")
    fq.fp8_cast_transpose_f32(x, recipe, fmt, scale_t, outs["amax"], outs["q_row"], outs["s_row"], outs["q_col"],
                              outs["s_col"])
    torch.cuda.synchronize()
    assert_status_ok()
    for name, g in bufs.items():
        g.check(name)
    assert f32bits(host(outs["amax"]))[0] == f32bits(oracle.amax_f32(xh)), "amax_out"
    if row:
        q_ref, s_ref = oracle.quantize_rowwise_f32(xh, kind, int(fmt), scale_np)
        assert_bytes_equal(host(outs["q_row"]), q_ref, "q_row")
        _check_scales(recipe, host(outs["s_row"]), oracle_scales_like(recipe, s_ref, rows, cols), "s_row")
    if col:
        q_ref, s_ref = oracle.quantize_colwise_f32(xh, kind, int(fmt), scale_np)
        assert_bytes_equal(host(outs["q_col"]), q_ref, "q_col")
        _check_scales(recipe, host(outs["s_col"]), oracle_scales_like(recipe, s_ref, cols, rows), "s_col")


RECIPES = [R.TENSOR, R.BLOCK_1x128, R.BLOCK_128x128, R.MX_1x32, R.MX_1x32_TILED]


@pytest.mark.parametrize("recipe", RECIPES)
@pytest.mark.parametrize("fmt", [F.E4M3, F.E5M2])
@pytest.mark.parametrize("row,col", [(True, True), (True, False), (False, True)])
def test_cast_f32_multi_tile(recipe, fmt, row, col):
    # 3 x 5 tiles of 128 x 128
    check_cast_f32(f32_input((384, 640), 11 + int(recipe)), recipe, fmt, row, col)


@pytest.mark.parametrize("recipe,shape", [
    (R.TENSOR, (1000, 304)),     # rows % 16 != 0: the plain per-tensor kernel
    (R.TENSOR, (1008, 304)),     # the tiled kernel, ragged last tiles both ways
    (R.TENSOR, (136, 200)),      # cols % 16 != 0
    (R.MX_1x32, (160, 96)),      # tiles hanging over both edges, row-major E8M0
    (R.BLOCK_1x128, (128, 896)),
])
def test_cast_f32_ragged_shapes_and_guards(recipe, shape):
    check_cast_f32(f32_input(shape, 21), recipe, F.E4M3, guard=True)


@pytest.mark.parametrize("recipe", [R.BLOCK_128x128, R.TENSOR, R.MX_1x32_TILED])
def test_cast_f32_weight_size(recipe):
    # a 4096 x 4096 FP32 master weight ~ N(0, 0.02): 1024 tiles, several per CTA
    check_cast_f32(f32_input((4096, 4096), 31, 0.02, outliers=False), recipe, F.E4M3)


def test_cast_f32_special_values():
    x = f32_input((256, 256), 41)
    x[0, :128] = 0.0                       # an all-zero 1x128 block: scale 1
    x[1, 5] = float("inf")                 # an infinite amax: scale 1, inf saturates
    x[2, 7] = float("nan")                 # NaN is ignored by the amaxes, stays NaN
    x[3, 0:32] = 1e-40                     # subnormal binary32 values
    x[4, 64] = 3.0e38                      # near FLT_MAX
    xh = host(x).astype(np.float32)
    for recipe in (R.BLOCK_1x128, R.MX_1x32):
        q, s, qc, sc = fq.cast_transpose(x, recipe, F.E4M3)
        torch.cuda.synchronize()
        assert_status_ok()
        for got, (q_ref, s_ref), what in ((q, oracle.quantize_rowwise_f32(xh, KIND[recipe], 0), "row"),
                                          (qc, oracle.quantize_colwise_f32(xh, KIND[recipe], 0), "col")):
            g, r = host(got), q_ref
            nan_g = (g & 0x7F) == 0x7F
            nan_r = (r & 0x7F) == 0x7F
            assert np.array_equal(nan_g, nan_r), f"{recipe.name} {what}: NaN positions"
            assert_bytes_equal(np.where(nan_r, 0, g), np.where(nan_r, 0, r), f"{recipe.name} {what}")


@pytest.mark.parametrize("n", [1, 3, 4, 4099, 1 << 20, (1 << 22) + 7])
def test_amax_f32_matches_oracle(n):
    x = f32_input((n,), 50 + n % 97, outliers=True)
    if n > 10:
        x[n // 2] = float("nan")
        x[n // 3] = -float(np.float32(12345.678))
    amax = torch.full((1,), 9.0, dtype=torch.float32, device="cuda")
    fq.fp8_amax_f32(x.view(1, n), amax)
    torch.cuda.synchronize()
    assert_status_ok()
    assert f32bits(host(amax))[0] == f32bits(oracle.amax_f32(host(x).astype(np.float32)))
