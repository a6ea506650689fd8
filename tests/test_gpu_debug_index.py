"""The debug library (kernels built with FP8Q_DEBUG_INDEX): every plain global access of
the GEMM (scale arrays, output and FP8-copy stores, the K-cut workspace and its counters)
and of the casts (scale arrays, MX scale atoms, the plain path's element stores) is checked
against its buffer's extent; an access out of range is skipped and reported as
FP8_ERR_INDEX, never made.  A stand-in for a memory checker: the calls below, over every
kernel variant and ragged shapes, must report nothing and give the release library's
results bit for bit.  The reporting path itself is checked with an index self-test that
touches no memory."""
import numpy as np
import pytest
import torch

import scaled_quantize_gemm_amax_gb300 as fq
from scaled_quantize_gemm_amax_gb300 import build as fqbuild
from scaled_quantize_gemm_amax_gb300 import workloads as wl
from gpu_util import R, F, require_gpu

pytestmark = pytest.mark.gpu
O = fq.OutDtype


@pytest.fixture(scope="module")
def libs():
    require_gpu()
    release = fq.load_library()
    debug = fq.load_library(fqbuild.build(debug=True))
    yield release, debug
    fq._lib = release


def _with(lib, fn):
    saved = fq._lib
    fq._lib = lib
    try:
        out = fn()
        torch.cuda.synchronize()
        st = fq.fp8_get_device_status()
    finally:
        fq._lib = saved
    return out, st


def test_index_self_test_reports_in_debug_only(libs):
    release, debug = libs
    _, st = _with(debug, lambda: fq.fp8_debug_index_check(4, 5))
    assert st == fq.Status.OK
    _, st = _with(debug, lambda: fq.fp8_debug_index_check(5, 5))
    assert st == fq.Status.ERR_INDEX
    _, st = _with(debug, lambda: fq.fp8_debug_index_check(-1, 5))
    assert st == fq.Status.ERR_INDEX
    _, st = _with(release, lambda: fq.fp8_debug_index_check(5, 5))
    assert st == fq.Status.OK


GEMMS = [
    # (ra, rb, M, N, K, out, fused): every kernel variant and work division
    (R.TENSOR, R.TENSOR, 4096, 4096, 512, O.FP32, False),          # pairs, stream-K
    (R.TENSOR, R.TENSOR, 256, 384, 4096, O.BF16, False),           # pairs, a sparse single wave cut in 8
    (R.TENSOR, R.TENSOR, 384, 640, 512, O.BF16, True),             # one CTA, fused FP8 copy of C
    (R.MX_1x32_TILED, R.MX_1x32_TILED, 2560, 2304, 8192, O.BF16, False),   # pairs, stream-K over one wave
    (R.MX_1x32_TILED, R.MX_1x32_TILED, 384, 640, 640, O.FP32, False),      # one CTA, ragged N tiles
    (R.BLOCK_1x128, R.BLOCK_128x128, 2048, 1536, 512, O.BF16, True),       # 256-deep stages, fused
    (R.BLOCK_1x128, R.BLOCK_128x128, 2048, 4096, 640, O.BF16, False),      # 256 x 160 tiles, last one 96 wide
    (R.BLOCK_1x128, R.BLOCK_128x128, 384, 768, 640, O.FP32, False),        # one CTA, 128-deep stages
    (R.BLOCK_1x128, R.BLOCK_1x128, 2048, 1536, 512, O.FP32, False),        # per-row B table on pairs
    (R.BLOCK_1x128, R.BLOCK_1x128, 512, 512, 8448, O.FP32, False),         # per-row B on one CTA
]


@pytest.mark.parametrize("ra,rb,m,n,k,out,fused", GEMMS)
def test_gemm_debug_checks_clean(libs, ra, rb, m, n, k, out, fused):
    release, debug = libs
    x = wl.normal_bf16((m, k), 5000 + m % 97, 1.0)
    w = wl.normal_bf16((n, k), 6000 + n % 89, 0.02)
    one = torch.ones(1, dtype=torch.float32, device="cuda")
    qa, sa, _, _ = fq.cast_transpose(x, ra, F.E4M3, one if ra == R.TENSOR else None, col=False)
    qb, sb, _, _ = fq.cast_transpose(w, rb, F.E4M3, one if rb == R.TENSOR else None, col=False)
    c_scale = torch.full((1,), 32.0, dtype=torch.float32, device="cuda")

    def run():
        if fused:
            return fq.scaled_gemm_amax(qa, F.E4M3, ra, sa, qb, F.E4M3, rb, sb, c_scale, out=out)
        return (fq.scaled_gemm(qa, F.E4M3, ra, sa, qb, F.E4M3, rb, sb, out=out),)

    ref, st = _with(release, run)
    assert st == fq.Status.OK
    got, st = _with(debug, run)
    assert st == fq.Status.OK, f"debug checks reported {st!r}"
    for a, b in zip(ref, got):
        if a is not None:
            assert torch.equal(a.view(torch.uint8), b.view(torch.uint8))


CASTS = [
    (R.TENSOR, (300, 517), False),            # plain path (ragged)
    (R.TENSOR, (384, 640), False),
    (R.BLOCK_1x128, (384, 640), False),
    (R.BLOCK_128x128, (256, 384), False),
    (R.MX_1x32, (160, 224), False),           # row-major E8M0, tiles hanging over both dims
    (R.MX_1x32_TILED, (384, 256), False),
    (R.BLOCK_1x128, (256, 384), True),        # binary32 inputs
    (R.BLOCK_128x128, (384, 256), True),
    (R.MX_1x32_TILED, (256, 640), True),
    (R.TENSOR, (200, 333), True),
]


@pytest.mark.parametrize("recipe,shape,f32", CASTS)
def test_cast_debug_checks_clean(libs, recipe, shape, f32):
    release, debug = libs
    x = wl.normal_bf16(shape, 7000 + shape[0], 1.0)
    if f32:
        x = x.float() * 1.0009765625   # off the BF16 grid
    one = torch.full((1,), 2.0, dtype=torch.float32, device="cuda")
    run = lambda: fq.cast_transpose(x, recipe, F.E4M3, one if recipe == R.TENSOR else None)
    ref, st = _with(release, run)
    assert st == fq.Status.OK
    got, st = _with(debug, run)
    assert st == fq.Status.OK, f"debug checks reported {st!r}"
    for a, b in zip(ref, got):
        assert torch.equal(a.view(torch.uint8), b.view(torch.uint8))
