"""GPU parity of the scaled FP8 GEMM on seeded random shapes: M, N, K drawn as multiples of
128 up to 2560 (M a multiple of 256 half of the time, so that both the single-CTA and the
CTA-pair kernels, the K-range cut of a sparse last wave, the 160-wide blockwise tiles for
odd K / 128 and the per-row-B table are all reached), every pairing, BF16 or FP32 output
drawn too.  Each case is compared with the oracle on every 7th row of C within the stated
bar, so that a dispatch or tiling mistake at some size boundary shows up."""
import numpy as np
import pytest

import scaled_quantize_gemm_amax_gb300 as fq
from scaled_quantize_gemm_amax_gb300 import workloads as wl
from gpu_util import R, F, require_gpu
from test_gpu_gemm import gemm_check

pytestmark = pytest.mark.gpu

PAIRINGS = [(R.TENSOR, R.TENSOR), (R.BLOCK_1x128, R.BLOCK_128x128), (R.BLOCK_1x128, R.BLOCK_1x128),
            (R.MX_1x32_TILED, R.MX_1x32_TILED)]


@pytest.fixture(scope="module", autouse=True)
def _gpu():
    require_gpu()


def _cases(n_per_pairing=8, seed=20261203):
    rng = np.random.default_rng(seed)
    out = []
    for pi, (ra, rb) in enumerate(PAIRINGS):
        for j in range(n_per_pairing):
            step_m = 256 if rng.random() < 0.5 else 128
            m = int(rng.integers(1, 2560 // step_m + 1)) * step_m
            n = int(rng.integers(1, 21)) * 128
            k = int(rng.integers(1, 21)) * 128
            out_fp32 = bool(rng.random() < 0.4)
            out.append(pytest.param(ra, rb, m, n, k, out_fp32, 1000 + 16 * pi + j,
                                    id=f"{ra.name}-{rb.name}-{m}x{n}x{k}-{'f32' if out_fp32 else 'bf16'}"))
    return out


@pytest.mark.parametrize("ra,rb,m,n,k,out_fp32,seed", _cases())
def test_gemm_random_shapes(ra, rb, m, n, k, out_fp32, seed):
    x = wl.normal_bf16((m, k), seed, 1.0)
    w = wl.normal_bf16((n, k), seed + 500, 0.02)
    rows = np.arange(0, m, 7)
    gemm_check(x, w, ra, rb, F.E4M3, F.E4M3, out=fq.OutDtype.FP32 if out_fp32 else fq.OutDtype.BF16, rows=rows)
