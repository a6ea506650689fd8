"""GPU parity of the cast-transpose on seeded random shapes: for every recipe, rows and
columns drawn within the recipe's blocking rule (per-tensor: any size, so both the tiled
and the plain path; MXFP8 with row-major scales: multiples of 32; the others: multiples of
128), a random choice of copies (row, column or both), format and value scale, every
output byte and scale compared with the oracle bit for bit (the amax too), for BF16 and
binary32 inputs."""
import numpy as np
import pytest

from scaled_quantize_gemm_amax_gb300 import workloads as wl
from gpu_util import R, F, check_cast, require_gpu
from test_gpu_quantize_f32 import check_cast_f32, f32_input

pytestmark = pytest.mark.gpu

RECIPES = [R.TENSOR, R.BLOCK_1x128, R.BLOCK_128x128, R.MX_1x32, R.MX_1x32_TILED]


@pytest.fixture(scope="module", autouse=True)
def _gpu():
    require_gpu()


def _dims(rng, recipe, row, col):
    if recipe == R.TENSOR:
        return int(rng.integers(1, 1100)), int(rng.integers(1, 1100))
    if recipe == R.MX_1x32:
        return int(rng.integers(1, 40)) * 32, int(rng.integers(1, 40)) * 32
    return int(rng.integers(1, 11)) * 128, int(rng.integers(1, 11)) * 128


def _cases(n_per_recipe=6, seed=3112026):
    rng = np.random.default_rng(seed)
    out = []
    for ri, rec in enumerate(RECIPES):
        for j in range(n_per_recipe):
            row, col = [(True, True), (True, False), (False, True)][int(rng.integers(0, 3))]
            r, c = _dims(rng, rec, row, col)
            fmt = F.E4M3 if rng.random() < 0.6 else F.E5M2
            sigma = float(10.0 ** rng.uniform(-3, 2))
            out.append(pytest.param(rec, r, c, row, col, fmt, sigma, 2000 + 10 * ri + j,
                                    id=f"{rec.name}-{r}x{c}-{'r' if row else ''}{'c' if col else ''}-{fmt.name}"))
    return out


@pytest.mark.parametrize("recipe,rows,cols,row,col,fmt,sigma,seed", _cases())
def test_cast_random_shapes(recipe, rows, cols, row, col, fmt, sigma, seed):
    x = wl.normal_bf16((rows, cols), seed, sigma)
    check_cast(x, recipe, fmt, row=row, col=col)


def _f32_cases(n=8, seed=3122026):
    rng = np.random.default_rng(seed)
    out = []
    for j in range(n):
        rec = RECIPES[j % len(RECIPES)]
        row, col = [(True, True), (True, False), (False, True)][int(rng.integers(0, 3))]
        r, c = _dims(rng, rec, row, col)
        fmt = F.E4M3 if rng.random() < 0.6 else F.E5M2
        out.append(pytest.param(rec, r, c, row, col, fmt, 2100 + j,
                                id=f"f32-{rec.name}-{r}x{c}-{'r' if row else ''}{'c' if col else ''}-{fmt.name}"))
    return out


@pytest.mark.parametrize("recipe,rows,cols,row,col,fmt,seed", _f32_cases())
def test_cast_f32_random_shapes(recipe, rows, cols, row, col, fmt, seed):
    # binary32 input (values not BF16-representable, a few outliers), the oracle quantizing
    # the same binary32 words; outputs between guard regions
    check_cast_f32(f32_input((rows, cols), seed), recipe, fmt, row, col, guard=True)
