"""GPU parity of the scaled FP8 GEMM against the oracle (dequantize exactly, float64
matmul) within the stated bar: ||C - C_ref||_F / ||C_ref||_F <= 1e-2 and
|C - C_ref|[m, n] <= 2e-2 * ||deq(A)[m, :]|| * ||deq(B)[n, :]|| / sqrt(K).

The oracle quantizes the same BF16 bytes itself (no oracle input comes from the
GPU); the GPU's FP8 bytes are additionally checked equal to the oracle's."""
import numpy as np
import pytest
import torch

import oracle
import scaled_quantize_gemm_amax_gb300 as fq
from scaled_quantize_gemm_amax_gb300 import workloads as wl
from gpu_util import R, F, KIND, assert_bytes_equal, assert_status_ok, bits16, host, require_gpu, tile_spread

pytestmark = pytest.mark.gpu

REL_FRO = 1e-2


@pytest.fixture(scope="module", autouse=True)
def _gpu():
    require_gpu()


def _quant_gpu(x, recipe, fmt, scale_np):
    scale_t = None
    if recipe == R.TENSOR:
        scale_t = torch.tensor([scale_np], dtype=torch.float32, device="cuda")
    q, s, _, _ = fq.cast_transpose(x, recipe, fmt, scale_t, None, row=True, col=False)
    return q, s


def _quant_oracle(xh, recipe, fmt):
    scale_np = None
    if recipe == R.TENSOR:
        scale_np, _ = oracle.tensor_scale(oracle.amax(xh), int(fmt))
    q, s = oracle.quantize_rowwise(xh, KIND[recipe], int(fmt), scale_np)
    return q, s, scale_np


def _oracle_recipe(recipe):
    return KIND[recipe]


def gemm_check(x, w, ra, rb, fa, fb, out=fq.OutDtype.BF16, rows=None):
    """Quantize x [M, K] and w [N, K] on both sides, run the GEMM, compare.

    rows: compare only these rows of C (all columns) -- for large shapes."""
    xh, wh = bits16(x), bits16(w)
    qa_ref, sa_ref, sca = _quant_oracle(xh, ra, fa)
    qb_ref, sb_ref, scb = _quant_oracle(wh, rb, fb)
    qa, sa = _quant_gpu(x, ra, fa, sca)
    qb, sb = _quant_gpu(w, rb, fb, scb)
    c = fq.scaled_gemm(qa, fa, ra, sa, qb, fb, rb, sb, out=out)
    torch.cuda.synchronize()
    assert_status_ok()
    assert_bytes_equal(host(qa), qa_ref, "A bytes")
    assert_bytes_equal(host(qb), qb_ref, "B bytes")
    c_gpu = host(c.float()).astype(np.float64)
    ka, kb = _oracle_recipe(ra), _oracle_recipe(rb)
    deq_b = oracle.dequantize(qb_ref, kb, int(fb), sb_ref)
    if rows is None:
        deq_a = oracle.dequantize(qa_ref, ka, int(fa), sa_ref)
        c_ref = deq_a @ deq_b.T
        c_cmp = c_gpu
    else:
        rows = np.asarray(rows)
        sa_rows = sa_ref[rows] if ka in (oracle.KIND_1x128, oracle.KIND_MX) else sa_ref
        deq_a = oracle.dequantize(qa_ref[rows], ka, int(fa), sa_rows)
        c_ref = deq_a @ deq_b.T
        c_cmp = c_gpu[rows]
    rel, worst = oracle.gemm_tolerance_check(c_cmp, c_ref, deq_a, deq_b)
    assert rel <= REL_FRO, f"relative Frobenius error {rel:.3e}"
    assert worst <= 1.0, f"max-abs bound exceeded by x{worst:.3f}"
    return rel, worst


PAIRS = [(R.TENSOR, R.TENSOR), (R.BLOCK_1x128, R.BLOCK_128x128), (R.BLOCK_1x128, R.BLOCK_1x128),
         (R.MX_1x32_TILED, R.MX_1x32_TILED)]


@pytest.mark.parametrize("ra,rb", PAIRS)
def test_gemm_small_single_tile(ra, rb):
    x = wl.normal_bf16((128, 128), 10, 1.0)
    w = wl.normal_bf16((128, 128), 11, 0.02)
    gemm_check(x, w, ra, rb, F.E4M3, F.E4M3)


@pytest.mark.parametrize("ra,rb", PAIRS)
@pytest.mark.parametrize("fa,fb", [(F.E4M3, F.E4M3), (F.E5M2, F.E4M3), (F.E4M3, F.E5M2)])
def test_gemm_multi_tile_formats(ra, rb, fa, fb):
    # 3 x 2-or-4 tiles, 5 K blocks; N = 512 is not a multiple of every tile width
    x = wl.normal_bf16((384, 640), 20, 1.0)
    w = wl.normal_bf16((512, 640), 21, 0.02)
    gemm_check(x, w, ra, rb, fa, fb)


@pytest.mark.parametrize("ra,rb", PAIRS)
def test_gemm_fp32_output_and_n_tail(ra, rb):
    # N = 384: the 256-wide tiles hang over N by half a tile
    x = wl.normal_bf16((256, 512), 30, 1.0)
    w = wl.normal_bf16((384, 512), 31, 1e-3)
    gemm_check(x, w, ra, rb, F.E5M2, F.E4M3, out=fq.OutDtype.FP32)


def test_gemm_config1_per_tensor_256():
    a, b = wl.cfg1_tensor_current("cuda")
    gemm_check(a, b, R.TENSOR, R.TENSOR, F.E4M3, F.E4M3)


def test_gemm_config2_blockwise_4096_full():
    x, w = wl.cfg2_blockwise("cuda")
    rel, worst = gemm_check(x, w, R.BLOCK_1x128, R.BLOCK_128x128, F.E4M3, F.E4M3)
    print(f"cfg2 rel_fro={rel:.3e} worst={worst:.3f}")


@pytest.mark.parametrize("name", ["qkv", "down"])
def test_gemm_config3_mx_sampled_rows(name):
    x, w = wl.cfg3_mx(name, "cuda")
    rng = np.random.default_rng(3)
    rows = np.unique(np.concatenate([[0, x.shape[0] - 1], rng.integers(0, x.shape[0], 126)]))
    gemm_check(x, w, R.MX_1x32_TILED, R.MX_1x32_TILED, F.E4M3, F.E4M3, rows=rows)


def test_gemm_k_zero_writes_zeros():
    a = torch.empty((128, 0), dtype=torch.uint8, device="cuda")
    b = torch.empty((256, 0), dtype=torch.uint8, device="cuda")
    s = torch.ones(1, dtype=torch.float32, device="cuda")
    c = torch.full((128, 256), 5.0, dtype=torch.bfloat16, device="cuda")
    fq.fp8_scaled_gemm(a, F.E4M3, R.TENSOR, s, b, F.E4M3, R.TENSOR, s, c)
    torch.cuda.synchronize()
    assert torch.count_nonzero(c).item() == 0


@pytest.mark.parametrize("ra,rb", PAIRS)
@pytest.mark.parametrize("m,n,k", [(256, 256, 128), (512, 640, 384), (768, 384, 256)])
def test_gemm_cta_pair_tiles(ra, rb, m, n, k):
    # M a multiple of 256: 2-CTA pairs (blockwise with K = 128 and 384: 160-wide pair tiles
    # with BF16 output, single CTAs with FP32 output)
    x = wl.normal_bf16((m, k), 40, 1.0)
    w = wl.normal_bf16((n, k), 41, 0.02)
    gemm_check(x, w, ra, rb, F.E4M3, F.E5M2 if k == 384 else F.E4M3,
               out=fq.OutDtype.FP32 if m == 768 else fq.OutDtype.BF16)


@pytest.mark.parametrize("m,n,k,out", [
    (2048, 1536, 512, fq.OutDtype.BF16),    # CTA pairs: 96 tiles of 256x128, more than pairs
    (2048, 1408, 512, fq.OutDtype.BF16),    # CTA pairs, N % 256 == 128
    (512, 256, 2048, fq.OutDtype.BF16),     # a long K that wraps the stage ring many times
    (768, 1024, 640, fq.OutDtype.FP32),     # odd K blocks, FP32 output: single CTAs
    (1536, 2304, 1152, fq.OutDtype.BF16),   # odd K blocks, BF16 output: 90 pair tiles 160 wide
])
def test_gemm_blockwise_pairs_many_tiles(m, n, k, out):
    # blockwise with M % 256 == 0: CTA pairs with 256-deep stages when K / 128 is even;
    # otherwise 160-wide pair tiles with 128-deep stages (BF16 output) or single CTAs
    # (FP32 output); each pair (CTA) walks several tiles
    x = wl.normal_bf16((m, k), 50, 1.0)
    w = wl.normal_bf16((n, k), 51, 0.02)
    gemm_check(x, w, R.BLOCK_1x128, R.BLOCK_128x128, F.E4M3, F.E4M3, out=out)


def _block_spread(t, seed):
    """Multiply each 1x128 block of t by its own power of two (exact in BF16), so that a
    scale taken from the wrong row, column or k-block is far off."""
    r, c = t.shape
    e = (torch.arange(r, device=t.device)[:, None] * 3 + torch.arange(c // 128, device=t.device)[None, :] * 5 + seed) % 7 - 3
    return t * torch.exp2(e.float()).repeat_interleave(128, dim=1).to(t.dtype)


@pytest.mark.parametrize("m,n,k,out,spread", [
    (2048, 1536, 512, fq.OutDtype.FP32, True),    # CTA pairs: 96 tiles, some pairs refill their B-scale table
    (4096, 2048, 256, fq.OutDtype.FP32, True),    # two k-blocks (the shortest pair K), 256 tiles: 3-4 a pair
    (1280, 768, 1024, fq.OutDtype.FP32, True),    # M = 5 x 256
    (1280, 768, 1024, fq.OutDtype.BF16, False),   # BF16 output
    (512, 1024, 8192, fq.OutDtype.FP32, True),    # 64 k-blocks: the largest table
    (512, 512, 8448, fq.OutDtype.FP32, True),     # 66 k-blocks: past the table, single CTAs
])
def test_gemm_blockwise_rows_b_many_tiles(m, n, k, out, spread):
    # 1x128 x 1x128 (the weight-gradient pairing: a scale per row of B and k-block): CTA
    # pairs reading B's scales from a per-tile table when K / 128 is even and at most 64,
    # single CTAs otherwise.  The spread inputs use FP32 output: with their range, the
    # exact product rounded to BF16 alone exceeds the max-abs bar (x1.04 at 1280x768x1024,
    # computed with the oracle), so BF16 output is checked on plain normal inputs.
    x = wl.normal_bf16((m, k), 60, 1.0)
    w = wl.normal_bf16((n, k), 61, 0.02)
    if spread:
        x, w = _block_spread(x, 1), _block_spread(w, 4)
    gemm_check(x, w, R.BLOCK_1x128, R.BLOCK_1x128, F.E4M3, F.E4M3, out=out)


@pytest.mark.parametrize("m,n,k", [
    (512, 512, 4096),      # CTA pairs, the bench's K: 32 k-blocks a tile
    (2048, 1536, 512),     # CTA pairs, several tiles a pair
    (384, 512, 1024),      # M % 256 != 0: single CTAs
    (512, 768, 640),       # K / 128 odd: single CTAs, 128-deep stages
])
def test_gemm_blockwise_128x128_b_tile_spread(m, n, k):
    # 1x128 x 128x128 with every 1x128 block of A and every 128x128 tile of B scaled by
    # its own power of two: a B scale taken from the wrong column block or k-block (or an
    # A scale from the wrong row or k-block) is off by 2x-64x and fails the bar, at the
    # bench's K too.  FP32 output: with this range the exact product rounded to BF16 uses
    # most of the max-abs bar by itself.
    x = tile_spread(wl.normal_bf16((m, k), 70, 1.0), 1, 128, 1, 3)
    w = tile_spread(wl.normal_bf16((n, k), 71, 0.02), 128, 128, 4, 3)
    gemm_check(x, w, R.BLOCK_1x128, R.BLOCK_128x128, F.E4M3, F.E4M3, out=fq.OutDtype.FP32)


@pytest.mark.parametrize("m,n,k,spread", [
    (2048, 4096, 640, False),    # 26 tiles of 160 columns a row of tiles, the last one 96 wide
    (4096, 2176, 384, True),     # last tile 96 wide; thread slices spanning two 128-column blocks
    (2048, 2560, 1152, True),    # N a multiple of 160: 128 tiles, two per pair
    (1536, 2304, 1152, False),   # 15 tiles a row, the last one 64 wide
    (512, 640, 384, False),      # a single wave
])
def test_gemm_blockwise_160_wide_tiles(m, n, k, spread):
    # 1x128 x 128x128 with BF16 output, M % 256 == 0 and K / 128 odd: 256 x 160 pair tiles
    # with 128-deep stages.  Spread: every 128x128 tile of B scaled by its own power of two
    # (2^-2..2^2), so that a B scale from the wrong column block or k-block moves the
    # relative Frobenius error far past 1e-2; the exact product rounded to BF16 alone uses
    # 0.70 / 0.62 of the max-abs bar at these shapes (oracle).
    x = wl.normal_bf16((m, k), 74, 1.0)
    w = wl.normal_bf16((n, k), 75, 0.02)
    if spread:
        w = tile_spread(w, 128, 128, 4, 2)
    gemm_check(x, w, R.BLOCK_1x128, R.BLOCK_128x128, F.E4M3, F.E4M3)


@pytest.mark.parametrize("m,n,k", [(2048, 4096, 640), (4096, 1920, 1152)])
def test_gemm_blockwise_160_matches_single_cta(m, n, k):
    # K / 128 odd: the 160-wide pair tiles (BF16 output) and the single-CTA 128 x 128 tiles
    # (FP32 output) add the same promoted partials in the same k-block order, so the BF16
    # result is the FP32 one rounded to nearest even, bit for bit.
    x = tile_spread(wl.normal_bf16((m, k), 76, 1.0), 1, 128, 2, 2)
    w = tile_spread(wl.normal_bf16((n, k), 77, 0.02), 128, 128, 3, 2)
    qa, sa, _, _ = fq.cast_transpose(x, R.BLOCK_1x128, F.E4M3, row=True, col=False)
    qb, sb, _, _ = fq.cast_transpose(w, R.BLOCK_128x128, F.E4M3, row=True, col=False)
    c16 = fq.scaled_gemm(qa, F.E4M3, R.BLOCK_1x128, sa, qb, F.E4M3, R.BLOCK_128x128, sb, out=fq.OutDtype.BF16)
    c32 = fq.scaled_gemm(qa, F.E4M3, R.BLOCK_1x128, sa, qb, F.E4M3, R.BLOCK_128x128, sb, out=fq.OutDtype.FP32)
    torch.cuda.synchronize()
    assert_status_ok()
    assert torch.equal(c16.view(torch.int16), c32.to(torch.bfloat16).view(torch.int16))


@pytest.mark.parametrize("m,n,k", [
    (512, 512, 4096),      # CTA pairs, 128 MX blocks along K
    (1024, 768, 512),      # CTA pairs, N % 256 == 0 over several tiles
    (384, 640, 640),       # M % 256 != 0: single CTAs, N tail
])
def test_gemm_mx_exponent_spread(m, n, k):
    # MXFP8 with every 1x32 block of both operands scaled by 2^e, e in [-8, 8]: each
    # block's E8M0 exponent differs from its neighbours', so an exponent applied to the
    # wrong 32-deep block, row or column is off by 2^(1..16).
    x = tile_spread(wl.normal_bf16((m, k), 72, 1.0), 1, 32, 2, 8)
    w = tile_spread(wl.normal_bf16((n, k), 73, 0.02), 1, 32, 5, 8)
    gemm_check(x, w, R.MX_1x32_TILED, R.MX_1x32_TILED, F.E4M3, F.E4M3, out=fq.OutDtype.FP32)
