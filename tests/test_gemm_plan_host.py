"""The GEMM's dispatch and work division as host logic, on the CPU (no GPU needed):
fp8_debug_gemm_plan runs the same functions fp8_scaled_gemm uses to pick the kernel
variant, the tile width and, on CTA pairs, stream-K shares or the K-range cut of a sparse
last wave.  Each case states the rule it checks, for a 152-SM part with 76 resident pairs
unless it says otherwise."""
import pytest

import scaled_quantize_gemm_amax_gb300 as fq

R, O = fq.Recipe, fq.OutDtype
TENSOR, BLK_A, BLK_B, MX = R.TENSOR, R.BLOCK_1x128, R.BLOCK_128x128, R.MX_1x32_TILED


def plan(ra, rb, out, m, n, k, fused=False, num_sms=152, resident_pairs=76):
    return fq.fp8_debug_gemm_plan(ra, rb, out, m, n, k, fused, num_sms, resident_pairs)


def test_per_tensor_4096_streamk():
    # 256 tiles on 76 pairs: three full waves and 28 tiles -> two whole waves, then shares
    p = plan(TENSOR, TENSOR, O.BF16, 4096, 4096, 4096)
    assert p == {"pair": 1, "variant": 0, "block_n": 256, "tiles": 256, "streamk": 1, "split": 1, "tail0": 152,
                 "launched": 76}


def test_per_tensor_8192_last_wave_cut():
    # 1024 tiles: 13 full waves and 36 tiles; K >= 8192 -> those tiles cut into 76 / 36 = 2 ranges
    p = plan(TENSOR, TENSOR, O.BF16, 8192, 8192, 8192)
    assert (p["streamk"], p["split"], p["tail0"], p["launched"]) == (0, 2, 988, 76)


def test_mx_one_full_wave_short_k_whole_tiles():
    # 128 tiles: one full wave and 52; K = 4096 -> neither shares nor a cut (52 > 76 / 2)
    p = plan(MX, MX, O.BF16, 2048, 4096, 4096)
    assert (p["variant"], p["tiles"], p["streamk"], p["split"], p["tail0"], p["launched"]) == (3, 128, 0, 1, 128, 76)


def test_mx_one_full_wave_long_k_streamk():
    # 90 tiles, one full wave, K = 8192 -> every tile shared out
    p = plan(MX, MX, O.BF16, 2560, 2304, 8192)
    assert (p["streamk"], p["tail0"], p["launched"]) == (1, 0, 76)


def test_single_partial_wave_cut_into_ranges():
    # one 256 x 256 tile: a sparse single wave -> min(76, K / 128, 8) = 8 ranges on 8 pairs
    p = plan(TENSOR, TENSOR, O.FP32, 256, 256, 4096)
    assert (p["tiles"], p["split"], p["tail0"], p["launched"]) == (1, 8, 0, 8)
    # K / 128 = 2 caps the ranges
    assert plan(TENSOR, TENSOR, O.FP32, 256, 256, 256)["split"] == 2


def test_fewer_resident_pairs():
    # 60 resident pairs: 256 tiles are four full waves and 16 -> no shares (more than three
    # waves), no cut (K < 8192 with full waves)
    p = plan(TENSOR, TENSOR, O.BF16, 4096, 4096, 4096, resident_pairs=60)
    assert (p["streamk"], p["split"], p["launched"]) == (0, 1, 60)


def test_blockwise_variants():
    # 1x128 x 128x128: 256-deep stages on pairs (K / 128 even), never cut
    p = plan(BLK_A, BLK_B, O.BF16, 4096, 4096, 4096)
    assert (p["pair"], p["variant"], p["block_n"], p["tiles"], p["streamk"], p["split"], p["launched"]) == \
        (1, 5, 128, 512, 0, 1, 76)
    # K / 128 odd, BF16 out: 256 x 160 pair tiles (26 a row of tiles, the last 96 wide)
    p = plan(BLK_A, BLK_B, O.BF16, 4096, 4096, 4224)
    assert (p["pair"], p["variant"], p["block_n"], p["tiles"]) == (1, 7, 160, 16 * 26)
    # ... not with FP32 output or a fused output cast: one CTA per 128 x 128 tile
    for out, fused in ((O.FP32, False), (O.BF16, True)):
        p = plan(BLK_A, BLK_B, out, 4096, 4096, 4224, fused=fused)
        assert (p["pair"], p["variant"], p["block_n"], p["tiles"], p["launched"]) == (0, 1, 128, 32 * 32, 152)
    # M % 256 != 0 with K / 128 even: one CTA, 256-deep stages
    p = plan(BLK_A, BLK_B, O.BF16, 384, 512, 1024)
    assert (p["pair"], p["variant"], p["tiles"]) == (0, 5, 3 * 4)


def test_weight_gradient_variants():
    # 1x128 x 1x128 (per-row B scales): pairs while K / 128 is even and at most 64
    assert plan(BLK_A, BLK_A, O.FP32, 4096, 4096, 4096)["variant"] == 6
    assert plan(BLK_A, BLK_A, O.FP32, 512, 1024, 8192)["variant"] == 6
    p = plan(BLK_A, BLK_A, O.FP32, 512, 512, 8448)
    assert (p["pair"], p["variant"]) == (0, 4)


def test_single_cta_kinds():
    # M % 256 != 0: one CTA per 128-row tile
    p = plan(TENSOR, TENSOR, O.BF16, 384, 640, 512)
    assert (p["pair"], p["variant"], p["block_n"], p["tiles"], p["launched"]) == (0, 0, 256, 3 * 3, 9)
    p = plan(MX, MX, O.FP32, 640, 1024, 512)
    assert (p["pair"], p["variant"], p["tiles"]) == (0, 3, 5 * 4)


def test_plan_argument_checks():
    with pytest.raises(fq.FP8Error) as e:
        plan(TENSOR, MX, O.BF16, 256, 256, 256)
    assert e.value.status == fq.Status.ERR_UNSUPPORTED
    with pytest.raises(fq.FP8Error) as e:
        plan(TENSOR, TENSOR, O.BF16, 256, 200, 256)
    assert e.value.status == fq.Status.ERR_SHAPE
