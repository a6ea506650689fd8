"""GPU parity of fp8_cast_transpose_multi: several casts (different recipes, formats,
shapes, with and without amax) in one launch, every output compared with the oracle
bit for bit, and with the single-job entry point."""
import numpy as np
import pytest
import torch

import oracle
import scaled_quantize_gemm_amax_gb300 as fq
from scaled_quantize_gemm_amax_gb300 import workloads as wl
from gpu_util import (R, F, KIND, assert_bytes_equal, assert_status_ok, bits16, f32bits, host, oracle_scales_like,
                      require_gpu)

pytestmark = pytest.mark.gpu


@pytest.fixture(scope="module", autouse=True)
def _gpu():
    require_gpu()


def check_job(x, recipe, fmt, scale_np, outs, amax_t):
    xh = bits16(x)
    rows, cols = xh.shape
    kind = KIND[recipe]
    qr, sr, qc, sc = outs
    if amax_t is not None:
        assert f32bits(host(amax_t))[0] == f32bits(oracle.amax(xh))[0], "amax_out"
    q_ref, s_ref = oracle.quantize_rowwise(xh, kind, int(fmt), scale_np)
    assert_bytes_equal(host(qr), q_ref, f"{recipe.name} q_row")
    s_ref = oracle_scales_like(recipe, s_ref, rows, cols)
    got = host(sr)
    assert_bytes_equal(got if got.dtype == np.uint8 else f32bits(got), s_ref if s_ref.dtype == np.uint8 else f32bits(s_ref),
                       f"{recipe.name} s_row")
    q_ref, s_ref = oracle.quantize_colwise(xh, kind, int(fmt), scale_np)
    assert_bytes_equal(host(qc), q_ref, f"{recipe.name} q_col")
    s_ref = oracle_scales_like(recipe, s_ref, cols, rows)
    got = host(sc)
    assert_bytes_equal(got if got.dtype == np.uint8 else f32bits(got), s_ref if s_ref.dtype == np.uint8 else f32bits(s_ref),
                       f"{recipe.name} s_col")


def test_cast_multi_four_recipes():
    xs = [wl.normal_bf16((384, 256), 80, 1.0), wl.normal_bf16((256, 512), 81, 0.02),
          wl.normal_bf16((256, 384), 82, 3.0), wl.normal_bf16((512, 128), 83, 1.0)]
    xs[0][:, 7] *= 100.0
    recipes = [R.BLOCK_1x128, R.BLOCK_128x128, R.MX_1x32_TILED, R.TENSOR]
    fmts = [F.E4M3, F.E4M3, F.E5M2, F.E5M2]
    scale_np = oracle.tensor_scale(oracle.amax(bits16(xs[3])), int(F.E5M2))[0]
    scales = [None, None, None, torch.tensor([scale_np], dtype=torch.float32, device="cuda")]
    amaxes = [torch.full((1,), 7.0, device="cuda"), None, torch.full((1,), 7.0, device="cuda"),
              torch.full((1,), 7.0, device="cuda")]
    outs = fq.cast_transpose_multi(list(zip(xs, recipes, fmts, scales, amaxes)))
    torch.cuda.synchronize()
    assert_status_ok()
    for x, r, f, sc, am, o in zip(xs, recipes, fmts, scales, amaxes, outs):
        check_job(x, r, f, scale_np if r == R.TENSOR else None, o, am)


def test_cast_multi_equals_single_calls_on_the_blockwise_workload():
    # the activation / weight pair of the blockwise fprop workload, in one launch
    x, w = wl.cfg2_blockwise("cuda")
    (mx_, ms_, mxt, mst), (mw, mws, mwt, mwst) = fq.cast_transpose_multi(
        [(x, R.BLOCK_1x128, F.E4M3, None, None), (w, R.BLOCK_128x128, F.E4M3, None, None)])
    sx = fq.cast_transpose(x, R.BLOCK_1x128, F.E4M3)
    sw = fq.cast_transpose(w, R.BLOCK_128x128, F.E4M3)
    torch.cuda.synchronize()
    assert_status_ok()
    for a, b in zip((mx_, ms_, mxt, mst, mw, mws, mwt, mwst), sx + sw):
        assert torch.equal(a.view(torch.uint8), b.view(torch.uint8))


@pytest.mark.parametrize("recipes,fmts,shapes", [
    ((R.BLOCK_1x128, R.BLOCK_128x128), (F.E4M3, F.E5M2), ((384, 640), (256, 384))),
    ((R.BLOCK_1x128, R.BLOCK_128x128), (F.E4M3, F.E4M3), ((2048, 1536), (1536, 2048))),
    ((R.MX_1x32_TILED, R.MX_1x32_TILED), (F.E4M3, F.E5M2), ((256, 384), (384, 256))),
    ((R.TENSOR, R.TENSOR), (F.E5M2, F.E4M3), ((128, 512), (384, 384))),
])
def test_cast_multi_two_job_pairings(recipes, fmts, shapes):
    # Two jobs whose recipes form a common pairing run in a kernel compiled for that pair
    # (each tile reads its job's parameters at fixed places); job 1's tiles follow job 0's
    # on every CTA, so the per-job amax hand-over is exercised where a CTA holds both.
    xs = [wl.normal_bf16(shapes[0], 84, 1.0), wl.normal_bf16(shapes[1], 85, 0.5)]
    xs[1][:, 3] *= 50.0
    scales, scale_nps = [], []
    for x, r, f in zip(xs, recipes, fmts):
        if r == R.TENSOR:
            s_np = oracle.tensor_scale(oracle.amax(bits16(x)), int(f))[0]
            scales.append(torch.tensor([s_np], dtype=torch.float32, device="cuda"))
            scale_nps.append(s_np)
        else:
            scales.append(None)
            scale_nps.append(None)
    amaxes = [torch.full((1,), 7.0, device="cuda"), torch.full((1,), 7.0, device="cuda")]
    outs = fq.cast_transpose_multi(list(zip(xs, recipes, fmts, scales, amaxes)))
    torch.cuda.synchronize()
    assert_status_ok()
    for x, r, f, s_np, am, o in zip(xs, recipes, fmts, scale_nps, amaxes, outs):
        check_job(x, r, f, s_np, o, am)


def test_cast_two_with_a_weight_above_the_byte_transpose_limit():
    # A 128x128 job of 16384 x 10240 (10240 tiles, more than 64 a CTA on 152 SMs) quantizes
    # its column copy from the BF16 tile; a small one transposes its row copy's bytes.  Both
    # beside a 1x128 job in the pairing kernel; sampled 128x128 tiles of the large job (each
    # tile's bytes and scale depend on that tile alone) and the whole small jobs against the
    # oracle.
    x = wl.normal_bf16((512, 384), 86, 1.0)
    big = wl.normal_bf16((16384, 10240), 87, 0.02)
    big[5000:5003, 7000] = 30.0
    for w in (big, wl.normal_bf16((256, 640), 88, 0.5)):
        (qx, sx, qxt, sxt), (qw, sw, qwt, swt) = fq.cast_transpose_multi(
            [(x, R.BLOCK_1x128, F.E4M3, None, None), (w, R.BLOCK_128x128, F.E4M3, None, None)])
        torch.cuda.synchronize()
        assert_status_ok()
        check_job(x, R.BLOCK_1x128, F.E4M3, None, (qx, sx, qxt, sxt), None)
        if w.shape[0] * w.shape[1] < (1 << 20):
            check_job(w, R.BLOCK_128x128, F.E4M3, None, (qw, sw, qwt, swt), None)
            continue
        rng = np.random.default_rng(89)
        tiles = [(0, 0), (127, 79), (5000 // 128, 7000 // 128)] + [tuple(t) for t in rng.integers(0, (128, 80), (5, 2))]
        for ti, tj in tiles:
            rs, cs = slice(ti * 128, ti * 128 + 128), slice(tj * 128, tj * 128 + 128)
            xt = bits16(w[rs, cs])
            q_ref, s_ref = oracle.quantize_rowwise(xt, KIND[R.BLOCK_128x128], int(F.E4M3))
            assert_bytes_equal(host(qw[rs, cs]), q_ref, f"q_row tile {ti},{tj}")
            assert f32bits(host(sw[ti, tj])) == f32bits(s_ref[0, 0])
            qc_ref, sc_ref = oracle.quantize_colwise(xt, KIND[R.BLOCK_128x128], int(F.E4M3))
            assert_bytes_equal(host(qwt[cs, rs]), qc_ref, f"q_col tile {ti},{tj}")
            assert f32bits(host(swt[tj, ti])) == f32bits(sc_ref[0, 0])
