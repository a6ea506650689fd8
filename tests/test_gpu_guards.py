"""Out-of-bounds writes: every output of every entry point sits between two 4 KB
guard regions filled with a sentinel byte, on ragged, tail and odd-tile shapes.
After each call the guards must be untouched and the outputs equal to the oracle's
(bit for bit; the GEMM within the stated bar), so a kernel that writes one byte
before or past any output buffer fails here even where the buffer's own contents
are right.  (compute-sanitizer is not available to these tests.)"""
import numpy as np
import pytest
import torch

import oracle
import scaled_quantize_gemm_amax_gb300 as fq
from scaled_quantize_gemm_amax_gb300 import workloads as wl
from gpu_util import (R, F, KIND, MX_RECIPES, Guarded, assert_bytes_equal, assert_status_ok, bits16, f32bits, host,
                      oracle_scales_like, require_gpu)

pytestmark = pytest.mark.gpu


@pytest.fixture(scope="module", autouse=True)
def _gpu():
    require_gpu()


def _scales_check(recipe, got, ref, what):
    if recipe in MX_RECIPES:
        assert_bytes_equal(got, ref, what)
    else:
        assert_bytes_equal(f32bits(got), f32bits(ref), what)


CAST_CASES = [
    (R.TENSOR, (1000, 304), F.E4M3),        # rows % 16 != 0: the plain per-tensor kernel
    (R.TENSOR, (1008, 304), F.E5M2),        # the tiled kernel with ragged last tiles both ways
    (R.TENSOR, (136, 200), F.E4M3),         # cols % 16 != 0: plain kernel, short rows
    (R.BLOCK_1x128, (384, 640), F.E4M3),
    (R.BLOCK_1x128, (128, 896), F.E5M2),    # one tile row
    (R.BLOCK_128x128, (384, 640), F.E4M3),
    (R.MX_1x32, (160, 96), F.E4M3),         # row-major E8M0, tiles hanging over both edges
    (R.MX_1x32_TILED, (384, 640), F.E5M2),
]


@pytest.mark.parametrize("recipe,shape,fmt", CAST_CASES)
def test_cast_transpose_writes_only_its_outputs(recipe, shape, fmt):
    rows, cols = shape
    x = wl.normal_bf16(shape, 300 + rows, 1.0)
    xh = bits16(x)
    scale_np = scale_t = None
    if recipe == R.TENSOR:
        scale_np, _ = oracle.tensor_scale(oracle.amax(xh), int(fmt))
        scale_t = torch.tensor([scale_np], dtype=torch.float32, device="cuda")
    shp_r, dt_r = fq.scale_shape(recipe, rows, cols)
    shp_c, dt_c = fq.scale_shape(recipe, cols, rows)
    g = {"q_row": Guarded((rows, cols), torch.uint8), "s_row": Guarded(shp_r, dt_r),
         "q_col": Guarded((cols, rows), torch.uint8), "s_col": Guarded(shp_c, dt_c),
         "amax": Guarded((1,), torch.float32)}
    fq.fp8_cast_transpose(x, recipe, fmt, scale_t, g["amax"].t, g["q_row"].t, g["s_row"].t, g["q_col"].t,
                          g["s_col"].t)
    torch.cuda.synchronize()
    assert_status_ok()
    for name, b in g.items():
        b.check(name)
    kind = KIND[recipe]
    assert f32bits(host(g["amax"].t))[0] == f32bits(oracle.amax(xh)), "amax_out"
    q_ref, s_ref = oracle.quantize_rowwise(xh, kind, int(fmt), scale_np)
    assert_bytes_equal(host(g["q_row"].t), q_ref, "q_row")
    _scales_check(recipe, host(g["s_row"].t), oracle_scales_like(recipe, s_ref, rows, cols), "s_row")
    q_ref, s_ref = oracle.quantize_colwise(xh, kind, int(fmt), scale_np)
    assert_bytes_equal(host(g["q_col"].t), q_ref, "q_col")
    _scales_check(recipe, host(g["s_col"].t), oracle_scales_like(recipe, s_ref, cols, rows), "s_col")


PAIRS = [(R.TENSOR, R.TENSOR), (R.BLOCK_1x128, R.BLOCK_128x128), (R.BLOCK_1x128, R.BLOCK_1x128),
         (R.MX_1x32_TILED, R.MX_1x32_TILED)]


def _operands(m, n, k, ra, rb, seed):
    """Both sides quantize the same BF16 bytes; returns GPU (qa, sa, qb, sb) and the
    oracle's dequantized operands."""
    x = wl.normal_bf16((m, k), seed, 1.0)
    w = wl.normal_bf16((n, k), seed + 1, 0.02)
    out = []
    deq = []
    for t, rec in ((x, ra), (w, rb)):
        th = bits16(t)
        sc_np = sc_t = None
        if rec == R.TENSOR:
            sc_np, _ = oracle.tensor_scale(oracle.amax(th), int(F.E4M3))
            sc_t = torch.tensor([sc_np], dtype=torch.float32, device="cuda")
        q, s, _, _ = fq.cast_transpose(t, rec, F.E4M3, sc_t, col=False)
        q_ref, s_ref = oracle.quantize_rowwise(th, KIND[rec], int(F.E4M3), sc_np)
        out += [q, s]
        deq.append(oracle.dequantize(q_ref, KIND[rec], int(F.E4M3), s_ref))
    return out, deq


def _gemm_bar(c, deq_a, deq_b):
    c_ref = deq_a @ deq_b.T
    rel, worst = oracle.gemm_tolerance_check(host(c.float()).astype(np.float64), c_ref, deq_a, deq_b)
    assert rel <= 1e-2 and worst <= 1.0, (rel, worst)


@pytest.mark.parametrize("ra,rb", PAIRS)
@pytest.mark.parametrize("m,n,k", [(256, 384, 512),    # CTA pairs, N tail (a 256-wide tile half outside)
                                   (384, 640, 640),    # single CTAs, N tail, odd k-blocks
                                   (128, 128, 256)])   # one tile
@pytest.mark.parametrize("out", [fq.OutDtype.BF16, fq.OutDtype.FP32])
def test_gemm_writes_only_c(ra, rb, m, n, k, out):
    (qa, sa, qb, sb), (deq_a, deq_b) = _operands(m, n, k, ra, rb, 400 + m + n)
    c = Guarded((m, n), torch.float32 if out == fq.OutDtype.FP32 else torch.bfloat16)
    fq.fp8_scaled_gemm(qa, F.E4M3, ra, sa, qb, F.E4M3, rb, sb, c.t, out)
    torch.cuda.synchronize()
    assert_status_ok()
    c.check("C")
    _gemm_bar(c.t, deq_a, deq_b)


@pytest.mark.parametrize("ra,rb", PAIRS)
@pytest.mark.parametrize("m,n,k", [(256, 384, 512), (384, 640, 640)])
def test_fused_gemm_writes_only_its_outputs(ra, rb, m, n, k):
    (qa, sa, qb, sb), (deq_a, deq_b) = _operands(m, n, k, ra, rb, 500 + m + n)
    c = Guarded((m, n), torch.bfloat16)
    c_q = Guarded((m, n), torch.uint8)
    c_amax = Guarded((1,), torch.float32)
    c_sinv = Guarded((1,), torch.float32)
    c_scale = torch.tensor([8.0], dtype=torch.float32, device="cuda")
    fq.fp8_scaled_gemm_amax(qa, F.E4M3, ra, sa, qb, F.E4M3, rb, sb, c.t, fq.OutDtype.BF16, c_amax.t, c_scale,
                            F.E4M3, c_q.t, c_sinv.t)
    torch.cuda.synchronize()
    assert_status_ok()
    for name, b in (("C", c), ("C_q", c_q), ("c_amax", c_amax), ("c_scale_inv", c_sinv)):
        b.check(name)
    _gemm_bar(c.t, deq_a, deq_b)
    cb = bits16(c.t)
    assert f32bits(host(c_amax.t))[0] == f32bits(oracle.amax(cb)), "amax of C"
    q_ref, _ = oracle.quantize_rowwise(cb, oracle.KIND_TENSOR, int(F.E4M3), np.float32(8.0))
    assert_bytes_equal(host(c_q.t), q_ref, "C_q")
    assert f32bits(host(c_sinv.t))[0] == f32bits(np.float32(1.0) / np.float32(8.0)), "c_scale_inv"


@pytest.mark.parametrize("recipe,shape", [(R.TENSOR, (1000, 304)), (R.TENSOR, (136, 200)),
                                          (R.BLOCK_1x128, (384, 640)), (R.BLOCK_128x128, (384, 640)),
                                          (R.MX_1x32, (160, 96)), (R.MX_1x32_TILED, (384, 640))])
def test_dequantize_writes_only_y(recipe, shape):
    rows, cols = shape
    x = wl.normal_bf16(shape, 600 + rows, 1.0, "cpu")
    xh = bits16(x)
    kind = KIND[recipe]
    scale = None
    if recipe == R.TENSOR:
        scale, _ = oracle.tensor_scale(oracle.amax(xh), int(F.E4M3))
    q, s = oracle.quantize_rowwise(xh, kind, int(F.E4M3), scale)
    ref = oracle.dequantize_bf16(q, kind, int(F.E4M3), s)
    s_dev = oracle.mx_to_tiled(s) if recipe == R.MX_1x32_TILED else s
    y = Guarded(shape, torch.bfloat16)
    fq.fp8_dequantize(torch.from_numpy(q).cuda(), recipe, F.E4M3, torch.from_numpy(np.ascontiguousarray(s_dev)).cuda(),
                      y.t)
    torch.cuda.synchronize()
    assert_status_ok()
    y.check("y")
    assert_bytes_equal(host(y.t.view(torch.int16)).view(np.uint16), ref, "y")


@pytest.mark.parametrize("k,n", [(3, 1000), (1, 8), (6, 4104)])
def test_allreduce_writes_only_its_outputs(k, n):
    g = (torch.randn((k, n), generator=torch.Generator(device="cuda").manual_seed(700 + n), device="cuda")
         * 1e-3).to(torch.bfloat16)
    amax = Guarded((1,), torch.float32)
    q = Guarded((k, n), torch.uint8)
    si = Guarded((1,), torch.float32)
    out = Guarded((n,), torch.float32)
    fq.fp8_allreduce_sum(g, F.E5M2, amax.t, q.t, si.t, out.t)
    torch.cuda.synchronize()
    assert_status_ok()
    for name, b in (("amax", amax), ("q", q), ("scale_inv", si), ("out", out)):
        b.check(name)
    a_ref, q_ref, si_ref, out_ref = oracle.allreduce_sum(bits16(g), int(F.E5M2))
    assert f32bits(host(amax.t))[0] == f32bits(a_ref), "amax"
    assert f32bits(host(si.t))[0] == f32bits(si_ref), "scale_inv"
    assert_bytes_equal(host(q.t), q_ref, "payloads")
    assert_bytes_equal(f32bits(host(out.t)), f32bits(out_ref), "reduced gradient")
