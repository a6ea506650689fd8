"""GPU parity of the floor-rule MXFP8 recipes (FP8_MX_1x32_FLOOR / _FLOOR_TILED, the
documented alternate of the guide's "MXFP8 scaling" exponent) against the oracle's
floor-rule quantizers: FP8 bytes and E8M0 bytes bit for bit, for bf16 and binary32 inputs,
both copies; the GEMM of floor-rule operands within the stated bar; dequantization bit for
bit.  Inputs include blocks whose scaled maximum lands above FMAX, where the floor rule
saturates."""
import numpy as np
import pytest
import torch

import oracle
import scaled_quantize_gemm_amax_gb300 as fq
from scaled_quantize_gemm_amax_gb300 import workloads as wl
from gpu_util import R, F, KIND, assert_bytes_equal, assert_status_ok, bits16, check_cast, host, require_gpu

pytestmark = pytest.mark.gpu

FLOOR = [R.MX_1x32_FLOOR, R.MX_1x32_FLOOR_TILED]


@pytest.fixture(scope="module", autouse=True)
def _gpu():
    require_gpu()


def saturating_input(shape, seed, device="cuda"):
    """N(0,1) with every 1x32 block's maximum given a significand of 1.9, so that under the
    floor rule it scales past FMAX (E4M3: 1.9 * 256 = 486 > 448) and saturates."""
    x = wl.normal_bf16(shape, seed, 1.0, device).float()
    blk = x.view(shape[0], shape[1] // 32, 32)
    amax = blk.abs().amax(dim=2, keepdim=True)
    e = torch.floor(torch.log2(amax))
    blk.mul_(torch.where(amax > 0, 1.9 * torch.exp2(e) / amax, torch.ones_like(amax)))
    return x.to(torch.bfloat16)


@pytest.mark.parametrize("recipe", FLOOR)
@pytest.mark.parametrize("fmt", [F.E4M3, F.E5M2])
def test_cast_floor_rule_bf16(recipe, fmt):
    check_cast(saturating_input((384, 640), 801), recipe, fmt)
    check_cast(wl.normal_bf16((256, 384), 802, 1.0), recipe, fmt, row=True, col=False)


def test_cast_floor_rule_ragged_row_major():
    check_cast(saturating_input((160, 96), 803), R.MX_1x32_FLOOR, F.E4M3)


@pytest.mark.parametrize("recipe", FLOOR)
def test_cast_floor_rule_f32(recipe):
    x = saturating_input((256, 512), 804).float() * (1.0 + torch.rand((256, 512), device="cuda") * 2.0 ** -10)
    xh = host(x).astype(np.float32)
    q, s, qc, sc = fq.cast_transpose(x, recipe, F.E4M3)
    torch.cuda.synchronize()
    assert_status_ok()
    for got_q, got_s, (q_ref, s_ref), rows, cols, what in (
            (q, s, oracle.quantize_rowwise_f32(xh, oracle.KIND_MX_FLOOR, 0), 256, 512, "row"),
            (qc, sc, oracle.quantize_colwise_f32(xh, oracle.KIND_MX_FLOOR, 0), 512, 256, "col")):
        assert_bytes_equal(host(got_q), q_ref, f"q {what}")
        s_exp = oracle.mx_to_tiled(s_ref) if recipe == R.MX_1x32_FLOOR_TILED else s_ref
        assert_bytes_equal(host(got_s).reshape(-1), np.asarray(s_exp).reshape(-1), f"s {what}")


def test_gemm_and_dequantize_floor_rule_operands():
    m, n, k = 512, 384, 1024
    x = saturating_input((m, k), 805)
    w = wl.normal_bf16((n, k), 806, 0.02)
    xh, wh = bits16(x), bits16(w)
    qa_ref, sa_ref = oracle.quantize_rowwise(xh, oracle.KIND_MX_FLOOR, 0)
    qb_ref, sb_ref = oracle.quantize_rowwise(wh, oracle.KIND_MX_FLOOR, 0)
    qa, sa, _, _ = fq.cast_transpose(x, R.MX_1x32_FLOOR_TILED, F.E4M3, col=False)
    qb, sb, _, _ = fq.cast_transpose(w, R.MX_1x32_FLOOR_TILED, F.E4M3, col=False)
    c = fq.scaled_gemm(qa, F.E4M3, R.MX_1x32_FLOOR_TILED, sa, qb, F.E4M3, R.MX_1x32_FLOOR_TILED, sb,
                       out=fq.OutDtype.FP32)
    y = fq.dequantize(qa, R.MX_1x32_FLOOR_TILED, F.E4M3, sa)
    torch.cuda.synchronize()
    assert_status_ok()
    assert_bytes_equal(host(qa), qa_ref, "A bytes")
    deq_a = oracle.dequantize(qa_ref, oracle.KIND_MX_FLOOR, 0, sa_ref)
    deq_b = oracle.dequantize(qb_ref, oracle.KIND_MX_FLOOR, 0, sb_ref)
    rel, worst = oracle.gemm_tolerance_check(host(c).astype(np.float64), deq_a @ deq_b.T, deq_a, deq_b)
    assert rel <= 1e-2 and worst <= 1.0, (rel, worst)
    y_ref = oracle.dequantize_bf16(qa_ref, oracle.KIND_MX_FLOOR, 0, sa_ref)
    assert_bytes_equal(host(y.view(torch.int16)).view(np.uint16), y_ref, "dequantized A")
