"""GPU parity of the GEMM with the fused output quantization (fp8_scaled_gemm_amax).

C itself is held to the GEMM bar against the oracle (test_gpu_gemm.gemm_check's
criteria).  The fused outputs are exact functions of the stored C, so they are
compared bit for bit with the oracle applied to the GPU's own C: the amax with
oracle.amax / oracle.amax_f32, the FP8 copy with the oracle's per-tensor quantizer
(bf16 C) or its encoder on binary32 products (fp32 C)."""
import numpy as np
import pytest
import torch

import oracle
import scaled_quantize_gemm_amax_gb300 as fq
from scaled_quantize_gemm_amax_gb300 import workloads as wl
from gpu_util import R, F, assert_bytes_equal, assert_status_ok, bits16, f32bits, host, require_gpu
from test_gpu_gemm import PAIRS, _quant_gpu, _quant_oracle

pytestmark = pytest.mark.gpu


@pytest.fixture(scope="module", autouse=True)
def _gpu():
    require_gpu()


def run_fused(x, w, ra, rb, fa, fb, c_scale, fc, out, keep_c=True):
    xh, wh = bits16(x), bits16(w)
    _, _, sca = _quant_oracle(xh, ra, fa)
    _, _, scb = _quant_oracle(wh, rb, fb)
    qa, sa = _quant_gpu(x, ra, fa, sca)
    qb, sb = _quant_gpu(w, rb, fb, scb)
    s_t = torch.tensor([c_scale], dtype=torch.float32, device="cuda")
    c, c_amax, c_q, c_sinv = fq.scaled_gemm_amax(qa, fa, ra, sa, qb, fb, rb, sb, s_t, fc, out, keep_c)
    c_plain = fq.scaled_gemm(qa, fa, ra, sa, qb, fb, rb, sb, out=out)
    torch.cuda.synchronize()
    assert_status_ok()
    return c, c_amax, c_q, c_sinv, c_plain


def check_fused(c_ref, c_amax, c_q, c_sinv, c_scale, fc, out):
    """The fused outputs against the oracle applied to the GPU's C (c_ref)."""
    if out == fq.OutDtype.BF16:
        cb = bits16(c_ref)
        assert f32bits(host(c_amax))[0] == f32bits(oracle.amax(cb))[0], "amax of C"
        q_ref, _ = oracle.quantize_rowwise(cb, oracle.KIND_TENSOR, int(fc), np.float32(c_scale))
    else:
        cf = host(c_ref).astype(np.float32)
        assert f32bits(host(c_amax))[0] == f32bits(oracle.amax_f32(cf))[0], "amax of C"
        q_ref = oracle.encode(cf * np.float32(c_scale), int(fc), True)
    assert_bytes_equal(host(c_q), q_ref, "C_q")
    si_ref = np.float32(1.0) / np.float32(c_scale)        # binary32 division, round to nearest
    assert f32bits(host(c_sinv))[0] == f32bits(si_ref)[0], "c_scale_inv"


@pytest.mark.parametrize("ra,rb", PAIRS)
@pytest.mark.parametrize("out", [fq.OutDtype.BF16, fq.OutDtype.FP32])
@pytest.mark.parametrize("n", [384, 512])
@pytest.mark.parametrize("k", [640, 512])
def test_fused_output_quantization_matches_oracle(ra, rb, out, n, k):
    # 512 x n output; N = 384 hangs over the 256-wide tiles, N = 512 fills them.  K = 640
    # (5 K blocks): the blockwise pairings run on single CTAs; K = 512 (4 K blocks): on CTA
    # pairs with 256-deep stages
    x = wl.normal_bf16((512, k), 60, 1.0)
    w = wl.normal_bf16((n, k), 61, 0.02)
    c_scale = 448.0 / 1.5          # outputs above 1.5 in magnitude saturate, most do not
    fc = F.E4M3
    c, c_amax, c_q, c_sinv, c_plain = run_fused(x, w, ra, rb, F.E4M3, F.E4M3, c_scale, fc, out)
    # the stored C is the plain GEMM's, bit for bit, and within the GEMM bar of the oracle
    assert torch.equal(c.view(torch.int16) if out == fq.OutDtype.BF16 else c.view(torch.int32),
                       c_plain.view(torch.int16) if out == fq.OutDtype.BF16 else c_plain.view(torch.int32))
    from test_gpu_gemm import gemm_check
    gemm_check(x, w, ra, rb, F.E4M3, F.E4M3, out=out)
    check_fused(c, c_amax, c_q, c_sinv, c_scale, fc, out)
    assert (host(c_q) == 0x7E).any() or (host(c_q) == 0xFE).any(), "no saturated output exercised"


@pytest.mark.parametrize("fc", [F.E4M3, F.E5M2])
def test_fused_without_c_and_e5m2(fc):
    # C not stored: the FP8 copy and amax equal those of a run that stores C
    x = wl.normal_bf16((256, 512), 62, 1.0)
    w = wl.normal_bf16((256, 512), 63, 0.02)
    c_scale = 2.0 ** 10
    _, amax1, q1, sinv1, c_plain = run_fused(x, w, R.TENSOR, R.TENSOR, F.E4M3, F.E4M3, c_scale, fc,
                                             fq.OutDtype.BF16, keep_c=False)
    check_fused(c_plain, amax1, q1, sinv1, c_scale, fc, fq.OutDtype.BF16)


def test_fused_delayed_scaling_chain():
    # Three steps of a layer output under delayed scaling: each GEMM quantizes its output
    # with the state's scale and records the amax; the history update then moves the scale.
    # Compared against the oracle's delayed-scaling state driven by the same amaxes.
    x = wl.normal_bf16((256, 256), 64, 1.0)
    w = wl.normal_bf16((256, 256), 65, 0.02)
    st = fq.DelayedScaling(16, F.E4M3)
    ref = oracle.DelayedState(16, oracle.E4M3)
    wh = bits16(w)
    for step in range(3):
        xs = x * (10.0 if step == 1 else 1.0)
        _, _, sca = _quant_oracle(bits16(xs), R.TENSOR, F.E4M3)
        _, _, scb = _quant_oracle(wh, R.TENSOR, F.E4M3)
        qa, sa = _quant_gpu(xs, R.TENSOR, F.E4M3, sca)
        qb, sb = _quant_gpu(w, R.TENSOR, F.E4M3, scb)
        c = torch.empty((256, 256), dtype=torch.bfloat16, device="cuda")
        c_q = torch.empty((256, 256), dtype=torch.uint8, device="cuda")
        s_used = float(host(st.scale)[0])
        fq.fp8_scaled_gemm_amax(qa, F.E4M3, R.TENSOR, sa, qb, F.E4M3, R.TENSOR, sb, c, fq.OutDtype.BF16, st.amax,
                                st.scale, F.E4M3, c_q, None)
        st.update()
        torch.cuda.synchronize()
        assert_status_ok()
        cb = bits16(c)
        q_ref, _ = oracle.quantize_rowwise(cb, oracle.KIND_TENSOR, oracle.E4M3, np.float32(s_used))
        assert_bytes_equal(host(c_q), q_ref, f"C_q step {step}")
        assert np.float32(s_used) == ref.scale
        ref.step(oracle.amax(cb))
        assert f32bits(host(st.scale))[0] == f32bits(ref.scale)[0], f"scale after step {step}"
