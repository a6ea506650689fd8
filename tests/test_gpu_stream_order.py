"""Stream order of the reductions that start early: fp8_amax / fp8_amax_f32, and casts with
amax_out, read their input before griddepcontrol.wait (the zeroing kernel the host
launches right before them has already waited for every earlier kernel).  Each case
enqueues a producer of the input on the same stream and the reduction right after it,
with no host synchronisation in between, and compares with the oracle on the final input:
a reduction that read the input before the producer finished would see the old values
(here scaled by a different factor, so the amax differs)."""
import numpy as np
import pytest
import torch

import oracle
import scaled_quantize_gemm_amax_gb300 as fq
from gpu_util import R, F, KIND, assert_bytes_equal, assert_status_ok, bits16, f32bits, host, require_gpu

pytestmark = pytest.mark.gpu


@pytest.fixture(scope="module", autouse=True)
def _gpu():
    require_gpu()


def _base(shape, seed, dtype=torch.bfloat16):
    g = torch.Generator(device="cuda")
    g.manual_seed(seed)
    return torch.randn(shape, generator=g, device="cuda").to(dtype)


@pytest.mark.parametrize("shape", [(8192, 8192), (1000, 1003)])
def test_amax_after_torch_producer(shape):
    amax = torch.empty(1, dtype=torch.float32, device="cuda")
    x = _base(shape, 1)
    for it in range(4):
        x.mul_(-3.0)            # the producer: every element changes (|x| grows by 3)
        fq.fp8_amax(x, amax)
        torch.cuda.synchronize()
        assert_status_ok()
        assert f32bits(host(amax))[0] == f32bits(oracle.amax(bits16(x))), f"iteration {it}"
        x.mul_(1.0 / 3.0)


def test_amax_f32_after_torch_producer():
    amax = torch.empty(1, dtype=torch.float32, device="cuda")
    x = _base((4096, 8192), 2, torch.float32)
    for it in range(4):
        x.mul_(-3.0)
        fq.fp8_amax_f32(x, amax)
        torch.cuda.synchronize()
        assert_status_ok()
        assert f32bits(host(amax))[0] == f32bits(oracle.amax_f32(host(x).astype(np.float32))), f"iteration {it}"
        x.mul_(1.0 / 3.0)


def test_amax_after_library_producer():
    # the producer is the library's own (programmatically launched) dequantize kernel
    x = _base((4096, 4096), 3)
    q, s, _, _ = fq.cast_transpose(x, R.BLOCK_1x128, F.E4M3, col=False)
    y = torch.empty_like(x)
    amax = torch.empty(1, dtype=torch.float32, device="cuda")
    for it in range(4):
        s.mul_(2.0)              # a different multiplier each time: a different y
        fq.fp8_dequantize(q, R.BLOCK_1x128, F.E4M3, s, y)
        fq.fp8_amax(y, amax)
        torch.cuda.synchronize()
        assert_status_ok()
        assert f32bits(host(amax))[0] == f32bits(oracle.amax(bits16(y))), f"iteration {it}"


@pytest.mark.parametrize("recipe", [R.TENSOR, R.BLOCK_1x128, R.MX_1x32_TILED])
def test_cast_with_amax_out_after_torch_producer(recipe):
    x = _base((4096, 4096), 4)
    amax = torch.empty(1, dtype=torch.float32, device="cuda")
    one = torch.ones(1, dtype=torch.float32, device="cuda")
    sc = one if recipe == R.TENSOR else None
    for it in range(3):
        x.mul_(-3.0)
        qr, sr, qc, scol = fq.cast_transpose(x, recipe, F.E4M3, sc, amax)
        torch.cuda.synchronize()
        assert_status_ok()
        xh = bits16(x)
        assert f32bits(host(amax))[0] == f32bits(oracle.amax(xh)), f"amax, iteration {it}"
        q_ref, _ = oracle.quantize_rowwise(xh, KIND[recipe], int(F.E4M3), 1.0 if recipe == R.TENSOR else None)
        assert_bytes_equal(host(qr), q_ref, f"q_row, iteration {it}")
        x.mul_(1.0 / 3.0)


def test_multi_cast_with_amax_out_after_torch_producers():
    x = _base((2048, 4096), 5)
    w = _base((4096, 4096), 6)
    ax = torch.empty(1, dtype=torch.float32, device="cuda")
    aw = torch.empty(1, dtype=torch.float32, device="cuda")
    for it in range(3):
        x.mul_(-3.0)
        w.mul_(5.0)
        (qx, _, _, _), (qw, _, _, _) = fq.cast_transpose_multi([(x, R.BLOCK_1x128, F.E4M3, None, ax),
                                                                  (w, R.BLOCK_128x128, F.E4M3, None, aw)])
        torch.cuda.synchronize()
        assert_status_ok()
        assert f32bits(host(ax))[0] == f32bits(oracle.amax(bits16(x))), f"x amax, iteration {it}"
        assert f32bits(host(aw))[0] == f32bits(oracle.amax(bits16(w))), f"w amax, iteration {it}"
        q_ref, _ = oracle.quantize_rowwise(bits16(w), KIND[R.BLOCK_128x128], int(F.E4M3), None)
        assert_bytes_equal(host(qw), q_ref, f"w q_row, iteration {it}")
        x.mul_(1.0 / 3.0)
        w.mul_(1.0 / 5.0)


def test_cast_f32_with_amax_out_after_torch_producer():
    x = _base((2048, 4096), 7, torch.float32)
    amax = torch.empty(1, dtype=torch.float32, device="cuda")
    for it in range(3):
        x.mul_(-3.0)
        qr, _, _, _ = fq.cast_transpose(x, R.BLOCK_128x128, F.E4M3, None, amax)
        torch.cuda.synchronize()
        assert_status_ok()
        xh = host(x).astype(np.float32)
        assert f32bits(host(amax))[0] == f32bits(oracle.amax_f32(xh)), f"amax, iteration {it}"
        q_ref, _ = oracle.quantize_rowwise_f32(xh, KIND[R.BLOCK_128x128], int(F.E4M3), None)
        assert_bytes_equal(host(qr), q_ref, f"q_row, iteration {it}")
        x.mul_(1.0 / 3.0)
