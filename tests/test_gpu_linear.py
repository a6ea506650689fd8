"""GPU parity of the FP8 linear layer (fprop, dgrad, wgrad through the C ABI)
against the oracle: the oracle quantizes the same BF16 operands with the recipe's
rules and computes each GEMM in float64; every output is held to the GEMM bar."""
import numpy as np
import pytest
import torch

import oracle
from scaled_quantize_gemm_amax_gb300 import Format
from scaled_quantize_gemm_amax_gb300 import linear as L
from scaled_quantize_gemm_amax_gb300 import workloads as wl
from gpu_util import assert_status_ok, bits16, host, require_gpu, tile_spread
import scaled_quantize_gemm_amax_gb300 as fq

pytestmark = pytest.mark.gpu

M, K, N = 256, 384, 512


@pytest.fixture(scope="module", autouse=True)
def _gpu():
    require_gpu()


def oracle_copies(xh, kind, fmt, scale=None):
    """Row- and column-wise oracle copies of bf16 bits (uint16) or float32 values."""
    if xh.dtype == np.float32:
        q_r, s_r = oracle.quantize_rowwise_f32(xh, kind, fmt, scale)
        q_c, s_c = oracle.quantize_colwise_f32(xh, kind, fmt, scale)
    else:
        q_r, s_r = oracle.quantize_rowwise(xh, kind, fmt, scale)
        q_c, s_c = oracle.quantize_colwise(xh, kind, fmt, scale)
    return (q_r, s_r), (q_c, s_c)


def host_bits(t):
    """The oracle's input form of a tensor: bf16 bit patterns, or float32 values."""
    return host(t).astype(np.float32) if t.dtype == torch.float32 else bits16(t)


def amax_of(h):
    return oracle.amax_f32(h) if h.dtype == np.float32 else oracle.amax(h)


def deq(qs, kind, fmt):
    return oracle.dequantize(qs[0], kind, fmt, qs[1])


def check(c_gpu, a_deq, b_deq, what):
    c_ref = a_deq @ b_deq.T
    rel, worst = oracle.gemm_tolerance_check(host(c_gpu.float()).astype(np.float64), c_ref, a_deq, b_deq)
    assert rel <= 1e-2 and worst <= 1.0, f"{what}: rel {rel:.3e} worst {worst:.3f}"


def run_layer(recipe, seed, steps=1, dtype=torch.bfloat16):
    torch.manual_seed(seed + 5000)   # weights independent of the seeded inputs' streams
    layer = L.FP8Linear(K, N, device="cuda")
    outs = []
    for step in range(steps):
        x = wl.normal_bf16((M, K), seed + 10 * step, 1.0)
        dy = wl.normal_bf16((M, N), seed + 10 * step + 1, 1e-3)
        if dtype == torch.float32:
            # general binary32 values (not bfloat16 ones)
            x = x.float() * (1.0 + torch.rand_like(x, dtype=torch.float32) * 2.0 ** -10)
            dy = dy.float() * (1.0 + torch.rand_like(dy, dtype=torch.float32) * 2.0 ** -10)
        x.requires_grad_(True)
        layer.weight.grad = None
        with L.fp8_autocast(fp8_recipe=recipe):
            y = layer(x)
        y.backward(dy)
        torch.cuda.synchronize()
        assert_status_ok()
        assert y.dtype == dtype and x.grad.dtype == dtype and layer.weight.grad.dtype == torch.float32
        outs.append((x.detach(), dy, layer.weight.detach().clone(), y.detach(), x.grad.clone(),
                     layer.weight.grad.clone()))
    return outs


KINDS = {"current": (oracle.KIND_TENSOR, oracle.KIND_TENSOR), "block": (oracle.KIND_1x128, oracle.KIND_128x128),
         "mx": (oracle.KIND_MX, oracle.KIND_MX)}


@pytest.mark.parametrize("name,recipe", [("current", L.Float8CurrentScaling()), ("block", L.Float8BlockScaling()),
                                         ("mx", L.MXFP8BlockScaling())])
@pytest.mark.parametrize("dtype", [torch.bfloat16, torch.float32])
def test_fp8_linear_three_gemms(name, recipe, dtype):
    # the FP32 master weight is quantized as it is; bf16 or float32 activations and
    # gradients go to the cast of their own dtype
    (x, dy, w32, y, dx, dw), = run_layer(recipe, 80, dtype=dtype)
    kx, kw = KINDS[name]
    fx, fdy = int(recipe.fwd_format), int(recipe.bwd_format)
    xh, wh, dyh = host_bits(x), host_bits(w32), host_bits(dy)
    sx = sw = sdy = None
    if name == "current":
        sx, _ = oracle.tensor_scale(amax_of(xh), fx)
        sw, _ = oracle.tensor_scale(amax_of(wh), fx)
        sdy, _ = oracle.tensor_scale(amax_of(dyh), fdy)
    x_r, x_c = oracle_copies(xh, kx, fx, sx)
    w_r, w_c = oracle_copies(wh, kw, fx, sw)
    dy_r, dy_c = oracle_copies(dyh, kx, fdy, sdy)
    check(y, deq(x_r, kx, fx), deq(w_r, kw, fx), "fprop")
    check(dx, deq(dy_r, kx, fdy), deq(w_c, kw, fx), "dgrad")
    check(dw, deq(dy_c, kx, fdy), deq(x_c, kx, fx), "wgrad")


def test_fp8_linear_delayed_scaling_steps():
    # delayed scaling: step t quantizes with the scale the history held before t (1 at t = 0)
    recipe = L.Float8DelayedScaling(history_len=16)
    outs = run_layer(recipe, 90, steps=3)
    st = {"x": oracle.DelayedState(16, oracle.E4M3), "w": oracle.DelayedState(16, oracle.E4M3),
          "dy": oracle.DelayedState(16, oracle.E5M2)}
    for step, (x, dy, w32, y, dx, dw) in enumerate(outs):
        xh, wh, dyh = bits16(x), host_bits(w32), bits16(dy)
        x_r, x_c = oracle_copies(xh, 0, oracle.E4M3, st["x"].scale[0])
        w_r, w_c = oracle_copies(wh, 0, oracle.E4M3, st["w"].scale[0])
        dy_r, dy_c = oracle_copies(dyh, 0, oracle.E5M2, st["dy"].scale[0])
        check(y, deq(x_r, 0, oracle.E4M3), deq(w_r, 0, oracle.E4M3), f"fprop step {step}")
        check(dx, deq(dy_r, 0, oracle.E5M2), deq(w_c, 0, oracle.E4M3), f"dgrad step {step}")
        check(dw, deq(dy_c, 0, oracle.E5M2), deq(x_c, 0, oracle.E4M3), f"wgrad step {step}")
        st["x"].step(oracle.amax(xh))
        st["w"].step(oracle.amax_f32(wh))
        st["dy"].step(oracle.amax(dyh))


@pytest.mark.parametrize("name,recipe", [("current", L.Float8CurrentScaling()), ("block", L.Float8BlockScaling()),
                                         ("mx", L.MXFP8BlockScaling())])
def test_dgrad_reads_the_weight_column_copy(name, recipe):
    # The dgrad GEMM of the layer's backward, dX = dY . W, reads W's column-wise copy
    # (W^T [K, N], K-major along N) made by the layer's own quantization.  W's tiles (or,
    # for MX, its 1x32 blocks along N in the column copy) and dY's blocks each carry their
    # own power of two, so a column-copy scale read for the wrong tile is off by 2x or
    # more.  FP32 output (the same GEMM the layer runs with BF16 output), because with
    # this range the exact product rounded to BF16 uses most of the max-abs bar itself.
    m, k_in, n_out = 512, 1024, 768
    kx, kw = L._kinds(recipe)
    fx, fdy = recipe.fwd_format, recipe.bwd_format
    if name == "mx":
        w16 = tile_spread(wl.normal_bf16((n_out, k_in), 95, 0.02), 32, 1, 3, 6)   # 32 x 1: blocks of W^T's rows
        dy = tile_spread(wl.normal_bf16((m, n_out), 96, 1e-3), 1, 32, 1, 6)
    else:
        w16 = tile_spread(wl.normal_bf16((n_out, k_in), 95, 0.02), 128, 128, 3, 3)
        dy = tile_spread(wl.normal_bf16((m, n_out), 96, 1e-3), 1, 128, 1, 3)
    # the layer quantizes its FP32 master weight: general binary32 values
    w32 = w16.float() * (1.0 + torch.rand_like(w16, dtype=torch.float32) * 2.0 ** -10)
    _, _, qwt, swt = L._quantize(w32, kw, fx, None)
    qdy, sdy, _, _ = L._quantize(dy, kx, fdy, None)
    dx = torch.empty((m, k_in), dtype=torch.float32, device="cuda")
    fq.fp8_scaled_gemm(qdy, fdy, kx, sdy, qwt, fx, kw, swt, dx, fq.OutDtype.FP32)
    torch.cuda.synchronize()
    assert_status_ok()
    okx, okw = KINDS[name]
    wh, dyh = host_bits(w32), bits16(dy)
    sw = sdy_s = None
    if name == "current":
        sw, _ = oracle.tensor_scale(oracle.amax_f32(wh), int(fx))
        sdy_s, _ = oracle.tensor_scale(oracle.amax(dyh), int(fdy))
    _, w_c = oracle_copies(wh, okw, int(fx), sw)
    dy_r, _ = oracle_copies(dyh, okx, int(fdy), sdy_s)
    # the column copy's bytes are the oracle's, bit for bit
    got_q = host(qwt)
    assert np.array_equal(got_q, w_c[0]), "W column copy bytes"
    check(dx, deq(dy_r, okx, int(fdy)), deq(w_c, okw, int(fx)), f"dgrad ({name})")
