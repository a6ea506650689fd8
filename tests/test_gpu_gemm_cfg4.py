"""GPU parity of the three GEMMs of each GPT-175B linear at full size (2048 tokens; QKV
12288 -> 36864, proj 12288 -> 12288, FC1 12288 -> 49152, FC2 49152 -> 12288), as the
benchmark sweep runs them: per-tensor scaling, X and W in E4M3, dY in E5M2, with the scales
of this step's tensors (current scaling, from the oracle's amax of the BF16 bytes);
fprop Y = X W^T (BF16), dgrad dX = dY W (BF16), wgrad dW = dY^T X (FP32).

The full products are out of the oracle's reach (up to 2.5 TFLOP in float64), so each GEMM
is checked on a seeded block of up to 256 x 256 output entries that includes the first and
last row and column: the oracle quantizes the BF16 rows and columns those entries need
(per-tensor quantization is elementwise, so those bytes are the whole tensor's), the GPU's
FP8 bytes of the same rows are compared bit for bit, and the entries are float64 dot
products of the dequantized operands, held to the GEMM bar."""
import numpy as np
import pytest
import torch

import oracle
import scaled_quantize_gemm_amax_gb300 as fq
from scaled_quantize_gemm_amax_gb300 import workloads as wl
from gpu_util import F, R, assert_bytes_equal, assert_status_ok, bits16, host, require_gpu

pytestmark = pytest.mark.gpu

NS = 256   # sampled rows and columns of each output


@pytest.fixture(scope="module", autouse=True)
def _gpu():
    require_gpu()


def sample(n, rng):
    idx = rng.choice(n, size=NS - 2, replace=False)
    return np.unique(np.concatenate([[0, n - 1], idx]))


def rows_of(t, idx):
    return host(t[torch.as_tensor(idx, device=t.device)])


def check_block(c, rows, cols, a_rows_bf16, b_rows_bf16, fa, fb, sa, sb, qa_gpu, qb_gpu, what):
    """c [M, N] on the GPU; a_rows_bf16 / b_rows_bf16 the BF16 rows of A and B for the
    sampled output rows / columns; qa_gpu / qb_gpu the GPU's FP8 bytes of the same rows."""
    qa, s_a = oracle.quantize_rowwise(a_rows_bf16, oracle.KIND_TENSOR, fa, sa)
    qb, s_b = oracle.quantize_rowwise(b_rows_bf16, oracle.KIND_TENSOR, fb, sb)
    assert_bytes_equal(qa_gpu, qa, what + ": A bytes")
    assert_bytes_equal(qb_gpu, qb, what + ": B bytes")
    da = oracle.dequantize(qa, oracle.KIND_TENSOR, fa, s_a)
    db = oracle.dequantize(qb, oracle.KIND_TENSOR, fb, s_b)
    c_ref = da @ db.T
    c_blk = host(c[torch.as_tensor(rows, device=c.device)][:, torch.as_tensor(cols, device=c.device)].float())
    rel, worst = oracle.gemm_tolerance_check(c_blk.astype(np.float64), c_ref, da, db)
    assert rel <= 1e-2, f"{what}: relative Frobenius error {rel:.3e}"
    assert worst <= 1.0, f"{what}: max-abs bound exceeded by x{worst:.3f}"


@pytest.mark.parametrize("name", list(wl.CFG4_LINEARS))
def test_gpt175b_linear_gemms_sampled(name):
    x, w, dy = wl.cfg4_step(name, 0, "cuda")
    tokens, fin = x.shape
    fout = w.shape[0]
    e4, e5 = int(F.E4M3), int(F.E5M2)
    xh, wh, dyh = bits16(x), bits16(w), bits16(dy)
    sx, _ = oracle.tensor_scale(oracle.amax(xh), e4)
    sw, _ = oracle.tensor_scale(oracle.amax(wh), e4)
    sdy, _ = oracle.tensor_scale(oracle.amax(dyh), e5)

    def cast(t, fmt, s):
        return fq.cast_transpose(t, R.TENSOR, fmt, torch.tensor([s], dtype=torch.float32, device="cuda"))

    qx, s_x, qxt, s_xt = cast(x, F.E4M3, sx)
    qw, s_w, qwt, s_wt = cast(w, F.E4M3, sw)
    qdy, s_dy, qdyt, s_dyt = cast(dy, F.E5M2, sdy)
    y = fq.scaled_gemm(qx, F.E4M3, R.TENSOR, s_x, qw, F.E4M3, R.TENSOR, s_w)
    dx = fq.scaled_gemm(qdy, F.E5M2, R.TENSOR, s_dy, qwt, F.E4M3, R.TENSOR, s_wt)
    dw = fq.scaled_gemm(qdyt, F.E5M2, R.TENSOR, s_dyt, qxt, F.E4M3, R.TENSOR, s_xt, out=fq.OutDtype.FP32)
    torch.cuda.synchronize()
    assert_status_ok()

    rng = np.random.default_rng(4000 + list(wl.CFG4_LINEARS).index(name))
    m = sample(tokens, rng)      # token rows
    n = sample(fout, rng)        # output features
    k = sample(fin, rng)         # input features
    # fprop: rows of X (tokens) against rows of W (output features)
    check_block(y, m, n, xh[m], wh[n], e4, e4, sx, sw, rows_of(qx, m), rows_of(qw, n), f"{name} fprop")
    # dgrad: rows of dY against rows of W^T, i.e. columns of W (input features)
    check_block(dx, m, k, dyh[m], np.ascontiguousarray(wh[:, k].T), e5, e4, sdy, sw, rows_of(qdy, m), rows_of(qwt, k),
                f"{name} dgrad")
    # wgrad: rows of dY^T (columns of dY) against rows of X^T (columns of X)
    check_block(dw, n, k, np.ascontiguousarray(dyh[:, n].T), np.ascontiguousarray(xh[:, k].T), e5, e4, sdy, sx,
                rows_of(qdyt, n), rows_of(qxt, k), f"{name} wgrad")
