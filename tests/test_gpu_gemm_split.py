"""The partial last wave of the per-tensor and MX GEMMs on CTA pairs, cut along K on
otherwise idle pairs: with two or three full waves (or one, when K >= 8192), all but the
last full wave run as whole tiles and every pair then takes an equal share of the
remaining tiles' K blocks (stream-K: a tile cut between two pairs is finished by the
first, which adds the second's FP32 values); with one partial wave only, or with
K >= 8192 and more waves, the last wave's tiles are cut into K ranges that range 0 adds
in order.  Parity with the oracle on
shapes of each kind, bit-identical results from repeated launches (the per-slot counters
are back at zero after every launch) and from two streams running at once (each stream
has its own workspace).  The wave counts assume the 76 resident pairs of a 152-SM part;
elsewhere the shapes still check parity."""
import numpy as np
import pytest
import torch

import scaled_quantize_gemm_amax_gb300 as fq
from scaled_quantize_gemm_amax_gb300 import workloads as wl
from gpu_util import R, F, assert_status_ok, host, require_gpu
from test_gpu_gemm import _quant_gpu, _quant_oracle, gemm_check

pytestmark = pytest.mark.gpu


@pytest.fixture(scope="module", autouse=True)
def _gpu():
    require_gpu()


SPLIT_PAIRS = [(R.TENSOR, R.TENSOR), (R.MX_1x32_TILED, R.MX_1x32_TILED)]


@pytest.mark.parametrize("ra,rb", SPLIT_PAIRS)
@pytest.mark.parametrize("m,n,k,out", [
    (256, 256, 4096, fq.OutDtype.BF16),     # one tile, 32 k-blocks: 8 ranges of 4
    (512, 384, 640, fq.OutDtype.FP32),      # 4 tiles (N ragged: half of the second column of tiles), 5 ranges
    (2560, 2304, 8192, fq.OutDtype.BF16),   # 90 tiles, one full wave: stream-K shares of 7.6 tiles' K blocks
    (2560, 2304, 4096, fq.OutDtype.BF16),   # the same with K = 4096: whole tiles
    (4096, 4096, 512, fq.OutDtype.FP32),    # 256 tiles, three full waves: two whole, then shares of 1.4 tiles
    (8192, 6144, 8192, fq.OutDtype.BF16),   # 768 tiles, ten full waves and 8 tail tiles in 8 ranges
    (4608, 4608, 512, fq.OutDtype.FP32),    # 324 tiles, four full waves, K < 8192: not cut
])
def test_split_tail_parity(ra, rb, m, n, k, out):
    # independent seeds for A and B (equal seeds would make B a multiple of A's rows, and
    # C's diagonal a sum of squares, which the max-abs bar does not describe)
    x = wl.normal_bf16((m, k), 700 + m % 97, 1.0)
    w = wl.normal_bf16((n, k), 900 + n % 89, 0.02)
    rows = None if m * n <= 2560 * 2304 else np.arange(0, m, 5)
    gemm_check(x, w, ra, rb, F.E4M3, F.E4M3, out=out, rows=rows)


def _operands(ra, rb, m, n, k, seed):
    x = wl.normal_bf16((m, k), seed, 1.0)
    w = wl.normal_bf16((n, k), seed + 1, 0.02)
    _, _, sca = _quant_oracle(x.view(torch.int16).cpu().numpy().view(np.uint16), ra, F.E4M3)
    _, _, scb = _quant_oracle(w.view(torch.int16).cpu().numpy().view(np.uint16), rb, F.E4M3)
    qa, sa = _quant_gpu(x, ra, F.E4M3, sca)
    qb, sb = _quant_gpu(w, rb, F.E4M3, scb)
    return qa, sa, qb, sb


@pytest.mark.parametrize("ra,rb", SPLIT_PAIRS)
def test_split_repeated_launches_identical(ra, rb):
    m, n, k = 2560, 2304, 8192
    qa, sa, qb, sb = _operands(ra, rb, m, n, k, 80)
    cs = [torch.empty((m, n), dtype=torch.bfloat16, device="cuda") for _ in range(4)]
    for c in cs:   # back to back on one stream: each launch finds the counters reset by the previous one
        fq.fp8_scaled_gemm(qa, F.E4M3, ra, sa, qb, F.E4M3, rb, sb, c)
    torch.cuda.synchronize()
    assert_status_ok()
    ref = host(cs[0].view(torch.int16))
    for i, c in enumerate(cs[1:], 1):
        assert np.array_equal(host(c.view(torch.int16)), ref), f"launch {i} differs from launch 0"


def test_split_two_streams_at_once():
    m, n, k = 2560, 2304, 8192
    ops = [_operands(R.TENSOR, R.TENSOR, m, n, k, 90), _operands(R.MX_1x32_TILED, R.MX_1x32_TILED, m, n, k, 92)]
    recs = [(R.TENSOR, R.TENSOR), (R.MX_1x32_TILED, R.MX_1x32_TILED)]
    refs = []
    for (qa, sa, qb, sb), (ra, rb) in zip(ops, recs):
        c = torch.empty((m, n), dtype=torch.bfloat16, device="cuda")
        fq.fp8_scaled_gemm(qa, F.E4M3, ra, sa, qb, F.E4M3, rb, sb, c)
        refs.append(c)
    torch.cuda.synchronize()
    streams = [torch.cuda.Stream(), torch.cuda.Stream()]
    outs = [[torch.empty((m, n), dtype=torch.bfloat16, device="cuda") for _ in range(3)] for _ in range(2)]
    for it in range(3):
        for s, (qa, sa, qb, sb), (ra, rb), o in zip(streams, ops, recs, outs):
            fq.fp8_scaled_gemm(qa, F.E4M3, ra, sa, qb, F.E4M3, rb, sb, o[it], stream=s)
    torch.cuda.synchronize()
    assert_status_ok()
    for ref, o in zip(refs, outs):
        for c in o:
            assert np.array_equal(host(c.view(torch.int16)), host(ref.view(torch.int16)))


def test_split_inside_cuda_graphs():
    # Stream-K shape (256 tiles, three full waves).  A stream that has no workspace yet when
    # a GEMM is captured gets whole tiles in its graph (no allocation inside a capture; the
    # stream may come from a pool that already gave it one, then it is used); once the
    # stream has one (after an eager call), a captured GEMM uses it.  Replays are
    # deterministic, the second graph gives the eager result bit for bit, and both stay
    # within the bar.
    m, n, k = 4096, 4096, 512
    x = wl.normal_bf16((m, k), 730, 1.0)
    w = wl.normal_bf16((n, k), 731, 0.02)
    qa, sa, qb, sb = _operands(R.TENSOR, R.TENSOR, m, n, k, 730)
    s = torch.cuda.Stream()
    c_whole = torch.empty((m, n), dtype=torch.float32, device="cuda")
    c_sk = torch.empty((m, n), dtype=torch.float32, device="cuda")
    run = lambda c: fq.fp8_scaled_gemm(qa, F.E4M3, R.TENSOR, sa, qb, F.E4M3, R.TENSOR, sb, c, fq.OutDtype.FP32,
                                       stream=s)
    g_whole = torch.cuda.CUDAGraph()
    with torch.cuda.graph(g_whole, stream=s):
        run(c_whole)                       # the stream has no workspace: whole tiles
    eager = torch.empty_like(c_sk)
    with torch.cuda.stream(s):
        run(eager)                         # allocates the stream's workspace: stream-K
    torch.cuda.synchronize()
    g_sk = torch.cuda.CUDAGraph()
    with torch.cuda.graph(g_sk, stream=s):
        run(c_sk)
    outs_whole, outs_sk = [], []
    for _ in range(3):
        g_whole.replay()
        g_sk.replay()
        torch.cuda.synchronize()
        outs_whole.append(host(c_whole).copy())
        outs_sk.append(host(c_sk).copy())
    assert_status_ok()
    for o in outs_sk:
        assert np.array_equal(o.view(np.uint32), host(eager).view(np.uint32))
    for o in outs_whole[1:]:
        assert np.array_equal(o.view(np.uint32), outs_whole[0].view(np.uint32))
    # both divisions against the oracle on sampled rows
    from test_gpu_gemm import _quant_oracle
    import oracle
    from gpu_util import bits16
    qa_ref, sa_ref, sca = _quant_oracle(bits16(x), R.TENSOR, F.E4M3)
    qb_ref, sb_ref, scb = _quant_oracle(bits16(w), R.TENSOR, F.E4M3)
    rows = np.arange(0, m, 9)
    deq_a = oracle.dequantize(qa_ref[rows], oracle.KIND_TENSOR, int(F.E4M3), sa_ref)
    deq_b = oracle.dequantize(qb_ref, oracle.KIND_TENSOR, int(F.E4M3), sb_ref)
    c_ref = deq_a @ deq_b.T
    for c in (outs_whole[0], outs_sk[0]):
        rel, worst = oracle.gemm_tolerance_check(c[rows].astype(np.float64), c_ref, deq_a, deq_b)
        assert rel <= 1e-2 and worst <= 1.0, (rel, worst)
