"""GPU parity of fp8_allreduce_sum (k ranks on one device) against the oracle,
bit for bit: the global amax, every rank's FP8 payload, scale_inv and the
reduced gradient."""
import numpy as np
import pytest
import torch

import oracle
import scaled_quantize_gemm_amax_gb300 as fq
from gpu_util import F, assert_bytes_equal, assert_status_ok, bits16, f32bits, host, require_gpu

pytestmark = pytest.mark.gpu


@pytest.fixture(scope="module", autouse=True)
def _gpu():
    require_gpu()


def rank_grads(k, n, seed, sigma=1e-3):
    g = torch.Generator(device="cuda")
    g.manual_seed(seed)
    x = torch.randn((k, n), generator=g, device="cuda") * sigma
    x *= torch.logspace(-2, 1, k, device="cuda")[:, None]      # ranks of different magnitude
    return x.to(torch.bfloat16)


def check(g, fmt):
    out, q, si, amax = fq.allreduce_sum(g, fmt)
    torch.cuda.synchronize()
    assert_status_ok()
    a_ref, q_ref, si_ref, out_ref = oracle.allreduce_sum(bits16(g), int(fmt))
    assert f32bits(host(amax))[0] == f32bits(a_ref), "amax"
    assert f32bits(host(si))[0] == f32bits(si_ref), "scale_inv"
    assert_bytes_equal(host(q), q_ref, "payloads")
    assert_bytes_equal(f32bits(host(out)), f32bits(out_ref), "reduced gradient")


@pytest.mark.parametrize("fmt", [F.E4M3, F.E5M2])
@pytest.mark.parametrize("k,n", [(1, 8), (2, 1024), (5, 4000), (8, 100000), (13, 2048)])
def test_allreduce_matches_oracle(fmt, k, n):
    check(rank_grads(k, n, 100 + k), fmt)


def test_allreduce_zero_gradients_and_one_outlier():
    g = torch.zeros((4, 512), dtype=torch.bfloat16, device="cuda")
    check(g, F.E5M2)                      # amax 0: scale 1, all-zero payloads and sum
    g[2, 7] = -3.0e4                      # one large element sets the shared range
    g[0, :] = 1.0e-3
    check(g, F.E4M3)


def test_allreduce_gpt175b_gradient_size():
    # 8 ranks of one 12288 x 1024 slice of a GPT-175B weight gradient (dY-like magnitudes)
    check(rank_grads(8, 12288 * 1024, 7, 1e-3), F.E5M2)
