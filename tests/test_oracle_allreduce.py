"""Pins of the oracle's FP8 gradient all-reduce with a shared scale (fp8_oracle.c:
orc_allreduce_sum): the global amax and scale follow the pinned per-tensor rules,
every payload is the pinned per-tensor cast, and for E4M3 the binary32 sum of the
decoded payloads is exact, so the result is the exact sum times scale_inv rounded
once, independent of rank order."""
import numpy as np
import pytest

import oracle


def rank_grads(k, n, seed, spread=True):
    rng = np.random.default_rng(seed)
    g = rng.standard_normal((k, n)).astype(np.float32)
    if spread:
        g *= (10.0 ** rng.uniform(-3, 1, (k, 1))).astype(np.float32)   # ranks of different magnitude
    return (g.view(np.uint32) >> 16).astype(np.uint16)


@pytest.mark.parametrize("k", [1, 2, 7, 64])
def test_allreduce_e4m3_is_exact_sum_times_scale_inv(k):
    g = rank_grads(k, 512, 40 + k)
    a, q, si, out = oracle.allreduce_sum(g, oracle.E4M3)
    assert a == oracle.amax(g)
    s, si_ref = oracle.tensor_scale(a, oracle.E4M3)
    assert si == si_ref
    q_ref, _ = oracle.quantize_rowwise(g, oracle.KIND_TENSOR, oracle.E4M3, s)
    assert np.array_equal(q, q_ref)
    exact = oracle.decode(q, oracle.E4M3).astype(np.float64).sum(axis=0)     # exact: E4M3 grid, k <= 64
    ref = (exact * np.float64(si)).astype(np.float32)                          # one rounding of an exact product
    assert np.array_equal(out, ref)
    # the same sum whatever the rank order
    perm = np.random.default_rng(k).permutation(k)
    assert np.array_equal(oracle.allreduce_sum(g[perm], oracle.E4M3)[3], out)


def test_allreduce_single_rank_is_the_per_tensor_round_trip():
    g = rank_grads(1, 1024, 50)
    a, q, si, out = oracle.allreduce_sum(g, oracle.E5M2)
    dec = oracle.decode(q[0], oracle.E5M2)
    assert np.array_equal(out, (dec.astype(np.float64) * np.float64(si)).astype(np.float32))
    # within half an FP8 step (relative 2^-3 for E5M2) of the input, nothing saturated
    x = (g[0].astype(np.uint32) << 16).view(np.float32)
    assert np.all(np.abs(out - x) <= np.abs(x) * 2.0 ** -3 + 2.0 ** -16 * si)


def test_allreduce_e5m2_sums_in_rank_order():
    # E5M2's range makes the binary32 sum inexact: the result is the rank-order sum
    g = rank_grads(3, 256, 51)
    a, q, si, out = oracle.allreduce_sum(g, oracle.E5M2)
    d = oracle.decode(q, oracle.E5M2)
    acc = np.zeros(256, np.float32)
    for r in range(3):
        acc = (acc + d[r]).astype(np.float32)
    assert np.array_equal(out, (acc * np.float32(si)).astype(np.float32))
    exact = d.astype(np.float64).sum(axis=0) * np.float64(si)
    assert np.all(np.abs(out - exact) <= 4 * np.spacing(np.abs(exact).astype(np.float32)) + 1e-30)
