"""Pins of the oracle's scaling recipes and GEMM against things other than itself.

Sources on the pages: per-tensor current and delayed scaling ("Colossal-AI FP8",
"current scaling" / "delayed scaling"; the guide's "tensor-level scaling"
section), blockwise 1x128 / 128x128 (the guide's "block-level scaling"),
MXFP8 1x32 with E8M0 scales (the guide's "MXFP8 scaling"), and the GEMM
dataflow (BF16 inputs quantized to FP8, FP32 accumulation, BF16 / FP32 out;
the search-result page's mixed-precision dataflow paragraph).
"""
from fractions import Fraction

import numpy as np
import pytest

import oracle
from conftest import golden_rows

FMT = {"e4m3": oracle.E4M3, "e5m2": oracle.E5M2}


def to_bf16_bits(x: np.ndarray) -> np.ndarray:
    """float32 -> bf16 bit patterns, round to nearest even (test-side helper)."""
    b = np.ascontiguousarray(x, np.float32).view(np.uint32).astype(np.uint64)
    rounded = (b + 0x7FFF + ((b >> 16) & 1)) >> 16
    return rounded.astype(np.uint16)


def bf16_to_f32(h: np.ndarray) -> np.ndarray:
    return (h.astype(np.uint32) << 16).view(np.float32)


def f32_from_bits(s):
    return np.array([int(s, 16)], np.uint32).view(np.float32)[0]


def bits_of(v):
    return int(np.array([v], np.float32).view(np.uint32)[0])


def randn_bf16(shape, seed, sigma=1.0):
    rng = np.random.default_rng(seed)
    return to_bf16_bits((rng.standard_normal(shape) * sigma).astype(np.float32))


# ----------------------------------------------------------------- amax
def test_amax_is_numpy_max_abs_and_order_free():
    x = randn_bf16((257, 129), 1)
    ref = np.max(np.abs(bf16_to_f32(x)))
    assert oracle.amax(x) == ref
    rng = np.random.default_rng(2)
    perm = rng.permutation(x.size)
    assert oracle.amax(x.reshape(-1)[perm].copy()) == ref
    # sign flips do not change it
    assert oracle.amax(x ^ np.uint16(0x8000)) == ref


def test_amax_ignores_nan_and_handles_specials():
    x = to_bf16_bits(np.array([1.0, -3.0, 2.0], np.float32))
    nan = np.array([0x7FC0, 0xFFC1], np.uint16)
    assert oracle.amax(np.concatenate([x, nan])) == 3.0
    assert oracle.amax(np.array([0x8000, 0x0000], np.uint16)) == 0.0      # -0, +0
    assert np.isinf(oracle.amax(np.array([0x3F80, 0xFF80], np.uint16)))   # 1, -inf
    assert oracle.amax(np.zeros(0, np.uint16)) == 0.0


def test_amax_f32_agrees_with_bf16_amax_and_is_order_free():
    # on bf16-representable values the float32 amax must equal the (pinned) bf16 one
    x = randn_bf16((129, 65), 3, 50.0)
    v = bf16_to_f32(x)
    assert oracle.amax_f32(v) == oracle.amax(x)
    rng = np.random.default_rng(4)
    w = (rng.standard_normal(4099) * 1e3).astype(np.float32)   # full float32 mantissas
    ref = np.max(np.abs(w))
    assert oracle.amax_f32(w) == ref
    assert oracle.amax_f32(-w[rng.permutation(w.size)]) == ref
    specials = np.array([np.nan, -0.0, 0.0, -7.5, np.float32(1e-45), -np.nan], np.float32)
    assert oracle.amax_f32(specials) == np.float32(7.5)
    assert np.isinf(oracle.amax_f32(np.array([1.0, -np.inf], np.float32)))
    assert oracle.amax_f32(np.zeros(0, np.float32)) == 0.0


# ----------------------------------------------------------------- scale
def test_tensor_scale_golden():
    for fmt, amax_b, s_b, si_b, *_ in golden_rows("tensor_scale.txt"):
        s, si = oracle.tensor_scale(f32_from_bits(amax_b), FMT[fmt])
        assert bits_of(s) == int(s_b, 16), (fmt, amax_b, hex(bits_of(s)))
        assert bits_of(si) == int(si_b, 16), (fmt, amax_b, hex(bits_of(si)))


@pytest.mark.parametrize("fmt", [oracle.E4M3, oracle.E5M2])
def test_tensor_scale_is_ieee_binary32_division(fmt):
    # library binary32 division (numpy) on many amax values, including subnormal ones
    rng = np.random.default_rng(3)
    amaxes = np.abs(rng.standard_normal(2000).astype(np.float32)) * np.exp2(
        rng.integers(-140, 100, 2000)).astype(np.float32)
    fmax = np.float32(oracle.fmax(fmt))
    with np.errstate(over="ignore", divide="ignore"):
        for a in amaxes:
            if not (a > 0 and np.isfinite(a)):
                continue
            s, si = oracle.tensor_scale(a, fmt)
            ref = fmax / np.float32(a)
            if np.isinf(ref):
                ref = np.finfo(np.float32).max
            assert bits_of(s) == bits_of(ref)
            assert bits_of(si) == bits_of(np.float32(1) / ref)


def test_current_scaling_never_saturates():
    # with scale = FMAX / amax, |x * scale| <= FMAX up to one rounding: the cast never clips
    for seed in range(5):
        x = randn_bf16((64, 96), 10 + seed, sigma=10.0 ** (seed - 2))
        for fmt in (oracle.E4M3, oracle.E5M2):
            s, _ = oracle.tensor_scale(oracle.amax(x), fmt)
            p = bf16_to_f32(x) * s
            assert np.max(np.abs(p)) <= np.float32(oracle.fmax(fmt)) * np.float32(1 + 2 ** -23)
            q, _ = oracle.quantize_rowwise(x, oracle.KIND_TENSOR, fmt, s)
            # the element holding the amax lands on (or within a rounding of) the largest code
            dq = np.abs(oracle.decode(q, fmt))
            assert dq.max() >= oracle.fmax(fmt) * (1 - 2 ** -3)


# ----------------------------------------------------------------- delayed
def test_delayed_history_hand_trace():
    st = oracle.DelayedState(16, oracle.E4M3)
    rows = golden_rows("delayed_history.txt")
    assert len(rows) == 32
    for step, amax_v, used, after, pos_after in rows:
        assert st.scale[0] == float(used), step
        st.step(np.float32(float(amax_v)))
        assert st.scale[0] == float(after), step
        assert st.scale_inv[0] == np.float32(1) / np.float32(float(after))
        assert st.pos[0] == int(pos_after), step


def test_delayed_checkpoint_resume_is_bit_identical():
    rng = np.random.default_rng(4)
    amaxes = (np.abs(rng.standard_normal(32)) * 3 + 0.1).astype(np.float32)
    full = oracle.DelayedState(16)
    for a in amaxes:
        full.step(a)
    first = oracle.DelayedState(16)
    for a in amaxes[:16]:
        first.step(a)
    resumed = first.copy()
    for a in amaxes[16:]:
        resumed.step(a)
    np.testing.assert_array_equal(resumed.hist, full.hist)
    assert resumed.pos[0] == full.pos[0]
    assert bits_of(resumed.scale[0]) == bits_of(full.scale[0])


def test_delayed_zero_window_keeps_scale():
    st = oracle.DelayedState(4)
    st.step(np.float32(0))
    assert st.scale[0] == 1.0 and st.pos[0] == 1


# ----------------------------------------------------------------- MX
def test_mx_exponent_golden():
    for fmt, amax_b, e, *_ in golden_rows("mx_exponent.txt"):
        assert oracle.mx_exponent(f32_from_bits(amax_b), FMT[fmt]) == int(e), (fmt, amax_b)


@pytest.mark.parametrize("fmt", [oracle.E4M3, oracle.E5M2])
def test_mx_exponent_is_minimal_power_of_two(fmt):
    rng = np.random.default_rng(5)
    fmax = oracle.fmax(fmt)
    vals = np.abs(rng.standard_normal(3000)).astype(np.float32) * np.exp2(
        rng.integers(-120, 120, 3000)).astype(np.float32)
    # exact boundaries fmax * 2^k and their binary32 neighbours
    for k in range(-100, 100, 7):
        b = np.float32(np.ldexp(fmax, k))
        vals = np.concatenate([vals, [b, np.nextafter(b, np.float32(0)), np.nextafter(b, np.float32(np.inf))]])
    for a in vals.astype(np.float32):
        if not (a > 0 and np.isfinite(a)):
            continue
        e = oracle.mx_exponent(a, fmt)
        assert -127 <= e <= 127
        if -127 < e:
            assert Fraction(float(a)) > Fraction(fmax) * Fraction(2) ** (e - 1)
        if e < 127:
            assert Fraction(float(a)) <= Fraction(fmax) * Fraction(2) ** e


# ----------------------------------------------------------------- recipes
def _check_block_recipe(x, q, s_inv, fmt, block_rows, block_cols):
    """Invariants of a FP32-scaled block recipe, checked block by block with numpy."""
    xf = bf16_to_f32(x).astype(np.float64)
    dq = oracle.decode(q, fmt).astype(np.float64)
    R, C = x.shape
    fmax = oracle.fmax(fmt)
    for br in range(R // block_rows):
        for bc in range(C // block_cols):
            sl = (slice(br * block_rows, (br + 1) * block_rows), slice(bc * block_cols, (bc + 1) * block_cols))
            blk = xf[sl]
            amax = np.max(np.abs(blk))
            si = s_inv[br, bc] if s_inv.ndim == 2 else s_inv[br * (C // block_cols) + bc]
            if amax == 0:
                assert si == 1.0
                continue
            # the stored multiplier is the reciprocal of FMAX/amax (so about amax/FMAX)
            assert abs(si * fmax / amax - 1) < 2 ** -22
            # the largest element maps to the top of the range
            assert np.max(np.abs(dq[sl])) >= fmax * (1 - 2 ** -3)
            # dequantized values are within half an FP8 step (relative 2^-4, E4M3) or the
            # subnormal spacing of the original values
            sub = 2.0 ** -9 if fmt == oracle.E4M3 else 2.0 ** -16
            rel = 2.0 ** -4 if fmt == oracle.E4M3 else 2.0 ** -3
            err = np.abs(dq[sl] * si - blk)
            assert np.all(err <= np.maximum(rel * np.abs(blk), sub * si) * (1 + 1e-5))


def test_blockwise_1x128_rows_are_independent_tiles():
    x = randn_bf16((8, 384), 6)
    x[3, 128:256] = to_bf16_bits(bf16_to_f32(x[3, 128:256]) * 100)   # an outlier tile
    q, s = oracle.quantize_rowwise(x, oracle.KIND_1x128, oracle.E4M3)
    assert s.shape == (8, 3)
    _check_block_recipe(x, q, s, oracle.E4M3, 1, 128)
    # changing one tile changes only that tile's bytes and scale
    x2 = x.copy()
    x2[3, 130] = to_bf16_bits(np.array([1000.0], np.float32))[0]
    q2, s2 = oracle.quantize_rowwise(x2, oracle.KIND_1x128, oracle.E4M3)
    diff = np.argwhere(q2 != q)
    assert np.all(diff[:, 0] == 3) and np.all((diff[:, 1] >= 128) & (diff[:, 1] < 256))
    assert np.argwhere(s2 != s).tolist() == [[3, 1]]


def test_blockwise_128x128_and_transpose_relation():
    x = randn_bf16((256, 384), 7, sigma=0.02)
    q, s = oracle.quantize_rowwise(x, oracle.KIND_128x128, oracle.E4M3)
    assert s.shape == (2, 3)
    _check_block_recipe(x, q, s, oracle.E4M3, 128, 128)
    qc, sc = oracle.quantize_colwise(x, oracle.KIND_128x128, oracle.E4M3)
    # the column-wise copy of a 128x128-scaled matrix is the transpose, scales transposed
    np.testing.assert_array_equal(qc, q.T)
    np.testing.assert_array_equal(sc, s.T)


def test_colwise_1x128_runs_along_rows():
    x = randn_bf16((256, 128), 8)
    x[0:128, 5] = to_bf16_bits(bf16_to_f32(x[0:128, 5]) * 50)
    qc, sc = oracle.quantize_colwise(x, oracle.KIND_1x128, oracle.E4M3)
    assert qc.shape == (128, 256) and sc.shape == (128, 2)
    xt = np.ascontiguousarray(x.T)
    _check_block_recipe(xt, qc, sc, oracle.E4M3, 1, 128)
    # column 5's first row tile has the outlier scale, its second tile does not
    assert sc[5, 0] > 10 * sc[5, 1]


@pytest.mark.parametrize("fmt", [oracle.E4M3, oracle.E5M2])
def test_per_tensor_matches_library_cast(fmt):
    ml_dtypes = pytest.importorskip("ml_dtypes")
    x = randn_bf16((33, 47), 9)
    s, si = oracle.tensor_scale(oracle.amax(x), fmt)
    q, sq = oracle.quantize_rowwise(x, oracle.KIND_TENSOR, fmt, s)
    t = ml_dtypes.float8_e4m3fn if fmt == oracle.E4M3 else ml_dtypes.float8_e5m2
    fmax = np.float32(oracle.fmax(fmt))
    p = np.clip(bf16_to_f32(x) * np.float32(s), -fmax, fmax).astype(np.float32)
    np.testing.assert_array_equal(q, p.astype(t).view(np.uint8))
    assert sq[0] == si
    qc, _ = oracle.quantize_colwise(x, oracle.KIND_TENSOR, fmt, s)
    np.testing.assert_array_equal(qc, q.T)


def test_mx_blocks_power_of_two_and_no_saturation():
    ml_dtypes = pytest.importorskip("ml_dtypes")
    x = randn_bf16((16, 256), 11)
    x[2, 64:96] = to_bf16_bits(bf16_to_f32(x[2, 64:96]) * 1000)
    x[5, 0:32] = 0
    q, e8 = oracle.quantize_rowwise(x, oracle.KIND_MX, oracle.E4M3)
    assert e8.shape == (16, 8) and e8.dtype == np.uint8
    assert e8[5, 0] == 127                      # zero block: scale 2^0 (reading)
    xf = bf16_to_f32(x)
    for r in range(16):
        for b in range(8):
            blk = xf[r, b * 32:(b + 1) * 32]
            e = int(e8[r, b]) - 127
            # the block after scaling by 2^-e stays within FMAX: the cast never clips
            assert np.max(np.abs(blk)) <= 448.0 * 2.0 ** e
            # library cast of the exactly scaled block reproduces the bytes
            ref = (blk * np.float32(2.0 ** -e)).astype(np.float32).astype(ml_dtypes.float8_e4m3fn).view(np.uint8)
            np.testing.assert_array_equal(q[r, b * 32:(b + 1) * 32], ref)
    assert e8[2, 2] > e8[2, 1]


# ----------------------------------------------------------------- GEMM
def _brute_force_gemm(qa, fa, ka, sa, qb, fb, kb, sb):
    """Exact rational C from FP8 codes decoded by ml_dtypes and the stored scales."""
    ml_dtypes = pytest.importorskip("ml_dtypes")

    def dec(q, f):
        t = ml_dtypes.float8_e4m3fn if f == oracle.E4M3 else ml_dtypes.float8_e5m2
        return q.view(t).astype(np.float64)

    def mult(kind, s, r, c):
        if kind == oracle.KIND_TENSOR:
            return Fraction(float(s[0]))
        if kind == oracle.KIND_1x128:
            return Fraction(float(s[r, c // 128]))
        if kind == oracle.KIND_128x128:
            return Fraction(float(s[r // 128, c // 128]))
        return Fraction(2) ** (int(s[r, c // 32]) - 127)

    A, B = dec(qa, fa), dec(qb, fb)
    M, K = A.shape
    N = B.shape[0]
    C = np.empty((M, N), np.float64)
    for m in range(M):
        for n in range(N):
            acc = Fraction(0)
            for k in range(K):
                acc += Fraction(A[m, k]) * mult(ka, sa, m, k) * Fraction(B[n, k]) * mult(kb, sb, n, k)
            C[m, n] = float(acc)
    return C


@pytest.mark.parametrize("combo", ["tensor", "1x128_128x128", "1x128_1x128", "mx"])
def test_gemm_matches_exact_rational_brute_force(combo):
    rng = np.random.default_rng(12)
    M, N, K = 3, 2, 256
    qa = rng.integers(0, 256, (M, K), dtype=np.uint8)
    qb = rng.integers(0, 256, (N, K), dtype=np.uint8)
    qa[(qa & 0x7F) >= 0x7F] = 0x11        # no NaN codes in E4M3 operands
    qb[(qb & 0x7C) == 0x7C] = 0x22        # no inf/NaN codes in E5M2 operands
    fa, fb = oracle.E4M3, oracle.E5M2
    if combo == "tensor":
        ka = kb = oracle.KIND_TENSOR
        sa = np.array([0.37], np.float32)
        sb = np.array([1.9e-3], np.float32)
    elif combo == "1x128_128x128":
        # pad to 128 rows for the 128x128 B scale grid (only N rows are used)
        ka, kb = oracle.KIND_1x128, oracle.KIND_128x128
        sa = rng.uniform(0.1, 4, (M, K // 128)).astype(np.float32)
        sb = rng.uniform(0.1, 4, (1, K // 128)).astype(np.float32)
    elif combo == "1x128_1x128":
        ka = kb = oracle.KIND_1x128
        sa = rng.uniform(0.1, 4, (M, K // 128)).astype(np.float32)
        sb = rng.uniform(0.1, 4, (N, K // 128)).astype(np.float32)
    else:
        ka = kb = oracle.KIND_MX
        sa = rng.integers(100, 150, (M, K // 32), dtype=np.uint8)
        sb = rng.integers(100, 150, (N, K // 32), dtype=np.uint8)
    got = oracle.scaled_gemm(qa, fa, ka, sa, qb, fb, kb, sb)
    ref = _brute_force_gemm(qa, fa, ka, sa, qb, fb, kb, sb)
    np.testing.assert_allclose(got, ref, rtol=1e-13, atol=1e-300)


def test_gemm_unit_scales_is_textbook_matmul():
    ml_dtypes = pytest.importorskip("ml_dtypes")
    rng = np.random.default_rng(13)
    qa = rng.integers(0, 0x7E, (5, 64), dtype=np.uint8)
    qb = rng.integers(0x80, 0xFE, (4, 64), dtype=np.uint8)
    one = np.array([1.0], np.float32)
    got = oracle.scaled_gemm(qa, oracle.E4M3, 0, one, qb, oracle.E4M3, 0, one)
    A = qa.view(ml_dtypes.float8_e4m3fn).astype(np.float64)
    B = qb.view(ml_dtypes.float8_e4m3fn).astype(np.float64)
    np.testing.assert_allclose(got, A @ B.T, rtol=1e-14)


def test_gemm_row_sampling_matches_full():
    x = randn_bf16((256, 256), 14)
    w = randn_bf16((128, 256), 15, 0.02)
    qa, sa = oracle.quantize_rowwise(x, oracle.KIND_1x128, oracle.E4M3)
    qb, sb = oracle.quantize_rowwise(w, oracle.KIND_128x128, oracle.E4M3)
    full = oracle.scaled_gemm(qa, 0, 1, sa, qb, 0, 2, sb)
    rows = [0, 7, 200, 255]
    part = oracle.scaled_gemm_rows(qa, 0, 1, sa, qb, 0, 2, sb, rows)
    # float64 matmuls of different shapes may block the sums differently
    np.testing.assert_allclose(part, full[rows], rtol=1e-12, atol=1e-15)


def test_quantized_gemm_close_to_bf16_gemm():
    # end-to-end sanity of quantize + GEMM against the unquantized product
    x = randn_bf16((128, 512), 16)
    w = randn_bf16((128, 512), 17, 0.02)
    qa, sa = oracle.quantize_rowwise(x, oracle.KIND_1x128, oracle.E4M3)
    qb, sb = oracle.quantize_rowwise(w, oracle.KIND_128x128, oracle.E4M3)
    c = oracle.scaled_gemm(qa, 0, 1, sa, qb, 0, 2, sb)
    ref = bf16_to_f32(x).astype(np.float64) @ bf16_to_f32(w).astype(np.float64).T
    rel = np.linalg.norm(c - ref) / np.linalg.norm(ref)
    assert rel < 0.05


def test_tolerance_check_detects_planted_errors():
    x = randn_bf16((128, 256), 18)
    w = randn_bf16((64, 256), 19, 0.02)
    qa, sa = oracle.quantize_rowwise(x, oracle.KIND_1x128, oracle.E4M3)
    qb, sb = oracle.quantize_rowwise(w, oracle.KIND_1x128, oracle.E4M3)
    ref = oracle.scaled_gemm(qa, 0, 1, sa, qb, 0, 1, sb)
    da, db = oracle.dequantize(qa, 1, 0, sa), oracle.dequantize(qb, 1, 0, sb)
    rel, worst = oracle.gemm_tolerance_check(ref.astype(np.float32), ref, da, db)
    assert rel < 1e-6 and worst < 1e-3
    bad = ref.copy()
    bad[5, 7] += 0.5 * np.abs(ref).max()
    assert oracle.gemm_tolerance_check(bad, ref, da, db)[1] > 1
    # a transposed-scale mistake (using B's scales for the wrong rows) is caught
    wrong = oracle.scaled_gemm(qa, 0, 1, sa, qb, 0, 1, sb[::-1].copy())
    rel_w, worst_w = oracle.gemm_tolerance_check(wrong, ref, da, db)
    assert rel_w > 1e-2 or worst_w > 1


# ----------------------------------------------------------------- MX tiled layout
def test_mx_tiled_layout_is_a_bijection_with_hand_positions():
    R, C = 256, 384
    off = oracle.mx_tiled_offsets(R, C)
    assert off.shape == (256, 12)
    assert np.array_equal(np.sort(off.ravel()), np.arange(R * C // 32))
    # hand-computed: row 0 block 0 -> 0; row 1 -> 16; row 32 -> 4; row 96 block 3 -> 15;
    # row 31 block 2 -> 31*16 + 2; row 128 block 0 -> atom (1, 0) -> 3*512; block 4 -> atom (0, 1) -> 512
    assert off[0, 0] == 0 and off[1, 0] == 16 and off[32, 0] == 4 and off[96, 3] == 15
    assert off[31, 2] == 31 * 16 + 2 and off[128, 0] == 3 * 512 and off[0, 4] == 512
    s = np.random.default_rng(0).integers(0, 255, (R, C // 32), dtype=np.uint8)
    np.testing.assert_array_equal(oracle.mx_from_tiled(oracle.mx_to_tiled(s), R, C), s)
