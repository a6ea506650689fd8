"""Helpers for the GPU parity tests (CUDA path vs the CPU oracle)."""
import numpy as np
import torch

import oracle
import scaled_quantize_gemm_amax_gb300 as fq
from scaled_quantize_gemm_amax_gb300 import build as fqbuild

R = fq.Recipe
F = fq.Format

KIND = {R.TENSOR: oracle.KIND_TENSOR, R.BLOCK_1x128: oracle.KIND_1x128, R.BLOCK_128x128: oracle.KIND_128x128,
        R.MX_1x32: oracle.KIND_MX, R.MX_1x32_TILED: oracle.KIND_MX, R.MX_1x32_FLOOR: oracle.KIND_MX_FLOOR,
        R.MX_1x32_FLOOR_TILED: oracle.KIND_MX_FLOOR}
MX_RECIPES = (R.MX_1x32, R.MX_1x32_TILED, R.MX_1x32_FLOOR, R.MX_1x32_FLOOR_TILED)
MX_TILED = (R.MX_1x32_TILED, R.MX_1x32_FLOOR_TILED)


def require_gpu():
    assert torch.cuda.is_available(), "the -m gpu tests need a CUDA device"
    fqbuild.build()
    fq.load_library()


def bits16(x: torch.Tensor) -> np.ndarray:
    return x.contiguous().view(torch.int16).cpu().numpy().view(np.uint16)


def host(t: torch.Tensor) -> np.ndarray:
    return t.detach().cpu().numpy()


def f32bits(a) -> np.ndarray:
    return np.ascontiguousarray(np.asarray(a, dtype=np.float32)).view(np.uint32)


def assert_bytes_equal(got: np.ndarray, ref: np.ndarray, what: str):
    got = np.asarray(got)
    ref = np.asarray(ref)
    assert got.shape == ref.shape, (what, got.shape, ref.shape)
    bad = np.argwhere(got != ref)
    if bad.size:
        idx = tuple(bad[0])
        raise AssertionError(f"{what}: {len(bad)} of {ref.size} differ; first at {idx}: got {got[idx]!r} "
                             f"ref {ref[idx]!r}")


def assert_status_ok():
    st = fq.fp8_get_device_status()
    assert st == fq.Status.OK, st


def oracle_scales_like(recipe, s_ref, rows, cols):
    """Oracle multipliers in the layout the GPU writes (MX tiled: permuted)."""
    if recipe in MX_TILED:
        return oracle.mx_to_tiled(s_ref).reshape(((rows + 127) // 128, (cols + 127) // 128, 512))
    return s_ref


def check_cast(x: torch.Tensor, recipe, fmt, row=True, col=True, scale_np=None):
    """Run the GPU cast-transpose and compare every output with the oracle.

    For the per-tensor recipe the scale is the oracle's current-scaling scale of x
    unless ``scale_np`` is given.  Returns the GPU outputs.
    """
    xh = bits16(x)
    rows, cols = xh.shape
    kind = KIND[recipe]
    scale_t = None
    if recipe == R.TENSOR:
        if scale_np is None:
            scale_np, _ = oracle.tensor_scale(oracle.amax(xh), int(fmt))
        scale_t = torch.tensor([scale_np], dtype=torch.float32, device=x.device)
    amax_t = torch.full((1,), 123.0, dtype=torch.float32, device=x.device)
    qr, sr, qc, sc = fq.cast_transpose(x, recipe, fmt, scale_t, amax_t, row=row, col=col)
    torch.cuda.synchronize()
    assert_status_ok()
    assert f32bits(host(amax_t))[0] == f32bits(oracle.amax(xh)), "amax_out"
    if row:
        q_ref, s_ref = oracle.quantize_rowwise(xh, kind, int(fmt), scale_np)
        assert_bytes_equal(host(qr), q_ref, "q_row")
        _check_scales(recipe, host(sr), oracle_scales_like(recipe, s_ref, rows, cols), "s_row")
    if col:
        q_ref, s_ref = oracle.quantize_colwise(xh, kind, int(fmt), scale_np)
        assert_bytes_equal(host(qc), q_ref, "q_col")
        _check_scales(recipe, host(sc), oracle_scales_like(recipe, s_ref, cols, rows), "s_col")
    return qr, sr, qc, sc


def _check_scales(recipe, got, ref, what):
    if recipe in MX_RECIPES:
        assert_bytes_equal(got, ref, what)
    else:
        assert_bytes_equal(f32bits(got), f32bits(ref), what)


def tile_spread(t: torch.Tensor, bh: int, bw: int, seed: int, span: int) -> torch.Tensor:
    """Multiply each bh x bw tile of t by its own power of two 2^e, e in [-span, span]
    (exact in BF16), so that a scale read for the wrong tile (row block, column block
    or k-block) is off by a factor of 2 or more instead of a few per cent."""
    r, c = t.shape
    i = torch.arange((r + bh - 1) // bh, device=t.device)[:, None]
    j = torch.arange((c + bw - 1) // bw, device=t.device)[None, :]
    e = (i * 3 + j * 5 + seed) % (2 * span + 1) - span
    f = torch.exp2(e.float()).repeat_interleave(bh, 0)[:r].repeat_interleave(bw, 1)[:, :c]
    return (t.float() * f).to(torch.bfloat16)


SENTINEL = 0xA5


class Guarded:
    """An output buffer with guard regions before and after it, every byte (the
    buffer's own included) filled with SENTINEL before the call: check() finds any
    write outside the buffer, which a comparison of the buffer alone cannot see."""

    def __init__(self, shape, dtype, guard_bytes: int = 4096, device="cuda"):
        esz = torch.empty((), dtype=dtype).element_size()
        self.n = 1
        for d in shape:
            self.n *= int(d)
        self.g = guard_bytes // esz
        self.esz = esz
        self.buf = torch.empty(2 * self.g + self.n, dtype=dtype, device=device)
        self.buf.view(torch.uint8).fill_(SENTINEL)
        self.t = self.buf[self.g:self.g + self.n].view(tuple(shape))

    def check(self, what: str):
        b = host(self.buf.view(torch.uint8))
        gb, nb = self.g * self.esz, self.n * self.esz
        before = np.flatnonzero(b[:gb] != SENTINEL)
        after = np.flatnonzero(b[gb + nb:] != SENTINEL)
        assert before.size == 0, f"{what}: {before.size} bytes written before the buffer (first at -{gb - before[0]})"
        assert after.size == 0, f"{what}: {after.size} bytes written past the end (first at +{after[0]})"
