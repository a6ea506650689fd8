"""CPU oracle for FP8 scaled quantization and the scaled FP8 GEMM.

TEST INFRASTRUCTURE ONLY: the test suite, ``__graft_entry__.smoke()`` and the
benchmark's CPU-baseline / reference leg are the only callers.  The product
path (the CUDA library and its binding) never imports this package, and this
package never imports the product path.

The element-wise arithmetic lives in ``fp8_oracle.c`` (plain C, compiled here
with gcc on first use).  This module only marshals numpy arrays and adds the
two compositions the pages describe:

* column-wise copies: the column-wise output of every recipe is the row-wise
  recipe applied to the transposed matrix (reading: "1x128 for activations and
  gradients" tiles run along the contiguous dimension of whichever copy is
  stored, so the transposed copy gets tiles along the original rows);
* the scaled GEMM: dequantize both operands exactly to float64 and multiply
  with a library float64 matmul (C = deq(A) . deq(B)^T, FP32 accumulation on
  the GPU is checked against this within the stated tolerance).

Recipe kinds (the ``kind`` argument of ``dequantize``): 0 per-tensor,
1 blockwise 1x128, 2 blockwise 128x128, 3 MXFP8 1x32 (E8M0).
"""
from __future__ import annotations

import ctypes
import os
import subprocess
import threading

import numpy as np

E4M3, E5M2 = 0, 1
KIND_TENSOR, KIND_1x128, KIND_128x128, KIND_MX = 0, 1, 2, 3
# MXFP8 with the floor-rule exponent (the documented alternate); its E8M0 scales are
# read like KIND_MX's everywhere else (dequantize, GEMM)
KIND_MX_FLOOR = 4

_HERE = os.path.dirname(os.path.abspath(__file__))
_SRC = os.path.join(_HERE, "fp8_oracle.c")
_BUILD = os.path.join(_HERE, "_build")
_LIB_PATH = os.path.join(_BUILD, "liboracle.so")
CFLAGS = ["-O2", "-std=c11", "-fPIC", "-shared", "-ffp-contract=off", "-fno-fast-math",
           "-fexcess-precision=standard", "-Wall", "-Wextra"]

_lib = None
_lock = threading.Lock()


def build(force: bool = False) -> str:
    """Compile the C oracle into ``oracle/_build/liboracle.so`` (if stale).

    FP8_ORACLE_LIB, when set, names an already-built oracle library to load
    instead (the mutation test loads deliberately broken copies this way)."""
    alt = os.environ.get("FP8_ORACLE_LIB")
    if alt:
        return alt
    os.makedirs(_BUILD, exist_ok=True)
    if (not force and os.path.exists(_LIB_PATH)
            and os.path.getmtime(_LIB_PATH) >= os.path.getmtime(_SRC)):
        return _LIB_PATH
    tmp = _LIB_PATH + f".tmp{os.getpid()}"
    subprocess.run(["gcc", *CFLAGS, _SRC, "-o", tmp, "-lm"], check=True)
    os.replace(tmp, _LIB_PATH)
    return _LIB_PATH


def _load():
    global _lib
    with _lock:
        if _lib is not None:
            return _lib
        lib = ctypes.CDLL(build())
        P = ctypes.c_void_p
        I64, I32, F = ctypes.c_int64, ctypes.c_int32, ctypes.c_float
        sig = {
            "orc_fmax": (F, [ctypes.c_int]),
            "orc_decode": (F, [ctypes.c_uint8, ctypes.c_int]),
            "orc_encode": (ctypes.c_uint8, [F, ctypes.c_int, ctypes.c_int]),
            "orc_decode_array": (None, [P, I64, ctypes.c_int, P]),
            "orc_encode_array": (None, [P, I64, ctypes.c_int, ctypes.c_int, P]),
            "orc_amax_bf16": (F, [P, I64]),
            "orc_amax_f32": (F, [P, I64]),
            "orc_round_bf16": (ctypes.c_uint16, [ctypes.c_double]),
            "orc_allreduce_sum": (None, [P, I32, I64, ctypes.c_int, P, P, P, P]),
            "orc_dequantize_bf16": (None, [P, I64, I64, ctypes.c_int, ctypes.c_int, P, P]),
            "orc_tensor_scale": (None, [F, ctypes.c_int, P, P]),
            "orc_history_step": (None, [P, I32, P, F, ctypes.c_int, P, P]),
            "orc_mx_exponent": (ctypes.c_int, [F, ctypes.c_int]),
            "orc_mx_exponent_floor": (ctypes.c_int, [F, ctypes.c_int]),
            "orc_quantize_mx_floor": (None, [P, I64, I64, ctypes.c_int, P, P]),
            "orc_quantize_mx_floor_f32": (None, [P, I64, I64, ctypes.c_int, P, P]),
            "orc_quantize_tensor": (None, [P, I64, I64, ctypes.c_int, F, P]),
            "orc_quantize_1x128": (None, [P, I64, I64, ctypes.c_int, P, P]),
            "orc_quantize_128x128": (None, [P, I64, I64, ctypes.c_int, P, P]),
            "orc_quantize_mx": (None, [P, I64, I64, ctypes.c_int, P, P]),
            "orc_transpose_bf16": (None, [P, I64, I64, P]),
            "orc_quantize_tensor_f32": (None, [P, I64, I64, ctypes.c_int, F, P]),
            "orc_quantize_1x128_f32": (None, [P, I64, I64, ctypes.c_int, P, P]),
            "orc_quantize_128x128_f32": (None, [P, I64, I64, ctypes.c_int, P, P]),
            "orc_quantize_mx_f32": (None, [P, I64, I64, ctypes.c_int, P, P]),
            "orc_transpose_f32": (None, [P, I64, I64, P]),
            "orc_dequantize": (None, [P, I64, I64, ctypes.c_int, ctypes.c_int, P, P]),
        }
        for name, (res, args) in sig.items():
            fn = getattr(lib, name)
            fn.restype = res
            fn.argtypes = args
        _lib = lib
        return lib


def _ptr(a: np.ndarray):
    assert a.flags["C_CONTIGUOUS"]
    return a.ctypes.data_as(ctypes.c_void_p)


def _bf16_bits(x) -> np.ndarray:
    """Accept a uint16 array of bf16 bit patterns (the only bf16 carrier here)."""
    x = np.ascontiguousarray(x)
    if x.dtype != np.uint16:
        raise TypeError("bf16 inputs are passed as uint16 bit patterns")
    return x


# ----------------------------------------------------------------- formats
def fmax(fmt: int) -> float:
    return float(_load().orc_fmax(fmt))


def decode(codes, fmt: int) -> np.ndarray:
    """FP8 codes (uint8) -> float32 values (exact)."""
    q = np.ascontiguousarray(codes, dtype=np.uint8)
    out = np.empty(q.shape, dtype=np.float32)
    _load().orc_decode_array(_ptr(q), q.size, fmt, _ptr(out))
    return out


def encode(values, fmt: int, saturate: bool) -> np.ndarray:
    """float32 values -> FP8 codes, round-to-nearest-even (see fp8_oracle.c)."""
    v = np.ascontiguousarray(values, dtype=np.float32)
    out = np.empty(v.shape, dtype=np.uint8)
    _load().orc_encode_array(_ptr(v), v.size, fmt, int(bool(saturate)), _ptr(out))
    return out


# ----------------------------------------------------------------- scaling
def amax(x_bf16) -> np.float32:
    x = _bf16_bits(x_bf16)
    return np.float32(_load().orc_amax_bf16(_ptr(x), x.size))


def amax_f32(values) -> np.float32:
    """max |v| over float32 values, NaN ignored (fp8_oracle.c: orc_amax_f32)."""
    v = np.ascontiguousarray(values, dtype=np.float32)
    return np.float32(_load().orc_amax_f32(_ptr(v), v.size))


def tensor_scale(amax_value, fmt: int):
    """Per-tensor current scaling: (scale, scale_inv) as float32."""
    s = np.zeros(1, np.float32)
    si = np.zeros(1, np.float32)
    _load().orc_tensor_scale(ctypes.c_float(float(np.float32(amax_value))), fmt, _ptr(s), _ptr(si))
    return s[0], si[0]


class DelayedState:
    """Delayed-scaling state {hist[len], pos, scale, scale_inv}, initial scale 1."""

    def __init__(self, length: int = 16, fmt: int = E4M3):
        self.hist = np.zeros(length, np.float32)
        self.pos = np.zeros(1, np.int32)
        self.scale = np.ones(1, np.float32)
        self.scale_inv = np.ones(1, np.float32)
        self.fmt = fmt

    def step(self, amax_value) -> None:
        _load().orc_history_step(_ptr(self.hist), self.hist.size, _ptr(self.pos),
                                 ctypes.c_float(float(np.float32(amax_value))), self.fmt,
                                 _ptr(self.scale), _ptr(self.scale_inv))

    def copy(self) -> "DelayedState":
        c = DelayedState(self.hist.size, self.fmt)
        c.hist[:] = self.hist
        c.pos[:] = self.pos
        c.scale[:] = self.scale
        c.scale_inv[:] = self.scale_inv
        return c


def mx_exponent(amax_value, fmt: int) -> int:
    return int(_load().orc_mx_exponent(ctypes.c_float(float(np.float32(amax_value))), fmt))


def mx_exponent_floor(amax_value, fmt: int) -> int:
    """The floor-rule MX exponent (fp8_oracle.c: orc_mx_exponent_floor)."""
    return int(_load().orc_mx_exponent_floor(ctypes.c_float(float(np.float32(amax_value))), fmt))


# ----------------------------------------------------------------- quantize
def transpose_bf16(x_bf16) -> np.ndarray:
    x = _bf16_bits(x_bf16)
    R, C = x.shape
    out = np.empty((C, R), np.uint16)
    _load().orc_transpose_bf16(_ptr(x), R, C, _ptr(out))
    return out


def quantize_rowwise(x_bf16, kind: int, fmt: int, scale=None):
    """Row-wise quantize of a [R, C] bf16 matrix.

    Returns (q uint8 [R, C], s) with s the stored dequantization multipliers:
    per-tensor: float32 [1] (scale_inv); 1x128: float32 [R, C/128];
    128x128: float32 [R/128, C/128]; MX: uint8 E8M0 [R, C/32].
    ``scale`` (float32) is required for the per-tensor kind only.
    """
    x = _bf16_bits(x_bf16)
    R, C = x.shape
    q = np.empty((R, C), np.uint8)
    lib = _load()
    if kind == KIND_TENSOR:
        sc = np.float32(scale)
        lib.orc_quantize_tensor(_ptr(x), R, C, fmt, ctypes.c_float(float(sc)), _ptr(q))
        s = np.array([np.float32(1.0) / sc], np.float32)
    elif kind == KIND_1x128:
        s = np.empty((R, C // 128), np.float32)
        lib.orc_quantize_1x128(_ptr(x), R, C, fmt, _ptr(q), _ptr(s))
    elif kind == KIND_128x128:
        s = np.empty((R // 128, C // 128), np.float32)
        lib.orc_quantize_128x128(_ptr(x), R, C, fmt, _ptr(q), _ptr(s))
    elif kind == KIND_MX:
        s = np.empty((R, C // 32), np.uint8)
        lib.orc_quantize_mx(_ptr(x), R, C, fmt, _ptr(q), _ptr(s))
    elif kind == KIND_MX_FLOOR:
        s = np.empty((R, C // 32), np.uint8)
        lib.orc_quantize_mx_floor(_ptr(x), R, C, fmt, _ptr(q), _ptr(s))
    else:
        raise ValueError(kind)
    return q, s


def quantize_colwise(x_bf16, kind: int, fmt: int, scale=None):
    """Column-wise copy: the row-wise recipe applied to the transposed matrix."""
    return quantize_rowwise(transpose_bf16(x_bf16), kind, fmt, scale)


def _f32(x) -> np.ndarray:
    x = np.ascontiguousarray(x)
    if x.dtype != np.float32:
        raise TypeError("binary32 inputs are passed as float32 arrays")
    return x


def transpose_f32(x_f32) -> np.ndarray:
    x = _f32(x_f32)
    R, C = x.shape
    out = np.empty((C, R), np.float32)
    _load().orc_transpose_f32(_ptr(x), R, C, _ptr(out))
    return out


def quantize_rowwise_f32(x_f32, kind: int, fmt: int, scale=None):
    """Row-wise quantize of a [R, C] binary32 matrix (the FP32 master copy of a weight):
    the same recipes and outputs as quantize_rowwise, element rule
    encode_sat(x * scale) with x the binary32 value itself."""
    x = _f32(x_f32)
    R, C = x.shape
    q = np.empty((R, C), np.uint8)
    lib = _load()
    if kind == KIND_TENSOR:
        sc = np.float32(scale)
        lib.orc_quantize_tensor_f32(_ptr(x), R, C, fmt, ctypes.c_float(float(sc)), _ptr(q))
        s = np.array([np.float32(1.0) / sc], np.float32)
    elif kind == KIND_1x128:
        s = np.empty((R, C // 128), np.float32)
        lib.orc_quantize_1x128_f32(_ptr(x), R, C, fmt, _ptr(q), _ptr(s))
    elif kind == KIND_128x128:
        s = np.empty((R // 128, C // 128), np.float32)
        lib.orc_quantize_128x128_f32(_ptr(x), R, C, fmt, _ptr(q), _ptr(s))
    elif kind == KIND_MX:
        s = np.empty((R, C // 32), np.uint8)
        lib.orc_quantize_mx_f32(_ptr(x), R, C, fmt, _ptr(q), _ptr(s))
    elif kind == KIND_MX_FLOOR:
        s = np.empty((R, C // 32), np.uint8)
        lib.orc_quantize_mx_floor_f32(_ptr(x), R, C, fmt, _ptr(q), _ptr(s))
    else:
        raise ValueError(kind)
    return q, s


def quantize_colwise_f32(x_f32, kind: int, fmt: int, scale=None):
    """Column-wise copy of a binary32 matrix: the row-wise recipe on its transpose."""
    return quantize_rowwise_f32(transpose_f32(x_f32), kind, fmt, scale)


# ----------------------------------------------------------------- MX tiled layout
def mx_tiled_offsets(rows: int, cols: int) -> np.ndarray:
    """Byte offset of exponent (r, b) (b = 32-column block) in the GEMM-ready tiled
    layout of a row-wise MX copy [rows, cols]: atoms of 128 rows x 4 blocks, 512 B
    each, atom (r/128, b/4) at ((r/128) * ceil(cols/128) + b/4) * 512, and inside an
    atom (r%32)*16 + ((r%128)/32)*4 + b%4 (the 32x4x4 arrangement the block-scaled
    MMA's scale-factor copy reads)."""
    r = np.arange(rows, dtype=np.int64)[:, None]
    b = np.arange(cols // 32, dtype=np.int64)[None, :]
    apr = (cols + 127) // 128
    return ((r // 128) * apr + b // 4) * 512 + (r % 32) * 16 + ((r % 128) // 32) * 4 + (b % 4)


def mx_to_tiled(s_rowmajor: np.ndarray) -> np.ndarray:
    rows, nb = s_rowmajor.shape
    cols = nb * 32
    out = np.zeros((((rows + 127) // 128) * ((cols + 127) // 128) * 512,), np.uint8)
    out[mx_tiled_offsets(rows, cols)] = s_rowmajor
    return out


def mx_from_tiled(tiled: np.ndarray, rows: int, cols: int) -> np.ndarray:
    return np.asarray(tiled).reshape(-1)[mx_tiled_offsets(rows, cols)]


# ----------------------------------------------------------------- GEMM
def dequantize(q, kind: int, fmt: int, s) -> np.ndarray:
    q = np.ascontiguousarray(q, dtype=np.uint8)
    R, C = q.shape
    s = np.ascontiguousarray(s, dtype=np.uint8 if kind in (KIND_MX, KIND_MX_FLOOR) else np.float32)
    out = np.empty((R, C), np.float64)
    _load().orc_dequantize(_ptr(q), R, C, fmt, kind, _ptr(s), _ptr(out))
    return out


def round_bf16(values) -> np.ndarray:
    """float64 values -> bfloat16 bit patterns (uint16), one rounding, ties to even."""
    v = np.ascontiguousarray(values, dtype=np.float64)
    f = _load().orc_round_bf16
    return np.array([f(float(x)) for x in v.reshape(-1)], dtype=np.uint16).reshape(v.shape)


def dequantize_bf16(q, kind: int, fmt: int, s) -> np.ndarray:
    """FP8 codes + multipliers -> bfloat16 bit patterns: the exact product rounded once."""
    q = np.ascontiguousarray(q, dtype=np.uint8)
    R, C = q.shape
    s = np.ascontiguousarray(s, dtype=np.uint8 if kind in (KIND_MX, KIND_MX_FLOOR) else np.float32)
    out = np.empty((R, C), np.uint16)
    _load().orc_dequantize_bf16(_ptr(q), R, C, fmt, kind, _ptr(s), _ptr(out))
    return out


def allreduce_sum(g_bf16, fmt: int):
    """FP8 all-reduce of k rank gradients (rows of g [k, n] bf16) with a shared scale.

    Returns (amax, q [k, n] uint8, scale_inv, out [n] float32)."""
    g = _bf16_bits(g_bf16)
    k, n = g.shape
    q = np.empty((k, n), np.uint8)
    out = np.empty(n, np.float32)
    a = np.zeros(1, np.float32)
    si = np.zeros(1, np.float32)
    _load().orc_allreduce_sum(_ptr(g), k, n, fmt, _ptr(a), _ptr(q), _ptr(si), _ptr(out))
    return a[0], q, si[0], out


def scaled_gemm(qa, fa, ka, sa, qb, fb, kb, sb) -> np.ndarray:
    """C[m, n] = sum_k deq(A)[m, k] * deq(B)[n, k] in float64 (A [M,K], B [N,K])."""
    return dequantize(qa, ka, fa, sa) @ dequantize(qb, kb, fb, sb).T


def scaled_gemm_rows(qa, fa, ka, sa, qb, fb, kb, sb, rows) -> np.ndarray:
    """Selected rows of C (all columns), dequantizing only the rows of A needed.

    Blockwise-A scales are indexed by the original row, so the scale rows are
    gathered with the data rows.
    """
    rows = np.asarray(rows, dtype=np.int64)
    qa = np.ascontiguousarray(qa)[rows]
    if ka in (KIND_1x128, KIND_MX, KIND_MX_FLOOR):
        sa = np.ascontiguousarray(sa)[rows]
    elif ka == KIND_128x128:
        raise ValueError("row sampling of a 128x128-scaled A is not supported")
    return dequantize(qa, ka, fa, sa) @ dequantize(qb, kb, fb, sb).T


def gemm_tolerance_check(c_gpu, c_ref, deq_a_rows, deq_b):
    """The stated GEMM bar.

    Returns (rel_fro, worst) where rel_fro = ||C - C_ref||_F / ||C_ref||_F must be
    <= 1e-2 and worst = max over (m, n) of |C - C_ref| / (2e-2 * ||a_m|| ||b_n|| / sqrt(K))
    must be <= 1.  ``deq_a_rows`` are the dequantized rows of A matching the rows
    of ``c_gpu``; ``deq_b`` is the dequantized B [N, K].
    """
    c_gpu = np.asarray(c_gpu, np.float64)
    diff = c_gpu - c_ref
    ref_norm = np.linalg.norm(c_ref)
    rel = float(np.linalg.norm(diff) / ref_norm) if ref_norm > 0 else float(np.linalg.norm(diff))
    K = deq_b.shape[1]
    bound = 2e-2 * np.outer(np.linalg.norm(deq_a_rows, axis=1), np.linalg.norm(deq_b, axis=1)) / np.sqrt(K)
    with np.errstate(divide="ignore", invalid="ignore"):
        ratio = np.where(bound > 0, np.abs(diff) / bound, np.where(diff == 0, 0.0, np.inf))
    return rel, float(ratio.max()) if ratio.size else 0.0
