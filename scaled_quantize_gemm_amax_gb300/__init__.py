"""FP8 scaled quantization and scaled FP8 GEMM for NVIDIA GB300 (sm_103a).

Python binding of libfp8q (C ABI in ``include/fp8q.h``).  Every step of the
path runs in the library's CUDA kernels; this module only marshals arguments
(torch tensors -> device pointers, the current torch stream) and allocates
output tensors with torch.  There is no fallback: every call raises when
``libfp8q.so`` has not been built (``scaled_quantize_gemm_amax_gb300/build.py``).

Entry points with the C names take tensors (or None for NULL) and raise
``FP8Error`` on a non-OK status: ``fp8_amax``, ``fp8_amax_f32``, ``fp8_compute_scale``,
``amax_history_update``, ``fp8_quantize``, ``fp8_cast_transpose``, ``fp8_cast_transpose_f32``,
``fp8_cast_transpose_multi``,
``fp8_dequantize``, ``fp8_allreduce_sum``, ``fp8_scaled_gemm``, ``fp8_scaled_gemm_amax``,
``fp8_get_device_status``, ``fp8_debug_wait_timeout``, ``fp8_debug_gemm_plan``,
``fp8_debug_index_check``.  ``cast_transpose`` /
``dequantize`` / ``scaled_gemm`` / ``scaled_gemm_amax`` are allocation helpers
over them; ``linear`` holds the FP8 linear layer and the autocast scope built
on these calls.
"""
from __future__ import annotations

import ctypes
import enum
import os

import torch

__all__ = [
    "Status", "Format", "Recipe", "OutDtype", "FP8Error", "lib_path", "load_library",
    "fp8_amax", "fp8_amax_f32", "fp8_compute_scale", "amax_history_update", "fp8_quantize", "fp8_cast_transpose",
    "fp8_cast_transpose_f32",
    "fp8_cast_transpose_multi", "CastJob",
    "fp8_dequantize", "fp8_allreduce_sum", "fp8_allreduce_sum_noalloc", "fp8_scaled_gemm", "fp8_scaled_gemm_amax", "fp8_get_device_status",
    "fp8_debug_wait_timeout", "fp8_debug_gemm_plan", "fp8_debug_index_check", "fp8_status_string",
    "scale_shape", "cast_transpose", "cast_transpose_multi", "dequantize", "allreduce_sum", "scaled_gemm", "scaled_gemm_amax",
    "DelayedScaling",
]


class Status(enum.IntEnum):
    OK = 0
    ERR_INVALID_ARG = 1
    ERR_SHAPE = 2
    ERR_ALIGNMENT = 3
    ERR_UNSUPPORTED = 4
    ERR_CUDA = 5
    ERR_TIMEOUT = 6
    ERR_DEVICE_STATE = 7
    ERR_INDEX = 8


class Format(enum.IntEnum):
    E4M3 = 0
    E5M2 = 1


class Recipe(enum.IntEnum):
    TENSOR = 0
    BLOCK_1x128 = 1
    BLOCK_128x128 = 2
    MX_1x32 = 3
    MX_1x32_TILED = 4
    MX_1x32_FLOOR = 5          # floor-rule exponent (the alternate); layouts as MX_1x32 / MX_1x32_TILED
    MX_1x32_FLOOR_TILED = 6


class OutDtype(enum.IntEnum):
    BF16 = 0
    FP32 = 1


class FP8Error(RuntimeError):
    def __init__(self, fn: str, status: int):
        self.status = Status(status)
        super().__init__(f"{fn}: {self.status.name}")


_PKG = os.path.dirname(os.path.abspath(__file__))


def lib_path() -> str:
    return os.path.join(_PKG, "libfp8q.so")


_lib = None

_P = ctypes.c_void_p
_I64 = ctypes.c_int64
_I32 = ctypes.c_int32
_E = ctypes.c_int
class CastJob(ctypes.Structure):
    """C layout of fp8_cast_job."""
    _fields_ = [("x", ctypes.c_void_p), ("rows", ctypes.c_int64), ("cols", ctypes.c_int64),
                ("recipe", ctypes.c_int), ("fmt", ctypes.c_int), ("scale", ctypes.c_void_p),
                ("amax_out", ctypes.c_void_p), ("q_row", ctypes.c_void_p), ("s_row", ctypes.c_void_p),
                ("q_col", ctypes.c_void_p), ("s_col", ctypes.c_void_p)]


_SIGNATURES = {
    "fp8_amax": [_P, _I64, _I64, _P, _P],
    "fp8_amax_f32": [_P, _I64, _I64, _P, _P],
    "fp8_cast_transpose_f32": [_P, _I64, _I64, _E, _E, _P, _P, _P, _P, _P, _P, _P],
    "fp8_compute_scale": [_P, _E, _P, _P, _P],
    "amax_history_update": [_P, _I32, _P, _P, _E, _P, _P, _P],
    "fp8_cast_transpose": [_P, _I64, _I64, _E, _E, _P, _P, _P, _P, _P, _P, _P],
    "fp8_quantize": [_P, _I64, _I64, _E, _E, _P, _P, _P, _P, _P],
    "fp8_cast_transpose_multi": [_P, _I32, _P],
    "fp8_dequantize": [_P, _I64, _I64, _E, _E, _P, _P, _P],
    "fp8_allreduce_sum": [_P, _I32, _I64, _E, _P, _P, _P, _P, _P],
    "fp8_allreduce_sum_noalloc": [_P, _I32, _I64, _E, _P, _P, _P, _P],
    "fp8_scaled_gemm": [_P, _E, _E, _P, _P, _E, _E, _P, _I64, _I64, _I64, _P, _E, _P],
    "fp8_scaled_gemm_amax": [_P, _E, _E, _P, _P, _E, _E, _P, _I64, _I64, _I64, _P, _E, _P, _P, _E, _P, _P, _P],
    "fp8_get_device_status": [_P],
    "fp8_debug_wait_timeout": [_P],
    "fp8_debug_gemm_plan": [_E, _E, _E, _I64, _I64, _I64, _I32, _I32, _I32, _P],
    "fp8_debug_index_check": [_I64, _I64, _P],
    "fp8_status_string": [_E],
}


def load_library(path: str | None = None):
    """Load libfp8q.so (raises OSError if it has not been built)."""
    global _lib
    if _lib is not None and path is None:
        return _lib
    p = path or lib_path()
    if not os.path.exists(p):
        raise OSError(f"libfp8q.so not built at {p}; run scaled_quantize_gemm_amax_gb300/build.py")
    lib = ctypes.CDLL(p)
    for name, args in _SIGNATURES.items():
        fn = getattr(lib, name)
        fn.argtypes = args
        fn.restype = ctypes.c_char_p if name == "fp8_status_string" else ctypes.c_int
    if path is None:
        _lib = lib
    return lib


def _ptr(t):
    if t is None:
        return None
    if isinstance(t, int):
        return t
    return t.data_ptr()


def _stream(stream):
    if stream is None:
        return torch.cuda.current_stream().cuda_stream
    if isinstance(stream, int):
        return stream
    return stream.cuda_stream


def _check(fn: str, status: int):
    if status != 0:
        raise FP8Error(fn, status)


def fp8_status_string(status: int) -> str:
    return load_library().fp8_status_string(int(status)).decode()


# ------------------------------------------------------------------ C-ABI calls
def fp8_amax(x, amax, stream=None):
    """amax[0] = max |x| (x: [rows, cols] bf16 tensor, amax: 1-float device tensor)."""
    rows, cols = (x.shape[0], x.numel() // max(x.shape[0], 1)) if x.dim() >= 1 else (1, 1)
    _check("fp8_amax", load_library().fp8_amax(_ptr(x), rows, cols, _ptr(amax), _stream(stream)))


def fp8_amax_f32(x, amax, stream=None):
    """amax[0] = max |x| of a float32 tensor."""
    rows, cols = (x.shape[0], x.numel() // max(x.shape[0], 1)) if x.dim() >= 1 else (1, 1)
    _check("fp8_amax_f32", load_library().fp8_amax_f32(_ptr(x), rows, cols, _ptr(amax), _stream(stream)))


def fp8_compute_scale(amax, fmt, scale, scale_inv, stream=None):
    _check("fp8_compute_scale",
           load_library().fp8_compute_scale(_ptr(amax), int(fmt), _ptr(scale), _ptr(scale_inv), _stream(stream)))


def amax_history_update(hist, pos, amax, fmt, scale, scale_inv, stream=None):
    _check("amax_history_update",
           load_library().amax_history_update(_ptr(hist), hist.numel(), _ptr(pos), _ptr(amax), int(fmt),
                                              _ptr(scale), _ptr(scale_inv), _stream(stream)))


def fp8_cast_transpose(x, recipe, fmt, scale, amax_out, q_row, s_row, q_col, s_col, stream=None):
    rows, cols = x.shape
    _check("fp8_cast_transpose",
           load_library().fp8_cast_transpose(_ptr(x), rows, cols, int(recipe), int(fmt), _ptr(scale),
                                             _ptr(amax_out), _ptr(q_row), _ptr(s_row), _ptr(q_col), _ptr(s_col),
                                             _stream(stream)))


def fp8_cast_transpose_f32(x, recipe, fmt, scale, amax_out, q_row, s_row, q_col, s_col, stream=None):
    rows, cols = x.shape
    _check("fp8_cast_transpose_f32",
           load_library().fp8_cast_transpose_f32(_ptr(x), rows, cols, int(recipe), int(fmt), _ptr(scale),
                                                 _ptr(amax_out), _ptr(q_row), _ptr(s_row), _ptr(q_col), _ptr(s_col),
                                                 _stream(stream)))


def fp8_cast_transpose_multi(jobs, stream=None):
    """jobs: sequence of (x, recipe, fmt, scale, amax_out, q_row, s_row, q_col, s_col), as fp8_cast_transpose."""
    arr = (CastJob * max(len(jobs), 1))()
    for i, (x, recipe, fmt, scale, amax_out, q_row, s_row, q_col, s_col) in enumerate(jobs):
        rows, cols = x.shape
        arr[i] = CastJob(_ptr(x), rows, cols, int(recipe), int(fmt), _ptr(scale), _ptr(amax_out), _ptr(q_row),
                         _ptr(s_row), _ptr(q_col), _ptr(s_col))
    _check("fp8_cast_transpose_multi",
           load_library().fp8_cast_transpose_multi(ctypes.cast(arr, ctypes.c_void_p), len(jobs), _stream(stream)))


def fp8_quantize(x, recipe, fmt, scale, amax_out, q, s, stream=None):
    rows, cols = x.shape
    _check("fp8_quantize",
           load_library().fp8_quantize(_ptr(x), rows, cols, int(recipe), int(fmt), _ptr(scale), _ptr(amax_out),
                                       _ptr(q), _ptr(s), _stream(stream)))


def fp8_dequantize(q, recipe, fmt, s, y, stream=None):
    rows, cols = q.shape
    _check("fp8_dequantize",
           load_library().fp8_dequantize(_ptr(q), rows, cols, int(recipe), int(fmt), _ptr(s), _ptr(y),
                                         _stream(stream)))


def fp8_allreduce_sum(g, fmt, amax, q, scale_inv, out, stream=None):
    k, n = g.shape
    _check("fp8_allreduce_sum",
           load_library().fp8_allreduce_sum(_ptr(g), k, n, int(fmt), _ptr(amax), _ptr(q), _ptr(scale_inv), _ptr(out),
                                            _stream(stream)))


def fp8_allreduce_sum_noalloc(g, fmt, q, scale_inv, out, stream=None):
    k, n = g.shape
    _check("fp8_allreduce_sum_noalloc",
           load_library().fp8_allreduce_sum_noalloc(_ptr(g), k, n, int(fmt), _ptr(q), _ptr(scale_inv), _ptr(out),
                                                    _stream(stream)))


def allreduce_sum(g, fmt=Format.E5M2, stream=None):
    """Allocate outputs and run fp8_allreduce_sum on g [k, n] (rank r's gradient in row r).

    Returns (out [n] fp32, q [k, n] u8, scale_inv, amax)."""
    k, n = g.shape
    dev = g.device
    amax = torch.empty(1, dtype=torch.float32, device=dev)
    q = torch.empty((k, n), dtype=torch.uint8, device=dev)
    scale_inv = torch.empty(1, dtype=torch.float32, device=dev)
    out = torch.empty(n, dtype=torch.float32, device=dev)
    fp8_allreduce_sum(g, fmt, amax, q, scale_inv, out, stream)
    return out, q, scale_inv, amax


def dequantize(q, recipe, fmt, s, stream=None):
    """Allocate y [rows, cols] bf16 and run fp8_dequantize."""
    y = torch.empty(q.shape, dtype=torch.bfloat16, device=q.device)
    fp8_dequantize(q, recipe, fmt, s, y, stream)
    return y


def fp8_scaled_gemm(a, fa, ra, sa, b, fb, rb, sb, c, out=OutDtype.BF16, stream=None):
    M, K = a.shape
    N = b.shape[0]
    _check("fp8_scaled_gemm",
           load_library().fp8_scaled_gemm(_ptr(a), int(fa), int(ra), _ptr(sa), _ptr(b), int(fb), int(rb), _ptr(sb),
                                          M, N, K, _ptr(c), int(out), _stream(stream)))


def fp8_scaled_gemm_amax(a, fa, ra, sa, b, fb, rb, sb, c, out, c_amax, c_scale, fc, c_q, c_scale_inv, stream=None):
    M, K = a.shape
    N = b.shape[0]
    _check("fp8_scaled_gemm_amax",
           load_library().fp8_scaled_gemm_amax(_ptr(a), int(fa), int(ra), _ptr(sa), _ptr(b), int(fb), int(rb),
                                               _ptr(sb), M, N, K, _ptr(c), int(out), _ptr(c_amax), _ptr(c_scale),
                                               int(fc), _ptr(c_q), _ptr(c_scale_inv), _stream(stream)))


def fp8_get_device_status(stream=None) -> Status:
    return Status(load_library().fp8_get_device_status(_stream(stream)))


def fp8_debug_wait_timeout(stream=None):
    _check("fp8_debug_wait_timeout", load_library().fp8_debug_wait_timeout(_stream(stream)))


def fp8_debug_index_check(index: int, extent: int, stream=None):
    _check("fp8_debug_index_check", load_library().fp8_debug_index_check(index, extent, _stream(stream)))


GEMM_VARIANTS = {0: "per-tensor", 1: "blockwise, one CTA, 128-deep stages", 3: "MXFP8",
                 4: "blockwise per-row B, one CTA", 5: "blockwise, 256-deep stages",
                 6: "blockwise per-row B, CTA pairs", 7: "blockwise, 256 x 160 pair tiles"}


def fp8_debug_gemm_plan(ra, rb, out, m: int, n: int, k: int, fused: bool = False, num_sms: int = 152,
                        resident_pairs: int = 0) -> dict:
    """The division fp8_scaled_gemm would choose (host logic only, no device call)."""
    plan = (ctypes.c_int64 * 8)()
    _check("fp8_debug_gemm_plan", load_library().fp8_debug_gemm_plan(int(ra), int(rb), int(out), m, n, k, int(fused),
                                                                      num_sms, resident_pairs, plan))
    keys = ("pair", "variant", "block_n", "tiles", "streamk", "split", "tail0", "launched")
    return dict(zip(keys, (int(v) for v in plan)))


# ------------------------------------------------------------------ allocation helpers
def scale_shape(recipe, rows: int, cols: int):
    """Shape and dtype of the multiplier array of a [rows, cols] row-wise copy."""
    recipe = Recipe(recipe)
    if recipe == Recipe.TENSOR:
        return (1,), torch.float32
    if recipe == Recipe.BLOCK_1x128:
        return (rows, cols // 128), torch.float32
    if recipe == Recipe.BLOCK_128x128:
        return (rows // 128, cols // 128), torch.float32
    if recipe in (Recipe.MX_1x32, Recipe.MX_1x32_FLOOR):
        return (rows, cols // 32), torch.uint8
    return ((rows + 127) // 128, (cols + 127) // 128, 512), torch.uint8


def cast_transpose(x, recipe, fmt, scale=None, amax_out=None, row=True, col=True, stream=None):
    """Allocate outputs with torch and run fp8_cast_transpose (bf16 x) or
    fp8_cast_transpose_f32 (float32 x).

    Returns (q_row, s_row, q_col, s_col); the parts not requested are None.
    """
    rows, cols = x.shape
    dev = x.device
    q_row = s_row = q_col = s_col = None
    if row:
        q_row = torch.empty((rows, cols), dtype=torch.uint8, device=dev)
        shp, dt = scale_shape(recipe, rows, cols)
        s_row = torch.empty(shp, dtype=dt, device=dev)
    if col:
        q_col = torch.empty((cols, rows), dtype=torch.uint8, device=dev)
        shp, dt = scale_shape(recipe, cols, rows)
        s_col = torch.empty(shp, dtype=dt, device=dev)
    if x.dtype == torch.float32:
        fp8_cast_transpose_f32(x, recipe, fmt, scale, amax_out, q_row, s_row, q_col, s_col, stream)
    elif x.dtype == torch.bfloat16:
        fp8_cast_transpose(x, recipe, fmt, scale, amax_out, q_row, s_row, q_col, s_col, stream)
    else:
        raise TypeError(f"cast_transpose takes bfloat16 or float32 input, not {x.dtype}")
    return q_row, s_row, q_col, s_col


def cast_transpose_multi(specs, stream=None):
    """specs: sequence of (x, recipe, fmt, scale, amax_out).  Allocates every job's outputs
    with torch and runs them in one fp8_cast_transpose_multi launch; returns a list of
    (q_row, s_row, q_col, s_col) per job."""
    outs, jobs = [], []
    for x, recipe, fmt, scale, amax_out in specs:
        rows, cols = x.shape
        dev = x.device
        q_row = torch.empty((rows, cols), dtype=torch.uint8, device=dev)
        shp, dt = scale_shape(recipe, rows, cols)
        s_row = torch.empty(shp, dtype=dt, device=dev)
        q_col = torch.empty((cols, rows), dtype=torch.uint8, device=dev)
        shp, dt = scale_shape(recipe, cols, rows)
        s_col = torch.empty(shp, dtype=dt, device=dev)
        outs.append((q_row, s_row, q_col, s_col))
        jobs.append((x, recipe, fmt, scale, amax_out, q_row, s_row, q_col, s_col))
    fp8_cast_transpose_multi(jobs, stream)
    return outs


def scaled_gemm(a, fa, ra, sa, b, fb, rb, sb, out=OutDtype.BF16, stream=None):
    """Allocate C [M, N] (bf16 or fp32) and run fp8_scaled_gemm."""
    M, N = a.shape[0], b.shape[0]
    c = torch.empty((M, N), dtype=torch.float32 if out == OutDtype.FP32 else torch.bfloat16, device=a.device)
    fp8_scaled_gemm(a, fa, ra, sa, b, fb, rb, sb, c, out, stream)
    return c


def scaled_gemm_amax(a, fa, ra, sa, b, fb, rb, sb, c_scale, fc=Format.E4M3, out=OutDtype.BF16, keep_c=True,
                     stream=None):
    """Allocate outputs and run fp8_scaled_gemm_amax.

    Returns (c or None, c_amax, c_q, c_scale_inv): C's FP8 copy with the given
    per-tensor scale (e.g. a DelayedScaling state's) and the amax of C."""
    M, N = a.shape[0], b.shape[0]
    dev = a.device
    c = None
    if keep_c:
        c = torch.empty((M, N), dtype=torch.float32 if out == OutDtype.FP32 else torch.bfloat16, device=dev)
    c_amax = torch.empty(1, dtype=torch.float32, device=dev)
    c_q = torch.empty((M, N), dtype=torch.uint8, device=dev)
    c_scale_inv = torch.empty(1, dtype=torch.float32, device=dev)
    fp8_scaled_gemm_amax(a, fa, ra, sa, b, fb, rb, sb, c, out, c_amax, c_scale, fc, c_q, c_scale_inv, stream)
    return c, c_amax, c_q, c_scale_inv


class DelayedScaling:
    """Device-resident delayed-scaling state of one tensor role (history ring,
    write position, scale, scale_inv), driven by ``amax_history_update``."""

    def __init__(self, length: int = 16, fmt=Format.E4M3, device="cuda"):
        self.fmt = Format(fmt)
        self.hist = torch.zeros(length, dtype=torch.float32, device=device)
        self.pos = torch.zeros(1, dtype=torch.int32, device=device)
        self.scale = torch.ones(1, dtype=torch.float32, device=device)
        self.scale_inv = torch.ones(1, dtype=torch.float32, device=device)
        self.amax = torch.zeros(1, dtype=torch.float32, device=device)

    def update(self, stream=None):
        """Fold self.amax (written by the cast's amax_out) into the history."""
        amax_history_update(self.hist, self.pos, self.amax, self.fmt, self.scale, self.scale_inv, stream)

    def state_dict(self):
        return {"hist": self.hist.clone(), "pos": self.pos.clone(), "scale": self.scale.clone(),
                "scale_inv": self.scale_inv.clone()}

    def load_state_dict(self, sd):
        for k in ("hist", "pos", "scale", "scale_inv"):
            getattr(self, k).copy_(sd[k])
