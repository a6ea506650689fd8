"""FP8 linear layer and autocast scope over the C ABI.

The FP8 quantized-training guide ("code changes") puts the gain in the three
GEMMs of a layer: their inputs are quantized, their outputs stay BF16 (the
weight gradient FP32), and a recipe object chosen in an ``fp8_autocast`` scope
says how (per-tensor ``Float8CurrentScaling``, blockwise ``Float8BlockScaling``).
The search-result page's dataflow paragraph fixes the precisions: BF16 input,
weights quantized to FP8 from a higher-precision copy, BF16 output, FP32 wgrad.

For Y = X W^T (X [M, K], W [N, K]) the three GEMMs, each C = A B^T with both
operands K-major, read these FP8 copies:
  fprop  Y  [M, N] = X_row  [M, K] . W_row  [N, K]^T          (BF16 out)
  dgrad  dX [M, K] = dY_row [M, N] . W_col  [K, N]^T          (BF16 out)
  wgrad  dW [N, K] = dY_col [N, M] . X_col  [K, M]^T          (FP32 out)
so every operand is quantized once with fp8_cast_transpose (row- and
column-wise copies in one pass).  Recipes:
  Float8CurrentScaling  per-tensor; scale from this step's amax (fp8_amax,
                        fp8_compute_scale, then the cast)
  Float8DelayedScaling  per-tensor; scale from the history of past amaxes
                        (the cast records this step's amax; amax_history_update
                        folds it in after the cast) -- Colossal-AI FP8 article,
                        "delayed scaling"
  Float8BlockScaling    X, dY 1x128 and W 128x128 FP32 scales (guide,
                        "block-level scaling")
  MXFP8BlockScaling     1x32 E8M0 scales everywhere (guide, "MXFP8 scaling")
Every computation runs in the library's kernels -- torch only allocates: the
FP32 master weight is quantized directly (fp8_cast_transpose_f32, with
fp8_amax_f32 for current scaling), bf16 or float32 activations and gradients
go to the cast of their own dtype, and each GEMM writes its output in the
dtype autograd expects (Y and dX in the input's dtype, dW in FP32).  M, N and
K must be multiples of 128 (the GEMM's tile), which the library checks.
"""
from __future__ import annotations

import contextlib
import dataclasses
import threading

import torch

from . import (DelayedScaling, Format, OutDtype, Recipe, amax_history_update, cast_transpose, fp8_amax,
               fp8_amax_f32, fp8_compute_scale, fp8_scaled_gemm)

__all__ = ["Float8CurrentScaling", "Float8DelayedScaling", "Float8BlockScaling", "MXFP8BlockScaling", "fp8_autocast",
           "get_fp8_recipe", "FP8Linear", "fp8_linear"]


@dataclasses.dataclass(frozen=True)
class Float8CurrentScaling:
    fwd_format: Format = Format.E4M3      # X, W
    bwd_format: Format = Format.E5M2      # dY


@dataclasses.dataclass(frozen=True)
class Float8DelayedScaling:
    history_len: int = 16
    fwd_format: Format = Format.E4M3
    bwd_format: Format = Format.E5M2


@dataclasses.dataclass(frozen=True)
class Float8BlockScaling:
    fwd_format: Format = Format.E4M3
    bwd_format: Format = Format.E4M3      # fine-grained scales leave E4M3's range enough for gradients


@dataclasses.dataclass(frozen=True)
class MXFP8BlockScaling:
    fwd_format: Format = Format.E4M3
    bwd_format: Format = Format.E4M3


_STATE = threading.local()


def get_fp8_recipe():
    """The recipe of the innermost active fp8_autocast scope (per-tensor current scaling outside one)."""
    stack = getattr(_STATE, "stack", None)
    return stack[-1] if stack else Float8CurrentScaling()


@contextlib.contextmanager
def fp8_autocast(enabled: bool = True, fp8_recipe=None):
    """Run FP8Linear layers inside the scope with ``fp8_recipe`` (default: current scaling)."""
    if not enabled:
        yield
        return
    stack = getattr(_STATE, "stack", None)
    if stack is None:
        stack = _STATE.stack = []
    stack.append(fp8_recipe if fp8_recipe is not None else Float8CurrentScaling())
    try:
        yield
    finally:
        stack.pop()


# ------------------------------------------------------------------ quantization of one operand
def _quantize(x, recipe_kind, fmt, delayed: DelayedScaling | None):
    """Row- and column-wise FP8 copies of a [R, C] bf16 or float32 matrix: (q_row, s_row, q_col, s_col)."""
    if x.dtype not in (torch.bfloat16, torch.float32):
        raise TypeError(f"FP8 linear operands are bfloat16 or float32, not {x.dtype}")
    if recipe_kind == Recipe.TENSOR:
        if delayed is not None:
            out = cast_transpose(x, Recipe.TENSOR, fmt, delayed.scale, delayed.amax)
            amax_history_update(delayed.hist, delayed.pos, delayed.amax, fmt, delayed.scale, delayed.scale_inv)
            return out
        amax = torch.empty(1, dtype=torch.float32, device=x.device)
        scale = torch.empty(1, dtype=torch.float32, device=x.device)
        scale_inv = torch.empty(1, dtype=torch.float32, device=x.device)
        (fp8_amax_f32 if x.dtype == torch.float32 else fp8_amax)(x, amax)
        fp8_compute_scale(amax, fmt, scale, scale_inv)
        return cast_transpose(x, Recipe.TENSOR, fmt, scale)
    return cast_transpose(x, recipe_kind, fmt)


def _kinds(recipe):
    """(X / dY recipe, W recipe) of a recipe object."""
    if isinstance(recipe, (Float8CurrentScaling, Float8DelayedScaling)):
        return Recipe.TENSOR, Recipe.TENSOR
    if isinstance(recipe, Float8BlockScaling):
        return Recipe.BLOCK_1x128, Recipe.BLOCK_128x128
    if isinstance(recipe, MXFP8BlockScaling):
        return Recipe.MX_1x32_TILED, Recipe.MX_1x32_TILED
    raise TypeError(f"unknown FP8 recipe {recipe!r}")


class _FP8LinearFn(torch.autograd.Function):
    @staticmethod
    def forward(ctx, x2d, weight, recipe, states):
        kx, kw = _kinds(recipe)
        fx, fdy = recipe.fwd_format, recipe.bwd_format
        # the master weight (FP32) is quantized as it is; its gradient goes to it in FP32,
        # as the wgrad GEMM produces it
        qx, sx, qxt, sxt = _quantize(x2d, kx, fx, states.get("x"))
        qw, sw, qwt, swt = _quantize(weight.detach().contiguous(), kw, fx, states.get("w"))
        out = OutDtype.FP32 if x2d.dtype == torch.float32 else OutDtype.BF16
        y = torch.empty((x2d.shape[0], weight.shape[0]), dtype=x2d.dtype, device=x2d.device)
        fp8_scaled_gemm(qx, fx, kx, sx, qw, fx, kw, sw, y, out)
        ctx.save_for_backward(qxt, sxt, qwt, swt)
        ctx.meta = (kx, kw, fx, fdy, states.get("dy"), x2d.dtype, weight.dtype)
        return y

    @staticmethod
    def backward(ctx, dy):
        qxt, sxt, qwt, swt = ctx.saved_tensors
        kx, kw, fx, fdy, st_dy, x_dtype, w_dtype = ctx.meta
        qdy, sdy, qdyt, sdyt = _quantize(dy.contiguous(), kx, fdy, st_dy)
        M, N = dy.shape
        K = qxt.shape[0]
        dx = torch.empty((M, K), dtype=x_dtype, device=dy.device)
        # dgrad: dY [M, N] . (W^T [K, N])^T; the W copy along N is its column-wise copy
        fp8_scaled_gemm(qdy, fdy, kx, sdy, qwt, fx, kw, swt, dx,
                        OutDtype.FP32 if x_dtype == torch.float32 else OutDtype.BF16)
        dw = torch.empty((N, K), dtype=w_dtype, device=dy.device)
        # wgrad: dY^T [N, M] . (X^T [K, M])^T, both column-wise copies (blockwise: 1x128 with 1x128);
        # FP32 for the FP32 master weight
        fp8_scaled_gemm(qdyt, fdy, kx, sdyt, qxt, fx, kx, sxt, dw,
                        OutDtype.FP32 if w_dtype == torch.float32 else OutDtype.BF16)
        return dx, dw, None, None


def fp8_linear(x, weight, recipe=None, states=None):
    """Y = X W^T through the three FP8 GEMMs (x [..., K] bf16 or float32, weight [N, K] float32)."""
    recipe = recipe if recipe is not None else get_fp8_recipe()
    lead = x.shape[:-1]
    x2d = x.reshape(-1, x.shape[-1]).contiguous()
    y = _FP8LinearFn.apply(x2d, weight, recipe, states or {})
    return y.reshape(*lead, weight.shape[0])


class FP8Linear(torch.nn.Module):
    """Linear layer (no bias) whose GEMMs run in FP8 under the active recipe.

    The FP32 master weight is quantized directly every step (the guide's "weight
    dual copy": FP8 weights come from a higher-precision copy).  Under a
    Float8DelayedScaling recipe the layer keeps one delayed-scaling state per
    tensor role (X and W in E4M3, dY in the backward format)."""

    def __init__(self, in_features: int, out_features: int, device=None, dtype=torch.float32):
        super().__init__()
        self.in_features, self.out_features = in_features, out_features
        self.weight = torch.nn.Parameter(torch.empty((out_features, in_features), device=device, dtype=dtype))
        torch.nn.init.normal_(self.weight, std=0.02)
        self._delayed = None

    def _states(self, recipe):
        if not isinstance(recipe, Float8DelayedScaling):
            return {}
        if self._delayed is None or self._delayed[0] != recipe:
            dev = self.weight.device
            self._delayed = (recipe, {
                "x": DelayedScaling(recipe.history_len, recipe.fwd_format, dev),
                "w": DelayedScaling(recipe.history_len, recipe.fwd_format, dev),
                "dy": DelayedScaling(recipe.history_len, recipe.bwd_format, dev),
            })
        return self._delayed[1]

    def forward(self, x):
        recipe = get_fp8_recipe()
        return fp8_linear(x, self.weight, recipe, self._states(recipe))
