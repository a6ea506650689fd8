"""Seeded synthetic inputs of the reference workloads.

This module only draws random BF16 tensors; it holds none of the method's
arithmetic.  Both the CUDA path (tests, bench) and the CPU oracle receive the
same bytes: tests generate on the GPU and copy the BF16 bits to the host.

Recipe (every tensor): float32 normal draws from ``torch.randn`` with a
``torch.Generator`` on the target device seeded with
``seed = 1000 * config + 100 * role + step`` (role: X = 0, W = 1, dY = 2),
times sigma, rounded to BF16 (round to nearest even).  Outliers multiply a
seeded subset of columns (configuration 2: 1 % of columns x 100) or elements
(the bandwidth sweep: 0.1 % of elements x 1000).  The same seed gives different
draws on CPU and GPU (different generators); each test states where it draws.
"""
from __future__ import annotations

import torch

ROLE_X, ROLE_W, ROLE_DY = 0, 1, 2


def seed_of(config: int, role: int, step: int = 0) -> int:
    return 1000 * config + 100 * role + step


def _gen(device, seed):
    g = torch.Generator(device=device)
    g.manual_seed(seed)
    return g


def normal_bf16(shape, seed: int, sigma: float = 1.0, device="cuda") -> torch.Tensor:
    g = _gen(device, seed)
    x = torch.randn(shape, generator=g, dtype=torch.float32, device=device)
    if sigma != 1.0:
        x.mul_(sigma)
    return x.to(torch.bfloat16)


def with_outlier_columns(x: torch.Tensor, seed: int, frac: float = 0.01, factor: float = 100.0) -> torch.Tensor:
    """Multiply a seeded ``frac`` of the columns by ``factor`` (in place, returns x)."""
    cols = x.shape[1]
    k = max(1, int(round(frac * cols)))
    g = _gen("cpu", seed + 7)
    idx = torch.randperm(cols, generator=g)[:k].to(x.device)
    x[:, idx] = (x[:, idx].float() * factor).to(torch.bfloat16)
    return x


def with_outlier_elements(x: torch.Tensor, seed: int, frac: float = 0.001, factor: float = 1000.0) -> torch.Tensor:
    """Multiply a seeded ``frac`` of the elements by ``factor`` (in place, returns x)."""
    n = x.numel()
    k = max(1, int(round(frac * n)))
    g = _gen(x.device, seed + 11)
    idx = torch.randint(0, n, (k,), generator=g, device=x.device)
    flat = x.view(-1)
    flat[idx] = (flat[idx].float() * factor).to(torch.bfloat16)
    return x


# --------------------------------------------------------------- configurations
def cfg1_tensor_current(device="cuda"):
    """Per-tensor current scaling, E4M3: A, B 256x256 ~ N(0, 1)."""
    return (normal_bf16((256, 256), seed_of(1, ROLE_X), 1.0, device),
            normal_bf16((256, 256), seed_of(1, ROLE_W), 1.0, device))


def cfg2_blockwise(device="cuda", m=4096, n=4096, k=4096):
    """Blockwise: X [m, k] ~ N(0, 1) with 1 % of columns x100 (1x128 scales),
    W [n, k] ~ N(0, 0.02) (128x128 scales); Y = X W^T."""
    x = with_outlier_columns(normal_bf16((m, k), seed_of(2, ROLE_X), 1.0, device), seed_of(2, ROLE_X))
    w = normal_bf16((n, k), seed_of(2, ROLE_W), 0.02, device)
    return x, w


# LLaMA-7B linear shapes with 8192 tokens: (M, N, K) of QKV, MLP up, MLP down
CFG3_SHAPES = {"qkv": (8192, 12288, 4096), "up": (8192, 11008, 4096), "down": (8192, 4096, 11008)}


def cfg3_mx(name: str, device="cuda"):
    """MXFP8: activations [M, K] ~ N(0, 1), weights [N, K] ~ N(0, 0.02)."""
    m, n, k = CFG3_SHAPES[name]
    idx = list(CFG3_SHAPES).index(name)
    x = normal_bf16((m, k), seed_of(3, ROLE_X, idx), 1.0, device)
    w = normal_bf16((n, k), seed_of(3, ROLE_W, idx), 0.02, device)
    return x, w


# GPT-175B layer linears with 2048 tokens: name -> (in_features, out_features)
CFG4_LINEARS = {"qkv": (12288, 36864), "proj": (12288, 12288), "fc1": (12288, 49152), "fc2": (49152, 12288)}
CFG4_TOKENS = 2048
CFG4_SPIKE_STEP = 8
CFG4_SPIKE = 10.0


def cfg4_step(name: str, step: int, device="cuda"):
    """Delayed scaling step `step` of one GPT-175B linear: X [2048, in] ~ N(0, 1)
    (x10 at the spike step), W [out, in] ~ N(0, 0.02) (fixed over steps),
    dY [2048, out] ~ N(0, 1e-3)."""
    fin, fout = CFG4_LINEARS[name]
    li = list(CFG4_LINEARS).index(name)
    x = normal_bf16((CFG4_TOKENS, fin), seed_of(4, ROLE_X, 10 * step + li) % (2 ** 63), 1.0, device)
    if step == CFG4_SPIKE_STEP:
        x = (x.float() * CFG4_SPIKE).to(torch.bfloat16)
    w = normal_bf16((fout, fin), seed_of(4, ROLE_W, li), 0.02, device)
    dy = normal_bf16((CFG4_TOKENS, fout), seed_of(4, ROLE_DY, 10 * step + li), 1e-3, device)
    return x, w, dy


CFG5_SIZES = (1024, 2048, 4096, 8192, 16384, 32768)


def cfg5_sweep(size: int, device="cuda"):
    """Bandwidth sweep: size x size ~ N(0, 1) with 0.1 % of elements x1000."""
    return with_outlier_elements(normal_bf16((size, size), seed_of(5, ROLE_X, CFG5_SIZES.index(size) if size in
                                                                   CFG5_SIZES else size), 1.0, device),
                                 seed_of(5, ROLE_X))
