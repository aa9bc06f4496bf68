"""Seeded synthetic inputs shared by the tests and the benchmark.

This module only draws random numbers and rounds them to the storage type; it
holds none of the GEMM or SwiGLU arithmetic.  Both the oracle side and the
CUDA side of a comparison receive the very tensors made here.

All draws use a CPU ``torch.Generator`` so the bits are the same on every
host.  FP32 draws are rounded to half formats with ``Tensor.to`` (round to
nearest even).  Within one workload, tensors are drawn in the order A, B, C
(or A, W1, W2) from one generator seeded with ``seed``.

Workloads (shapes and distributions of the GEMM/SwiGLU benchmark set):

* ``gemm_f16_small``  — A, B ~ U(-1, 1) as fp16, C ~ U(-1, 1) fp32, 256^3.
* ``gemm_bf16``       — A, B ~ N(0, 1) as bf16 (square 4096 / 8192).
* ``swiglu``          — A ~ N(0, 1) bf16 [M x K]; W1, W2 ~ N(0, 0.02) bf16
                        [K x N] (small model: K=896, N=4864; 8B class:
                        K=4096, N=14336).
* ``skinny``          — A [M x 16384], B [16384 x 4096], C [M x 4096], all
                        ~ N(0, 1) bf16.
"""
from __future__ import annotations

import torch


def generator(seed: int) -> torch.Generator:
    g = torch.Generator(device="cpu")
    g.manual_seed(int(seed))
    return g


def uniform(shape, g, lo=-1.0, hi=1.0, dtype=torch.float32):
    x = torch.rand(*shape, generator=g, dtype=torch.float32) * (hi - lo) + lo
    return x.to(dtype)


def normal(shape, g, std=1.0, dtype=torch.bfloat16):
    x = torch.randn(*shape, generator=g, dtype=torch.float32) * std
    return x.to(dtype)


def small_ints(shape, g, lo=-8, hi=8, dtype=torch.bfloat16):
    """Integers in [lo, hi]: exact in fp16/bf16 and in every partial sum of a
    short dot product, for exact-equality checks."""
    x = torch.randint(lo, hi + 1, tuple(shape), generator=g, dtype=torch.int64)
    return x.to(dtype)


def stored_shape(trans: int, rows: int, cols: int):
    """Shape in which op(X) of shape rows x cols is stored row-major:
    X itself (trans = 0) or X^T (trans = 1)."""
    return (cols, rows) if trans else (rows, cols)


def gemm_f16_small(seed: int = 0, M: int = 256, N: int = 256, K: int = 256):
    g = generator(seed)
    A = uniform((M, K), g, dtype=torch.float16)
    B = uniform((K, N), g, dtype=torch.float16)
    C = uniform((M, N), g, dtype=torch.float32)
    return A, B, C


def gemm_bf16(M: int, N: int, K: int, transA: int = 0, transB: int = 0,
              seed: int = 1, c: bool = False, dist: str = "normal",
              dtype=torch.bfloat16):
    """A, B (and C when ``c``) in their STORED shapes for the given ops."""
    g = generator(seed)
    draw = normal if dist == "normal" else small_ints
    A = draw(stored_shape(transA, M, K), g, dtype=dtype)
    B = draw(stored_shape(transB, K, N), g, dtype=dtype)
    C = draw((M, N), g, dtype=dtype) if c else None
    return A, B, C


def swiglu(M: int, K: int, N: int, seed: int = 3, w_std: float = 0.02):
    g = generator(seed)
    A = normal((M, K), g, std=1.0)
    W1 = normal((K, N), g, std=w_std)
    W2 = normal((K, N), g, std=w_std)
    return A, W1, W2


def skinny(M: int, N: int = 4096, K: int = 16384, seed: int = 4):
    g = generator(seed)
    A = normal((M, K), g)
    B = normal((K, N), g)
    C = normal((M, N), g)
    return A, B, C


def to_e4m3(x: torch.Tensor):
    """Per-tensor scaled e4m3 copy of x: returns (q, scale) with q = x / scale
    rounded to e4m3 (round to nearest even) and scale = max|x| / 448, so the
    largest magnitude maps to e4m3's largest finite value."""
    amax = float(x.abs().max())
    scale = amax / 448.0 if amax > 0 else 1.0
    return (x / scale).to(torch.float8_e4m3fn), scale


def swiglu_e4m3(M: int, K: int, N: int, seed: int = 3, w_std: float = 0.02):
    """e4m3 A (N(0,1) fits without a scale) and e4m3 W1, W2 sharing one
    per-tensor scale (the interleaved weight is one tensor): returns
    (A, W1, W2, scale_w)."""
    g = generator(seed)
    A = torch.randn(M, K, generator=g).to(torch.float8_e4m3fn)
    W1 = torch.randn(K, N, generator=g) * w_std
    W2 = torch.randn(K, N, generator=g) * w_std
    amax = max(float(W1.abs().max()), float(W2.abs().max()))
    scale = amax / 448.0 if amax > 0 else 1.0
    return A, (W1 / scale).to(torch.float8_e4m3fn), (W2 / scale).to(torch.float8_e4m3fn), scale
