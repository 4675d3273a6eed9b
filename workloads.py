"""Seeded synthetic inputs shared by the tests, the smoke check and the bench.

This module holds no arithmetic of the method: it only draws random bf16 /
int8 tensors on the CPU with torch's default generator algorithm (so the CUDA
library and the CPU oracle see identical bits) and names the shapes.

Shapes and distributions follow the pages:

* "test_int4_quantized_gemm.py": MODEL_SHAPES, SMALL_SHAPES, W4A8 buckets
  1..4, weights ``torch.randn(n, k, dtype=torch.bfloat16)`` seeded per shape
  (``n ^ k`` for model shapes, ``n + k`` for small shapes), the outlier
  activations of Int4QuantizedGemmPrecisionTest (channels 0, K/3, 2K/3, K-1
  scaled by 50, 35, 25, 20).
* "gpt-fast issue #114": the 8192 x 8192 int8 weight-only GEMV with per-row
  bf16 scales and a bf16 activation row.

The activation seed rule ``n ^ k ^ (1000 + m)`` and the draw order (weights
first, then scales, then activations) are this library's choice.
"""
from __future__ import annotations

import torch

GROUP = 32

# "test_int4_quantized_gemm.py": MODEL_SHAPES / SMALL_SHAPES, as (N, K).
MODEL_SHAPES = ((8448, 6656), (6656, 4096), (39936, 6656), (6656, 19968), (256, 6656))
SMALL_SHAPES = ((768, 256), (256, 768), (1536, 512))
W4A8_BUCKETS = (1, 2, 3, 4)

# The five workloads (N, K, Ms) of the hot path.
TINY_W4A16 = dict(N=256, K=768, M=1, seed=0)
W8_GEMV = dict(N=8192, K=8192, M=1, seed=1)
W4A16_GEMV_SHAPES = ((8448, 6656), (6656, 4096), (6656, 19968), (256, 6656))
W4A16_GEMV_MS = (1, 2, 3, 4)
W4A8_SHAPE = (39936, 6656)
W4A8_MS = (1, 2, 3, 4)
TC_SHAPES = ((39936, 6656), (6656, 19968), (1536, 512))
TC_MS = (16, 64)
# W8 at the skinny-GEMM sizes (on the tensor core)
W8_TC_MS = (16, 64)


def _gen(seed: int) -> torch.Generator:
    return torch.Generator(device="cpu").manual_seed(int(seed))


def w4_seed(N: int, K: int) -> int:
    """Weight seed of a model shape ("test_int4_quantized_gemm.py": n ^ k)."""
    return N ^ K


def x_seed(N: int, K: int, M: int) -> int:
    return N ^ K ^ (1000 + M)


def randn_bf16(shape, seed: int) -> torch.Tensor:
    return torch.randn(*shape, dtype=torch.bfloat16, generator=_gen(seed))


def w4_weight(N: int, K: int, seed: int | None = None) -> torch.Tensor:
    """Dense bf16 weight [N, K] (CPU) to be quantized to INT4."""
    return randn_bf16((N, K), w4_seed(N, K) if seed is None else seed)


def activation(M: int, K: int, seed: int) -> torch.Tensor:
    return randn_bf16((M, K), seed)


def outlier_activation(M: int, K: int, seed: int) -> torch.Tensor:
    """Gaussian bf16 rows with four outlier channels (precision-test recipe)."""
    x = randn_bf16((M, K), seed)
    channels = torch.tensor((0, K // 3, 2 * K // 3, K - 1))
    factors = torch.tensor((50.0, 35.0, 25.0, 20.0), dtype=torch.bfloat16)
    x[:, channels] *= factors
    return x


def tiny_w4a16():
    """N=256, K=768, M=1; one generator seeded 0 draws W then x."""
    g = _gen(TINY_W4A16["seed"])
    N, K, M = TINY_W4A16["N"], TINY_W4A16["K"], TINY_W4A16["M"]
    W = torch.randn(N, K, dtype=torch.bfloat16, generator=g)
    x = torch.randn(M, K, dtype=torch.bfloat16, generator=g)
    return W, x


def w8_inputs(N: int = W8_GEMV["N"], K: int = W8_GEMV["K"], M: int = 1,
              seed: int = W8_GEMV["seed"]):
    """int8 weight uniform in [-128, 127], bf16 per-row scales, bf16 x."""
    g = _gen(seed)
    W = torch.randint(-128, 128, (N, K), dtype=torch.int8, generator=g)
    scales = torch.randn(N, dtype=torch.bfloat16, generator=g)
    x = torch.randn(M, K, dtype=torch.bfloat16, generator=g)
    return W, scales, x
