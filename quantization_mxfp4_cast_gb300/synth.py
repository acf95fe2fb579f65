"""Seeded synthetic inputs shared by the tests, the benchmark and the oracle
checks.  This module only draws random numbers (CPU torch generator, fp32
``randn * sigma`` rounded to bf16); it holds none of the method's arithmetic
and imports neither the CUDA library nor the oracle.

The shapes stand in for the Llama-3.1 8B / 70B MaxText training runs that the
jax-aiter README ("Supported ops", FP4 GEMM row; "Quick start") quotes its
MXFP4 speedups on; weights, datasets and the model are not used.
"""
from __future__ import annotations

import torch

SEED_TINY = 0
SEED_X = 1
SEED_W = 2
SEED_DY = 3
SEED_OUTLIER = 4


def normal_bf16(shape, sigma: float, seed: int) -> torch.Tensor:
    g = torch.Generator(device="cpu")
    g.manual_seed(seed)
    return (torch.randn(*shape, generator=g, dtype=torch.float32) * sigma).to(torch.bfloat16)


def with_outliers(x: torch.Tensor, frac: float = 1e-3, factor: float = 50.0,
                  seed: int = SEED_OUTLIER) -> torch.Tensor:
    """Scale a Bernoulli(frac) subset of entries by `factor` (activation outliers)."""
    g = torch.Generator(device="cpu")
    g.manual_seed(seed)
    mask = torch.rand(*x.shape, generator=g) < frac
    y = x.float()
    y[mask] *= factor
    return y.to(torch.bfloat16)


def tiny(M: int = 256, N: int = 256, K: int = 512):
    """Tiny forward GEMM: A[M,K], B[N,K] ~ N(0,1), one generator seeded 0, A drawn first."""
    g = torch.Generator(device="cpu")
    g.manual_seed(SEED_TINY)
    a = torch.randn(M, K, generator=g, dtype=torch.float32).to(torch.bfloat16)
    b = torch.randn(N, K, generator=g, dtype=torch.float32).to(torch.bfloat16)
    return a, b


def cast_input(rows: int = 8192, cols: int = 4096) -> torch.Tensor:
    """Activations ~ N(0,1) with 0.1% of the entries scaled by 50."""
    return with_outliers(normal_bf16((rows, cols), 1.0, SEED_X))


def linear_layer(M: int, N: int, K: int, x_sigma: float, w_sigma: float = 0.02,
                 dy_sigma: float = 1e-3):
    """One linear layer's training inputs: X[M,K], W[N,K], dY[M,N]."""
    x = normal_bf16((M, K), x_sigma, SEED_X)
    w = normal_bf16((N, K), w_sigma, SEED_W)
    dy = normal_bf16((M, N), dy_sigma, SEED_DY)
    return x, w, dy


# name -> (M, N, K, x_sigma) of the Llama-shaped linear layers
LLAMA_SHAPES = {
    "llama8b_gate_up": (8192, 28672, 4096, 1.0),
    "llama8b_down": (8192, 4096, 14336, 0.02),
    "llama70b_qkv": (8192, 10240, 8192, 1.0),
    "llama70b_o": (8192, 8192, 8192, 1.0),
    "llama70b_gate_up": (8192, 57344, 8192, 1.0),
    "llama70b_down": (8192, 8192, 28672, 1.0),
}
