"""Seeded synthetic inputs (bf16 bit patterns) shared by the tests, the benchmark
and the oracle checks.  This module holds no arithmetic of the method: it draws
numbers, applies the outlier recipes and rounds to bf16.

Recipes (Llama-3.1-8B-shaped linear layers; the pages train on C4, which is
replaced by these distributions):
  X   ~ N(0, 1) with 1% of feature channels (columns) scaled x50
  W   ~ N(0, 0.02)
  dY  ~ N(0, 1e-4) with 2% of tokens (rows) scaled x20
  sweep tensors: 0.1 * Student-t(df=3) with 0.1% of entries scaled x100
Seeds: workload index c uses base 1000*c; X / W / dY use base + 0 / 1 / 2.
"""
from __future__ import annotations

import numpy as np


def rng(seed: int) -> np.random.Generator:
    return np.random.Generator(np.random.PCG64(seed))


def bf16_bits(a: np.ndarray) -> np.ndarray:
    """fp32 -> bf16 (round to nearest even) as uint16 bit patterns."""
    a = np.ascontiguousarray(a, dtype=np.float32)
    u = a.view(np.uint32).astype(np.uint64)
    r = (u + 0x7FFF + ((u >> 16) & 1)) >> 16
    return r.astype(np.uint16)


def bf16_to_f32(b: np.ndarray) -> np.ndarray:
    return (np.ascontiguousarray(b, dtype=np.uint16).astype(np.uint32) << 16).view(np.float32)


def _n_outliers(frac: float, n: int) -> int:
    return max(1, int(round(frac * n)))


def activations(M: int, K: int, seed: int) -> np.ndarray:
    """X [M, K]: N(0,1), 1% of channels x50."""
    g = rng(seed)
    x = g.standard_normal((M, K), dtype=np.float32)
    cols = g.permutation(K)[:_n_outliers(0.01, K)]
    x[:, cols] *= np.float32(50.0)
    return bf16_bits(x)


def weights(N: int, K: int, seed: int, std: float = 0.02) -> np.ndarray:
    """W [N, K]: N(0, std)."""
    g = rng(seed)
    w = g.standard_normal((N, K), dtype=np.float32) * np.float32(std)
    return bf16_bits(w)


def output_grads(M: int, N: int, seed: int) -> np.ndarray:
    """dY [M, N]: N(0, 1e-4), 2% of tokens x20."""
    g = rng(seed)
    d = g.standard_normal((M, N), dtype=np.float32) * np.float32(1e-4)
    rows = g.permutation(M)[:_n_outliers(0.02, M)]
    d[rows, :] *= np.float32(20.0)
    return bf16_bits(d)


def heavy_tailed(R: int, C: int, seed: int) -> np.ndarray:
    """0.1 * Student-t(df=3) with 0.1% of entries x100."""
    g = rng(seed)
    t = (g.standard_t(3, size=(R, C)) * 0.1).astype(np.float32)
    flat = t.reshape(-1)
    idx = g.permutation(flat.size)[:_n_outliers(0.001, flat.size)]
    flat[idx] *= np.float32(100.0)
    return bf16_bits(t)


def linear_inputs(M: int, N: int, K: int, base_seed: int):
    """(X [M,K], W [N,K], dY [M,N]) for one linear layer."""
    return (activations(M, K, base_seed + 0), weights(N, K, base_seed + 1),
            output_grads(M, N, base_seed + 2))


# Llama-3.1-8B linear shapes at T tokens: (name, N = out features, K = in features)
LLAMA8B_LINEARS = (
    ("qkv", 6144, 4096),
    ("o", 4096, 4096),
    ("gate_up", 14336, 4096),
    ("down", 4096, 14336),
)

LLAMA8B_BLOCK_LINEARS = (
    ("q", 4096, 4096), ("k", 1024, 4096), ("v", 1024, 4096), ("o", 4096, 4096),
    ("gate", 14336, 4096), ("up", 14336, 4096), ("down", 4096, 14336),
)
