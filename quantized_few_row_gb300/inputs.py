"""Seeded synthetic inputs shared by the tests, the smoke check and the bench.

This module only draws random numbers: it holds none of the mat-vec's or the
block formats' arithmetic.  Weights are drawn as W ~ N(0, 0.02) and inputs as
x ~ N(0, 1), both float32, from numpy's PCG64 (host) or a seeded torch
generator (device, for the large bench workloads).  Quantizing the drawn
weights into blocks is done by whoever consumes them (the oracle's quantizer
in the tests, the library's ``rem_quantize`` in the bench).
"""
from __future__ import annotations

import numpy as np

W_STD = 0.02
X_STD = 1.0


def normal(shape, seed: int, std: float = 1.0) -> np.ndarray:
    """float32 N(0, std^2) array from PCG64(seed)."""
    g = np.random.Generator(np.random.PCG64(seed))
    return (g.standard_normal(size=shape, dtype=np.float32) * np.float32(std)).astype(np.float32)


def weights(rows: int, k: int, seed: int) -> np.ndarray:
    return normal((rows, k), seed, W_STD)


def activations(m: int, k: int, seed: int) -> np.ndarray:
    return normal((m, k), seed, X_STD)


def uniform_bytes(count: int, seed: int) -> np.ndarray:
    g = np.random.Generator(np.random.PCG64(seed))
    return g.integers(0, 256, size=count, dtype=np.uint8)


def small_ints(shape, seed: int, lo: int, hi: int) -> np.ndarray:
    """Integers in [lo, hi] as float32 (exactly representable inputs)."""
    g = np.random.Generator(np.random.PCG64(seed))
    return g.integers(lo, hi + 1, size=shape).astype(np.float32)


def torch_normal(shape, seed: int, std: float, device):
    """Device-side N(0, std^2) float32 tensor from a seeded torch generator."""
    import torch
    g = torch.Generator(device=device)
    g.manual_seed(seed)
    t = torch.empty(shape, dtype=torch.float32, device=device)
    t.normal_(0.0, std, generator=g)
    return t
