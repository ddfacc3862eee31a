"""Seeded synthetic inputs shared by the tests, the bench and the oracle.

This module holds none of the cache method's arithmetic: it only draws random
numbers and rounds them to bf16.  Recipe:

* Generator: NumPy PCG64 seeded with (role seed, chunk index).  Role seeds:
  0 = K, 1 = V, 2 = Q, 3 = outlier masks.
* Values: N(0, 1) in float32.  With ``outliers=True`` an independent
  Bernoulli(0.01) mask per element multiplies the value by 20.
* Values are rounded to bf16 (round to nearest even) and returned as uint16
  bit patterns of shape [T][H][d]; ``bf16_to_f32`` widens them exactly.
* A run does not draw fresh data for every call: the pool of ``POOL`` distinct
  chunks per role is uploaded once, and call (step, layer, pass) uses entry
  ``pool_index(step, layer, pass_)``.
"""
from __future__ import annotations

import numpy as np

ROLE_SEED = {"k": 0, "v": 1, "q": 2, "mask": 3}
POOL = 16


def _f32_to_bf16_bits(x: np.ndarray) -> np.ndarray:
    u = np.asarray(x, np.float32).view(np.uint32).astype(np.uint64)
    rounding = ((u >> 16) & 1) + 0x7FFF
    return ((u + rounding) >> 16).astype(np.uint16)


def bf16_to_f32(bits: np.ndarray) -> np.ndarray:
    """uint16 bf16 bit patterns -> float32 (exact)."""
    return (np.asarray(bits, np.uint16).astype(np.uint32) << 16).view(np.float32)


def chunk(role: str, index: int, T: int, H: int, d: int, outliers: bool = False) -> np.ndarray:
    """One seeded [T][H][d] chunk as bf16 bit patterns (uint16)."""
    rng = np.random.Generator(np.random.PCG64([ROLE_SEED[role], int(index)]))
    x = rng.standard_normal((T, H, d), dtype=np.float32)
    if outliers:
        mrng = np.random.Generator(np.random.PCG64([ROLE_SEED["mask"], ROLE_SEED[role], int(index)]))
        mask = mrng.random((T, H, d)) < 0.01
        x = np.where(mask, x * np.float32(20.0), x).astype(np.float32)
    return _f32_to_bf16_bits(x)


def pool_index(step: int, layer: int, pass_: int, num_layers: int) -> int:
    """Pool entry for (step, layer, pass); pass 4 is the K/V write of the step."""
    return (step * num_layers * 5 + layer * 5 + pass_) % POOL
