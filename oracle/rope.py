"""1-D rotary position embedding (RoPE).  Test infrastructure.

The pages say RoPE is applied to K once, when a chunk is written, and that at
each position reset one delta rotation is applied to the cached window
([ai.info] § "La gestione della cache spostata al momento della scrittura";
[neurocartel] § "Кэш: 240 attention calls и работа на запись";
[wechild] ¶8).  They do not give the RoPE layout.  Readings used here:

* Interleaved pairs (x[2i], x[2i+1]) of a head vector of length d are rotated
  by the angle p * w_i, with w_i = theta ** (-2i/d), i < d/2, theta = 10000,
  p the token's absolute 1-D position.
* The angle and its cosine and sine are evaluated in float64 and rounded once
  to float32.  Each value is computed with the C library's ``pow``, ``cos``
  and ``sin`` (Python's ``math`` module), one call per element.
* The rotation itself runs in float32 with every product and sum rounded
  separately (no fused multiply-add):
      y0 = x0*c - x1*s
      y1 = x0*s + x1*c
"""
from __future__ import annotations

import math

import numpy as np

_TABLE_CACHE: dict = {}


def freqs(d: int, theta: float = 10000.0) -> list:
    """w_i = theta ** (-2i/d) in float64, i < d/2."""
    return [math.pow(float(theta), -2.0 * i / d) for i in range(d // 2)]


def angle_table(positions, d: int, theta: float = 10000.0):
    """(cos, sin) float32 arrays of shape [len(positions), d/2].

    Entry [n, i] is fp32(cos(p_n * w_i)) / fp32(sin(p_n * w_i)), the angle
    formed and evaluated in float64.  Negative positions are allowed (the
    delta rotation of a reset uses -delta).
    """
    positions = [int(p) for p in np.asarray(positions).reshape(-1)]
    w = freqs(d, theta)
    key = (d, float(theta))
    cache = _TABLE_CACHE.setdefault(key, {})
    c = np.empty((len(positions), d // 2), dtype=np.float32)
    s = np.empty((len(positions), d // 2), dtype=np.float32)
    for n, p in enumerate(positions):
        row = cache.get(p)
        if row is None:
            ang = [float(p) * wi for wi in w]
            row = (np.array([math.cos(a) for a in ang], dtype=np.float32),
                   np.array([math.sin(a) for a in ang], dtype=np.float32))
            cache[p] = row
        c[n], s[n] = row
    return c, s


def rotate(x: np.ndarray, cos: np.ndarray, sin: np.ndarray) -> np.ndarray:
    """Rotate interleaved pairs of x [..., d] (float32) by per-pair angles.

    cos/sin broadcast against x[..., 0::2].  Arithmetic in float32, each
    operation rounded on its own.
    """
    x = np.asarray(x, dtype=np.float32)
    x0 = x[..., 0::2]
    x1 = x[..., 1::2]
    c = np.asarray(cos, dtype=np.float32)
    s = np.asarray(sin, dtype=np.float32)
    y = np.empty_like(x)
    a = (x0 * c).astype(np.float32)
    b = (x1 * s).astype(np.float32)
    y[..., 0::2] = (a - b).astype(np.float32)
    a = (x0 * s).astype(np.float32)
    b = (x1 * c).astype(np.float32)
    y[..., 1::2] = (a + b).astype(np.float32)
    return y


def rotate_at(x: np.ndarray, positions, d: int, theta: float = 10000.0) -> np.ndarray:
    """Rotate rows x[n, ..., d] by position positions[n]."""
    c, s = angle_table(positions, d, theta)
    extra = x.ndim - 2
    shape = (c.shape[0],) + (1,) * extra + (c.shape[1],)
    return rotate(x, c.reshape(shape), s.reshape(shape))
