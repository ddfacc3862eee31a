"""Rotary position embedding (RoPE), 1-D and 3-D video layouts.  Test infrastructure.

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

3-D video layout (optional, ``layout=(S, W, pairs_t, pairs_h)``).  The pages do
not say how the video model lays out its positions; the plain reading for a
(time, height, width) token grid: a token's running index p = frame * S + s
(S tokens per frame, W per row) has coordinates t = p // S, h = (p % S) // W,
w = (p % S) % W.  The d/2 pairs split into three bands -- pairs [0, pairs_t)
rotate by t, the next pairs_h by h, the rest by w -- each band with its own
frequencies theta ** (-2k / d_band), k < d_band / 2, d_band = 2 * pairs in the
band.  A shift by whole frames changes only t, so a position reset rotates only
the temporal band.
"""
from __future__ import annotations

import math

import numpy as np

_TABLE_CACHE: dict = {}


def freqs(d: int, theta: float = 10000.0) -> list:
    """w_i = theta ** (-2i/d) in float64, i < d/2."""
    return [math.pow(float(theta), -2.0 * i / d) for i in range(d // 2)]


def coords_3d(p: int, S: int, W: int):
    """(t, h, w) of running token index p in frames of S tokens, W per row."""
    t, s = divmod(int(p), S)
    return t, s // W, s % W


def pair_angles(p: int, d: int, theta: float = 10000.0, layout=None) -> list:
    """float64 angle of each of the d/2 pairs for running position p."""
    if layout is None:
        return [float(p) * wi for wi in freqs(d, theta)]
    S, W, pt, ph = layout
    pw = d // 2 - pt - ph
    t, h, w = coords_3d(p, S, W)
    ang = [float(t) * wi for wi in freqs(2 * pt, theta)]
    ang += [float(h) * wi for wi in freqs(2 * ph, theta)]
    ang += [float(w) * wi for wi in freqs(2 * pw, theta)]
    return ang


def angle_table(positions, d: int, theta: float = 10000.0, layout=None):
    """(cos, sin) float32 arrays of shape [len(positions), d/2].

    Entry [n, i] is fp32(cos(a)) / fp32(sin(a)) of pair i's angle a at position
    p_n (1-D: p_n * w_i; 3-D: the band's coordinate times its frequency), formed
    and evaluated in float64.  Negative positions are allowed (the delta
    rotation of a reset uses -delta).
    """
    positions = [int(p) for p in np.asarray(positions).reshape(-1)]
    key = (d, float(theta), layout)
    cache = _TABLE_CACHE.setdefault(key, {})
    c = np.empty((len(positions), d // 2), dtype=np.float32)
    s = np.empty((len(positions), d // 2), dtype=np.float32)
    for n, p in enumerate(positions):
        row = cache.get(p)
        if row is None:
            ang = pair_angles(p, d, theta, layout)
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


def rotate_at(x: np.ndarray, positions, d: int, theta: float = 10000.0, layout=None) -> np.ndarray:
    """Rotate rows x[n, ..., d] by position positions[n]."""
    c, s = angle_table(positions, d, theta, layout)
    extra = x.ndim - 2
    shape = (c.shape[0],) + (1,) * extra + (c.shape[1],)
    return rotate(x, c.reshape(shape), s.reshape(shape))
