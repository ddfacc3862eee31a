"""The naive cache upkeep and the write-time cache, as plain NumPy.  Test infrastructure.

Both classes hold one transformer block's KV cache for H heads of size d and a
window of R tokens, fed chunks of T tokens (bf16 values passed as float32).

NaiveWindow follows the upkeep the pages say the launch software did: on
every attention call it re-applies RoPE to the whole window, re-quantises it
and shifts the window ([wechild] ¶7; [neurocartel] § "Кэш: 240 attention
calls и работа на запись"; [ai.info] § "La gestione della cache spostata al
momento della scrittura").  The window is a list in logical order; a write
appends and drops the oldest rows (a copy, on purpose).  Rotation happens only
inside ``attend``; a position reset only changes the stored positions.

WriteTimeRing follows the method the pages describe: a ring buffer that
overwrites the oldest slots instead of copying, RoPE and FP8 quantisation
applied once when a chunk is written, and one delta rotation of the cached
window when positions reset ([ai.info] and [neurocartel], same sections;
[wechild] ¶8).

Readings of what the pages leave open (kept identical in both classes):

* One scale per (head, written chunk), frozen at write time and kept by every
  slot of that chunk for life, through partial eviction and rebase.
* K's chunk amax is the largest pair norm fl32(sqrt(fl32(x0*x0 + x1*x1))) over
  the chunk's un-rotated bf16 pairs (a rotation cannot change it); V's chunk
  amax is the largest |v|.  scale = fl32(amax / 448), inv = fl32(448 / amax);
  amax == 0 gives scale = inv = 1.
* code = e4m3_rne_satfinite(fl32(x * inv)); dequantised value
  fl32(decode(code) * scale) where the value feeds float32 arithmetic.
* Slot of the j-th token of write w (ring starts empty at slot 0):
  (head + j) mod R with head = (w * T) mod R for fixed T; after the write
  head += T (mod R), count = min(count + T, R), next_pos += T.
* Position reset: delta = next_pos - count; every cached position drops by
  delta (the window becomes positions [0, count)); next_pos = count.  The
  write-time ring applies the rotation by -delta to each cached K in place,
  re-quantising with the slot's frozen scale; V is left alone.
* Q of an attention call sits at the positions of the latest write; it is
  rotated there and quantised per row (plain amax over the row's d values),
  and the attention uses the dequantised Q.
"""
from __future__ import annotations

import numpy as np

from . import e4m3, rope
from .attention import attention_fp64

F32 = np.float32


def chunk_amax_k(k: np.ndarray) -> np.ndarray:
    """Per-head K amax of a chunk k [T][H][d] (float32 holding bf16): largest pair norm."""
    k = np.asarray(k, dtype=F32)
    x0 = k[..., 0::2]
    x1 = k[..., 1::2]
    n2 = (x0 * x0).astype(F32) + (x1 * x1).astype(F32)
    norm = np.sqrt(n2.astype(F32)).astype(F32)
    if norm.shape[0] == 0:
        return np.zeros(k.shape[1], dtype=F32)
    return norm.max(axis=(0, 2)).astype(F32)


def chunk_amax_v(v: np.ndarray) -> np.ndarray:
    """Per-head V amax of a chunk v [T][H][d]: largest |v|."""
    v = np.asarray(v, dtype=F32)
    if v.shape[0] == 0:
        return np.zeros(v.shape[1], dtype=F32)
    return np.abs(v).max(axis=(0, 2)).astype(F32)


def scale_inv(amax: np.ndarray):
    """(scale, inv) in float32 from amax; amax == 0 -> (1, 1)."""
    amax = np.asarray(amax, dtype=F32)
    zero = amax == 0
    safe = np.where(zero, F32(1), amax).astype(F32)
    scale = (safe / F32(448.0)).astype(F32)
    inv = (F32(448.0) / safe).astype(F32)
    scale = np.where(zero, F32(1), scale).astype(F32)
    inv = np.where(zero, F32(1), inv).astype(F32)
    return scale, inv


def quantise(x: np.ndarray, inv: np.ndarray) -> np.ndarray:
    """e4m3 codes of fl32(x * inv); inv broadcasts against x."""
    y = (np.asarray(x, dtype=F32) * np.asarray(inv, dtype=F32)).astype(F32)
    return e4m3.encode(y)


def dequantise_f32(code: np.ndarray, scale: np.ndarray) -> np.ndarray:
    """fl32(decode(code) * scale)."""
    return (e4m3.decode(code).astype(F32) * np.asarray(scale, dtype=F32)).astype(F32)


def dequantise_f64(code: np.ndarray, scale: np.ndarray) -> np.ndarray:
    """decode(code) * scale in float64 (exact product of two float32 values)."""
    return e4m3.decode(code) * np.asarray(scale, dtype=np.float64)


def quantise_q(q: np.ndarray, positions, d: int, theta: float, layout=None):
    """Rotate q [T][H][d] at positions[T] and quantise each (token, head) row.

    Returns (codes uint8 [T][H][d], amax float32 [T][H]).
    """
    qr = rope.rotate_at(np.asarray(q, dtype=F32), positions, d, theta, layout)
    amax = np.abs(qr).max(axis=2).astype(F32) if qr.shape[0] else np.zeros(qr.shape[:2], F32)
    _, inv = scale_inv(amax)
    codes = quantise(qr, inv[..., None])
    return codes, amax


def dequantised_q(q: np.ndarray, positions, d: int, theta: float, layout=None) -> np.ndarray:
    codes, amax = quantise_q(q, positions, d, theta, layout)
    scale, _ = scale_inv(amax)
    return dequantise_f64(codes, scale[..., None])


class NaiveWindow:
    """Shift-the-window cache that redoes RoPE and quantisation on every call."""

    def __init__(self, capacity: int, num_heads: int, head_dim: int, theta: float = 10000.0, layout=None):
        self.R, self.H, self.d, self.theta = capacity, num_heads, head_dim, float(theta)
        self.layout = layout
        self.k = np.zeros((0, num_heads, head_dim), F32)   # un-rotated bf16 values
        self.v = np.zeros((0, num_heads, head_dim), F32)
        self.pos = np.zeros(0, np.int64)
        self.chunk = np.zeros(0, np.int64)
        self.gidx = np.zeros(0, np.int64)                   # token index since the ring was created
        self.kamax = {}                                     # chunk id -> float32 [H]
        self.vamax = {}
        self.next_pos = 0
        self.writes = 0
        self.tokens = 0
        self.resets = 0
        self.last_pos = 0
        self.last_n = 0

    @property
    def count(self) -> int:
        return int(self.k.shape[0])

    def write(self, k: np.ndarray, v: np.ndarray) -> None:
        k = np.asarray(k, F32)
        v = np.asarray(v, F32)
        T = k.shape[0]
        c = self.writes
        self.kamax[c] = chunk_amax_k(k)
        self.vamax[c] = chunk_amax_v(v)
        pos = self.next_pos + np.arange(T, dtype=np.int64)
        # append, then shift the window by dropping the oldest rows (a copy)
        self.k = np.concatenate([self.k, k])[-self.R:].copy()
        self.v = np.concatenate([self.v, v])[-self.R:].copy()
        self.pos = np.concatenate([self.pos, pos])[-self.R:].copy()
        self.chunk = np.concatenate([self.chunk, np.full(T, c, np.int64)])[-self.R:].copy()
        self.gidx = np.concatenate([self.gidx, self.tokens + np.arange(T, dtype=np.int64)])[-self.R:].copy()
        self.last_pos, self.last_n = self.next_pos, T
        self.next_pos += T
        self.tokens += T
        self.writes += 1

    def rewrite(self, k: np.ndarray, v: np.ndarray) -> None:
        """The next denoise pass's k, v for the latest chunk: its rows (the newest T of
        the window) take the new values and the chunk its new amax; nothing shifts."""
        k = np.asarray(k, F32)
        v = np.asarray(v, F32)
        T = k.shape[0]
        assert self.writes > 0 and T == self.last_n
        c = self.writes - 1
        self.kamax[c] = chunk_amax_k(k)
        self.vamax[c] = chunk_amax_v(v)
        self.k[-T:] = k
        self.v[-T:] = v

    def rebase(self) -> int:
        delta = self.next_pos - self.count
        self.pos = self.pos - delta
        self.next_pos = self.count
        self.last_pos -= delta
        self.resets += 1
        return int(delta)

    def chunk_scales(self):
        """Per-row (kscale, kinv, vscale, vinv), each float32 [count][H]."""
        ka = np.stack([self.kamax[int(c)] for c in self.chunk]) if self.count else np.zeros((0, self.H), F32)
        va = np.stack([self.vamax[int(c)] for c in self.chunk]) if self.count else np.zeros((0, self.H), F32)
        ks, ki = scale_inv(ka)
        vs, vi = scale_inv(va)
        return ks, ki, vs, vi, ka, va

    def cache_codes(self):
        """Re-rotate and re-quantise the whole window (the per-call upkeep).

        Returns (k codes, v codes, kscale, vscale) in logical order.
        """
        ks, ki, vs, vi, _, _ = self.chunk_scales()
        kr = rope.rotate_at(self.k, self.pos, self.d, self.theta, self.layout)
        k8 = quantise(kr, ki[..., None])
        v8 = quantise(self.v, vi[..., None])
        return k8, v8, ks, vs

    def attend(self, q: np.ndarray) -> np.ndarray:
        """Naive per-call upkeep, then float64 attention.  q [T][H][d] -> O [T][H][d]."""
        k8, v8, ks, vs = self.cache_codes()
        kd = dequantise_f64(k8, ks[..., None])
        vd = dequantise_f64(v8, vs[..., None])
        qpos = self.last_pos + np.arange(q.shape[0], dtype=np.int64)
        qd = dequantised_q(q, qpos, self.d, self.theta, self.layout)
        return attention_fp64(qd, kd, vd)


class WriteTimeRing:
    """Ring-buffer cache: RoPE and FP8 once at write, delta rotation at reset."""

    def __init__(self, capacity: int, num_heads: int, head_dim: int, theta: float = 10000.0, layout=None):
        R, H, d = capacity, num_heads, head_dim
        self.R, self.H, self.d, self.theta = R, H, d, float(theta)
        self.layout = layout
        self.k8 = np.zeros((H, R, d), np.uint8)
        self.v8 = np.zeros((H, R, d), np.uint8)
        self.kamax = np.zeros((H, R), F32)
        self.vamax = np.zeros((H, R), F32)
        self.pos = np.full(R, -1, np.int64)
        self.chunk = np.full(R, -1, np.int64)
        self.head = 0
        self.count = 0
        self.next_pos = 0
        self.writes = 0
        self.resets = 0
        self.last_pos = 0
        self.last_n = 0

    def write(self, k: np.ndarray, v: np.ndarray) -> np.ndarray:
        """Write one chunk k, v [T][H][d]; returns the slots used."""
        k = np.asarray(k, F32)
        v = np.asarray(v, F32)
        T = k.shape[0]
        assert 0 < T <= self.R
        slots = (self.head + np.arange(T)) % self.R
        pos = self.next_pos + np.arange(T, dtype=np.int64)
        self._store(k, v, slots, pos, self.writes)
        self.last_pos, self.last_n = self.next_pos, T
        self.head = (self.head + T) % self.R
        self.count = min(self.count + T, self.R)
        self.next_pos += T
        self.writes += 1
        return slots

    def rewrite(self, k: np.ndarray, v: np.ndarray) -> np.ndarray:
        """The next denoise pass's k, v [T][H][d] for the latest chunk; returns its slots.

        The model runs its blocks four times per step and each pass makes new K
        and V for the newest chunk (ai.info, "La gestione della cache spostata al
        momento della scrittura": four passes, 240 attention calls per step).  The
        pages say nothing more; the plain reading: the same slots, positions and
        chunk id as the latest write, a new per-head scale from the new amax, and
        no change to head, count, next_pos or the write counter.
        """
        k = np.asarray(k, F32)
        v = np.asarray(v, F32)
        T = k.shape[0]
        assert self.writes > 0 and T == self.last_n
        slots = (self.head - T + np.arange(T)) % self.R
        pos = self.last_pos + np.arange(T, dtype=np.int64)
        self._store(k, v, slots, pos, self.writes - 1)
        return slots

    def _store(self, k, v, slots, pos, chunk_id):
        """RoPE K at ``pos``, quantise K and V with this chunk's scales, store at ``slots``."""
        ka = chunk_amax_k(k)
        va = chunk_amax_v(v)
        _, ki = scale_inv(ka)
        _, vi = scale_inv(va)
        kr = rope.rotate_at(k, pos, self.d, self.theta, self.layout)   # [T][H][d]
        k8 = quantise(kr, ki[None, :, None])
        v8 = quantise(v, vi[None, :, None])
        self.k8[:, slots, :] = k8.transpose(1, 0, 2)
        self.v8[:, slots, :] = v8.transpose(1, 0, 2)
        self.kamax[:, slots] = ka[:, None]
        self.vamax[:, slots] = va[:, None]
        self.pos[slots] = pos
        self.chunk[slots] = chunk_id

    def rebase(self) -> int:
        """Delta-rotate every cached K by -delta in place; returns delta."""
        delta = self.next_pos - self.count
        if delta != 0 and self.count > 0:
            valid = np.nonzero(self.pos >= 0)[0]
            c, s = rope.angle_table([-delta], self.d, self.theta, self.layout)   # [1][d/2]
            # pairs the reset turns: all of them in 1-D; in the 3-D layout a reset
            # moves whole frames and only the time band turns -- the other pairs'
            # codes stay as stored (a rotation by exactly zero could still flip
            # the sign of a zero code)
            n = self.d // 2 if self.layout is None else self.layout[2]
            ks, ki = scale_inv(self.kamax[:, valid])                 # [H][n]
            x = dequantise_f32(self.k8[:, valid, :2 * n], ks[..., None])
            xr = rope.rotate(x, c[0, :n], s[0, :n])
            self.k8[:, valid, :2 * n] = quantise(xr, ki[..., None])
            self.pos[valid] -= delta
        self.next_pos = self.count
        self.last_pos -= delta
        self.resets += 1
        return int(delta)

    def valid_slots(self) -> np.ndarray:
        return np.nonzero(self.pos >= 0)[0]

    def attend(self, q: np.ndarray, heads=None, rows=None) -> np.ndarray:
        """float64 attention of q [T][H][d] over the finished cache.

        ``heads`` / ``rows`` select a subset of heads and query rows (sampled
        parity at full size); the result has the selected shape.
        """
        T = q.shape[0]
        heads = np.arange(self.H) if heads is None else np.asarray(heads)
        rows = np.arange(T) if rows is None else np.asarray(rows)
        valid = self.valid_slots()
        ks, _ = scale_inv(self.kamax[np.ix_(heads, valid)])
        vs, _ = scale_inv(self.vamax[np.ix_(heads, valid)])
        kd = dequantise_f64(self.k8[np.ix_(heads, valid)], ks[..., None]).transpose(1, 0, 2)
        vd = dequantise_f64(self.v8[np.ix_(heads, valid)], vs[..., None]).transpose(1, 0, 2)
        qpos = self.last_pos + rows.astype(np.int64)
        qd = dequantised_q(np.asarray(q, F32)[np.ix_(rows, heads)], qpos, self.d, self.theta, self.layout)
        return attention_fp64(qd, kd, vd)
