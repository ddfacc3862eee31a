"""Plant plausible mistakes in the oracle (CPU only) and check that a pin catches each.

Every case swaps one oracle function for a subtly wrong version (a flipped sign,
an off-by-one index, a dropped term, a transposed operand, truncation instead of
round-to-nearest-even) and runs the pin that should catch it.  The pin must fail.
"""
import numpy as np
import pytest

import oracle.attention as attention_mod
import oracle.e4m3 as e4m3_mod
import oracle.rope as rope_mod
import oracle.schemes as schemes_mod
import tests.test_oracle_attention as t_att
import tests.test_oracle_e4m3 as t_e4m3
import tests.test_oracle_ring as t_ring
import tests.test_oracle_rope as t_rope
import tests.test_oracle_schemes as t_sch


def _rotate_sign_flipped(x, cos, sin):
    x = np.asarray(x, np.float32)
    y = np.empty_like(x)
    y[..., 0::2] = x[..., 0::2] * cos + x[..., 1::2] * sin
    y[..., 1::2] = -x[..., 0::2] * sin + x[..., 1::2] * cos
    return y


def _rotate_halves(x, cos, sin):
    # "rotate-half" pairing (i, i + d/2) instead of the interleaved (2i, 2i + 1)
    x = np.asarray(x, np.float32)
    h = x.shape[-1] // 2
    y = np.empty_like(x)
    y[..., :h] = x[..., :h] * cos - x[..., h:] * sin
    y[..., h:] = x[..., :h] * sin + x[..., h:] * cos
    return y


def _freqs_off_by_one(d, theta=10000.0):
    import math
    return [math.pow(float(theta), -2.0 * (i + 1) / d) for i in range(d // 2)]


def _encode_truncating(x):
    x = np.asarray(x, np.float64)
    a = np.abs(x)
    _, E = np.frexp(np.where(a > 0, a, 1.0))
    q = np.ldexp(1.0, np.maximum(E - 1, -6) - 3)
    v = np.minimum(np.floor(a / q) * q, 448.0) * np.sign(x)
    return _ORIG_ENCODE(v)


def _encode_nan_above_max(x):
    # overflow to the NaN code instead of saturating at 448
    x = np.asarray(x, np.float64)
    out = _ORIG_ENCODE(np.clip(x, -448.0, 448.0))
    return np.where(np.abs(x) > 448.0, np.where(np.signbit(x), 0xFF, 0x7F), out).astype(np.uint8)


def _encode_ties_away(x):
    # ties rounded away from zero instead of to the even code
    x = np.asarray(x, np.float64)
    a = np.abs(x)
    _, E = np.frexp(np.where(a > 0, a, 1.0))
    q = np.ldexp(1.0, np.maximum(E - 1, -6) - 3)
    v = np.minimum(np.floor(a / q + 0.5) * q, 448.0) * np.where(np.signbit(x), -1.0, 1.0)
    return _ORIG_ENCODE(v)


def _encode_flush_subnormals(x):
    # magnitudes below the smallest normal (2^-6) flushed to zero
    x = np.asarray(x, np.float64)
    return _ORIG_ENCODE(np.where(np.abs(x) < 2.0 ** -6, 0.0 * x, x))


def _attention_no_scale(q, k, v):
    return _ORIG_ATT(np.asarray(q) * np.sqrt(np.asarray(q).shape[-1]), k, v)


def _attention_transposed(q, k, v):
    # softmax over the query axis instead of the key axis
    q = np.asarray(q, np.float64); k = np.asarray(k, np.float64); v = np.asarray(v, np.float64)
    T, H, d = q.shape
    out = np.zeros((T, H, d))
    for h in range(H):
        s = q[:, h] @ k[:, h].T / np.sqrt(d)
        p = np.exp(s - s.max(axis=0, keepdims=True))
        p = p / p.sum(axis=0, keepdims=True)
        out[:, h] = p @ v[:, h]
    return out


def _amax_plain(k):
    return np.abs(np.asarray(k, np.float32)).max(axis=(0, 2)).astype(np.float32)


_ORIG_ENCODE = e4m3_mod.encode
_ORIG_ATT = attention_mod.attention_fp64


class _RingOffByOne(schemes_mod.WriteTimeRing):
    def write(self, k, v):
        slots = super().write(k, v)
        self.head = (self.head + 1) % self.R if self.writes % 3 == 0 else self.head
        return slots


class _RewriteNextSlots(schemes_mod.WriteTimeRing):
    # rewrite lands on the slots after the latest chunk instead of on it
    def rewrite(self, k, v):
        T = np.asarray(k).shape[0]
        slots = (self.head + np.arange(T)) % self.R
        pos = self.last_pos + np.arange(T, dtype=np.int64)
        self._store(np.asarray(k, np.float32), np.asarray(v, np.float32), slots, pos, self.writes - 1)
        return slots


class _RewriteNextPositions(schemes_mod.WriteTimeRing):
    # rewrite rotates K at next_pos (the positions of the chunk to come)
    def rewrite(self, k, v):
        T = np.asarray(k).shape[0]
        slots = (self.head - T + np.arange(T)) % self.R
        pos = self.next_pos + np.arange(T, dtype=np.int64)
        self._store(np.asarray(k, np.float32), np.asarray(v, np.float32), slots, pos, self.writes - 1)
        return slots


class _RewriteStaleScale(schemes_mod.WriteTimeRing):
    # rewrite keeps the first pass's K amax instead of taking the new chunk's
    def rewrite(self, k, v):
        T = np.asarray(k).shape[0]
        slots = (self.head - T + np.arange(T)) % self.R
        old = self.kamax[:, slots].copy()
        super().rewrite(k, v)
        _, ki = schemes_mod.scale_inv(old[:, 0])
        kr = rope_mod.rotate_at(np.asarray(k, np.float32), self.last_pos + np.arange(T), self.d, self.theta)
        self.k8[:, slots, :] = schemes_mod.quantise(kr, ki[None, :, None]).transpose(1, 0, 2)
        self.kamax[:, slots] = old
        return slots


def _rebase_planted(self, sign=-1, turn_v=False, rescale=False, shift_pos=True, shift_q=True):
    # the reset's steps (1-D) with one step made wrong
    delta = self.next_pos - self.count
    if delta != 0 and self.count > 0:
        valid = np.nonzero(self.pos >= 0)[0]
        c, s = rope_mod.angle_table([sign * delta], self.d, self.theta)
        ks, ki = schemes_mod.scale_inv(self.kamax[:, valid])
        x = schemes_mod.dequantise_f32(self.k8[:, valid, :], ks[..., None])
        xr = rope_mod.rotate(x, c[0], s[0])
        if rescale:   # a new scale from the rotated values instead of the frozen one
            amax = np.abs(xr).max(axis=2).astype(np.float32)
            _, ki = schemes_mod.scale_inv(amax)
            self.kamax[:, valid] = amax
        self.k8[:, valid, :] = schemes_mod.quantise(xr, ki[..., None])
        if turn_v:
            vs, vi = schemes_mod.scale_inv(self.vamax[:, valid])
            y = schemes_mod.dequantise_f32(self.v8[:, valid, :], vs[..., None])
            self.v8[:, valid, :] = schemes_mod.quantise(rope_mod.rotate(y, c[0], s[0]), vi[..., None])
        if shift_pos:
            self.pos[valid] -= delta
    self.next_pos = self.count
    if shift_q:
        self.last_pos -= delta
    self.resets += 1
    return int(delta)


class _RebaseDeltaSign(schemes_mod.WriteTimeRing):
    def rebase(self):
        return _rebase_planted(self, sign=+1)


class _RebaseTurnsV(schemes_mod.WriteTimeRing):
    def rebase(self):
        return _rebase_planted(self, turn_v=True)


class _RebaseRescales(schemes_mod.WriteTimeRing):
    def rebase(self):
        return _rebase_planted(self, rescale=True)


class _RebaseKeepsPositions(schemes_mod.WriteTimeRing):
    def rebase(self):
        return _rebase_planted(self, shift_pos=False)


class _RebaseKeepsQPositions(schemes_mod.WriteTimeRing):
    def rebase(self):
        return _rebase_planted(self, shift_q=False)


def _coords_swapped(p, S, W):
    t, s = divmod(int(p), S)
    return t, s % W, s // W


def _pair_angles_full_width(p, d, theta=10000.0, layout=None):
    # every band takes the frequencies of the whole head width
    if layout is None:
        return _ORIG_PAIR_ANGLES(p, d, theta, None)
    S, W, pt, ph = layout
    t, h, w = rope_mod.coords_3d(p, S, W)
    f = rope_mod.freqs(d, theta)
    return [float(t) * f[i] for i in range(pt)] + [float(h) * f[pt + i] for i in range(ph)] + \
        [float(w) * f[pt + ph + i] for i in range(d // 2 - pt - ph)]


_ORIG_PAIR_ANGLES = rope_mod.pair_angles


def _quantise_q_per_column(q, positions, d, theta, layout=None):
    # scale per column (over tokens) instead of per (token, head) row
    qr = rope_mod.rotate_at(np.asarray(q, dtype=np.float32), positions, d, theta, layout)
    amax = np.abs(qr).max(axis=0, keepdims=True).astype(np.float32)
    _, inv = schemes_mod.scale_inv(amax)
    codes = schemes_mod.quantise(qr, inv)
    return codes, np.broadcast_to(np.abs(qr).max(axis=2), qr.shape[:2]).astype(np.float32)


CASES = [
    ("rotation sign", [(rope_mod, "rotate", _rotate_sign_flipped)], t_rope.test_unit_vector_rotates_to_cos_sin),
    ("rotate-half pairing", [(rope_mod, "rotate", _rotate_halves)], t_rope.test_matches_complex_multiplication),
    ("frequency index", [(rope_mod, "freqs", _freqs_off_by_one)], t_rope.test_frequencies_closed_form),
    ("e4m3 truncation", [(e4m3_mod, "encode", _encode_truncating)], t_e4m3.test_encode_random_float32_matches_library),
    ("e4m3 overflow to NaN", [(e4m3_mod, "encode", _encode_nan_above_max)], t_e4m3.test_satfinite),
    ("e4m3 ties away from zero", [(e4m3_mod, "encode", _encode_ties_away)], t_e4m3.test_encode_at_rounding_midpoints),
    ("e4m3 subnormals flushed", [(e4m3_mod, "encode", _encode_flush_subnormals)],
     lambda: t_e4m3.test_encode_matches_library_cast_all_bf16(1.0)),
    ("missing 1/sqrt(d)", [(t_att, "attention_fp64", _attention_no_scale)], t_att.test_scale_is_one_over_sqrt_d),
    ("softmax axis", [(t_att, "attention_fp64", _attention_transposed)], t_att.test_rows_are_convex_combinations_and_key_order_free),
    ("K amax not pair norm", [(t_sch, "chunk_amax_k", _amax_plain)], t_sch.test_amax_k_is_largest_pair_norm_bruteforce),
    ("ring head drift", [(t_ring, "WriteTimeRing", _RingOffByOne)], lambda: t_ring.test_logical_order_equals_shifted_window(96, 32)),
    ("3-D height/width swapped", [(rope_mod, "coords_3d", _coords_swapped)], t_rope.test_3d_each_band_is_1d_rope_at_its_coordinate),
    ("3-D band frequencies", [(rope_mod, "pair_angles", _pair_angles_full_width)], t_rope.test_3d_each_band_is_1d_rope_at_its_coordinate),
    ("Q scale per column", [(schemes_mod, "quantise_q", _quantise_q_per_column)], t_sch.test_q_rows_reach_the_top_code_and_stay_within_half_a_step),
    ("rewrite slots", [(t_ring, "WriteTimeRing", _RewriteNextSlots)], lambda: t_ring.test_rewrite_equals_writing_that_chunk(10, 4, 3)),
    ("rewrite positions", [(t_ring, "WriteTimeRing", _RewriteNextPositions)], t_ring.test_rewrite_after_reset_uses_the_shifted_positions),
    ("rewrite stale scale", [(t_ring, "WriteTimeRing", _RewriteStaleScale)], lambda: t_ring.test_rewrite_equals_writing_that_chunk(12, 4, 3)),
    ("rebase delta sign", [(t_sch, "WriteTimeRing", _RebaseDeltaSign)],
     lambda: t_sch.test_rebase_within_one_pair_step_of_fresh_rotation(96, 32, 2, 64)),
    ("rebase turns V", [(t_sch, "WriteTimeRing", _RebaseTurnsV)],
     lambda: t_sch.test_rebase_within_one_pair_step_of_fresh_rotation(96, 32, 2, 64)),
    ("rebase re-scales K", [(t_ring, "WriteTimeRing", _RebaseRescales)],
     t_ring.test_reset_keeps_scales_and_rebases_positions_to_the_window),
    ("rebase keeps positions", [(t_ring, "WriteTimeRing", _RebaseKeepsPositions)],
     t_ring.test_reset_keeps_scales_and_rebases_positions_to_the_window),
    ("rebase leaves Q positions", [(t_sch, "WriteTimeRing", _RebaseKeepsQPositions)],
     t_sch.test_attention_nearly_unchanged_by_a_reset),
]


@pytest.mark.parametrize("name,patches,pin", CASES, ids=[c[0] for c in CASES])
def test_planted_mistake_is_caught(monkeypatch, name, patches, pin):
    for mod, attr, fn in patches:
        monkeypatch.setattr(mod, attr, fn)
    rope_mod._TABLE_CACHE.clear()
    with pytest.raises(AssertionError):
        pin()
    rope_mod._TABLE_CACHE.clear()
