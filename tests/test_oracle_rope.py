"""Pins for the oracle's RoPE: closed-form rotations, composition, inverse, norm."""
import math

import numpy as np

from oracle import rope


def test_frequencies_closed_form():
    # d = 4, theta = 10000: w = (1, 10000**-0.5 = 0.01)
    w = rope.freqs(4, 10000.0)
    assert w[0] == 1.0 and abs(w[1] - 0.01) < 1e-17
    w = rope.freqs(128, 10000.0)
    assert w[0] == 1.0
    assert abs(w[32] - 0.01) < 1e-15                    # 10000**(-64/128)
    assert abs(w[63] - 10000.0 ** (-126 / 128)) < 1e-18
    assert all(a > b for a, b in zip(w, w[1:]))        # strictly decreasing


def test_position_zero_is_identity():
    rng = np.random.default_rng(0)
    x = rng.standard_normal((5, 3, 64)).astype(np.float32)
    y = rope.rotate_at(x, np.zeros(5, np.int64), 64)
    assert np.array_equal(x, y)


def test_unit_vector_rotates_to_cos_sin():
    # pair 0 has w = 1: (1, 0) at position p -> (cos p, sin p); (0, 1) -> (-sin p, cos p)
    d = 4
    for p in [1, 7, 100, 31794]:
        x = np.array([[[1.0, 0.0, 0.0, 1.0]]], np.float32)
        y = rope.rotate_at(x, [p], d)[0, 0]
        assert y[0] == np.float32(math.cos(p)) and y[1] == np.float32(math.sin(p))
        # pair 1 has w = 0.01
        a = p * 0.01
        assert abs(y[2] + math.sin(a)) < 1e-7 and abs(y[3] - math.cos(a)) < 1e-7


def test_matches_complex_multiplication():
    rng = np.random.default_rng(1)
    d, T = 128, 50
    x = rng.standard_normal((T, 2, d)).astype(np.float32) * 4
    pos = rng.integers(0, 40000, T)
    y = rope.rotate_at(x, pos, d)
    z = (x[..., 0::2].astype(np.float64) + 1j * x[..., 1::2].astype(np.float64))
    w = np.array(rope.freqs(d))
    z = z * np.exp(1j * pos[:, None, None] * w[None, None, :])
    assert np.max(np.abs(y[..., 0::2] - z.real)) < 1e-5
    assert np.max(np.abs(y[..., 1::2] - z.imag)) < 1e-5


def test_pair_norm_preserved():
    rng = np.random.default_rng(2)
    x = rng.standard_normal((40, 4, 128)).astype(np.float32) * 20
    y = rope.rotate_at(x, rng.integers(0, 37582, 40), 128)
    n0 = np.hypot(x[..., 0::2].astype(np.float64), x[..., 1::2])
    n1 = np.hypot(y[..., 0::2].astype(np.float64), y[..., 1::2])
    assert np.max(np.abs(n0 - n1) / np.maximum(n0, 1e-30)) < 1e-6


def test_composition_delta_rotation():
    """rotate(p) then rotate(-delta) equals rotate(p - delta) within 1e-6 (relative to max|x|)."""
    rng = np.random.default_rng(3)
    d = 128
    x = rng.standard_normal((64, 4, d)).astype(np.float32)
    x[rng.random(x.shape) < 0.01] *= 20
    p = rng.integers(26006, 37582, 64)
    for delta in [26006, 31794, 1248, 1344, 1]:
        c, s = rope.angle_table([-delta], d)
        twice = rope.rotate(rope.rotate_at(x, p, d), c[0], s[0])
        fresh = rope.rotate_at(x, p - delta, d)
        err = np.max(np.abs(twice.astype(np.float64) - fresh)) / np.max(np.abs(x))
        assert err < 1e-6, (delta, err)


def test_negative_position_inverts():
    rng = np.random.default_rng(4)
    x = rng.standard_normal((10, 1, 64)).astype(np.float32)
    p = rng.integers(0, 37582, 10)
    y = rope.rotate_at(x, p, 64)
    back = rope.rotate_at(y, -p, 64)
    assert np.max(np.abs(back - x)) < 1e-5
    # cos is even and sin is odd, value for value
    c1, s1 = rope.angle_table([12345], 64)
    c2, s2 = rope.angle_table([-12345], 64)
    assert np.array_equal(c1, c2) and np.array_equal(s1, -s2)


def test_angles_formed_in_float64():
    # p * w_i rounded to float32 before cos/sin would miss the float64 value by up to ~2e-3 here
    d = 128
    p = 37581
    c, s = rope.angle_table([p], d)
    w = rope.freqs(d)
    for i in (0, 1, 5):
        assert c[0, i] == np.float32(math.cos(p * w[i]))
        assert s[0, i] == np.float32(math.sin(p * w[i]))


# ---- 3-D video layout: frames of S tokens, W per row; pairs split (t, h, w)

def _layout(d, S, W, pt, ph):
    assert pt + ph < d // 2
    return (S, W, pt, ph)


def test_3d_one_token_frames_is_1d_rope_on_the_time_band():
    # S = W = 1: every token is its own frame at h = w = 0, so the time band is the
    # 1-D RoPE of width 2 pt at the token's index and the other pairs stay exactly
    d, pt, ph = 64, 12, 10
    lay = _layout(d, 1, 1, pt, ph)
    rng = np.random.default_rng(1)
    x = rng.standard_normal((40, 3, d)).astype(np.float32)
    pos = rng.integers(0, 30000, size=40)
    y = rope.rotate_at(x, pos, d, layout=lay)
    assert np.array_equal(y[..., :2 * pt], rope.rotate_at(x[..., :2 * pt], pos, 2 * pt))
    assert np.array_equal(y[..., 2 * pt:], x[..., 2 * pt:])


def test_3d_each_band_is_1d_rope_at_its_coordinate():
    # frames of 12 tokens in rows of 4: band h sees the row, band w the column,
    # band t the frame; each band equals the 1-D RoPE of its width at that index
    d, S, W, pt, ph = 128, 12, 4, 22, 21
    pw = d // 2 - pt - ph
    lay = _layout(d, S, W, pt, ph)
    rng = np.random.default_rng(2)
    pos = np.arange(5 * S + 3)
    x = rng.standard_normal((len(pos), 2, d)).astype(np.float32)
    y = rope.rotate_at(x, pos, d, layout=lay)
    t, s = pos // S, pos % S
    bands = [(0, pt, t), (pt, ph, s // W), (pt + ph, pw, s % W)]
    for start, n, coord in bands:
        sl = slice(2 * start, 2 * (start + n))
        assert np.array_equal(y[..., sl], rope.rotate_at(x[..., sl], coord, 2 * n))


def test_3d_frame_shift_composes():
    # rotating at p and then by -delta frames equals rotating at p - delta (fp32)
    d, S, W = 128, 12, 4
    lay = _layout(d, S, W, 22, 21)
    rng = np.random.default_rng(3)
    x = rng.standard_normal((64, d)).astype(np.float32)
    pos = rng.integers(6000, 9000, size=64)
    delta = 250 * S
    c, s = rope.angle_table([-delta], d, layout=lay)
    twice = rope.rotate(rope.rotate_at(x, pos, d, layout=lay), c[0], s[0])
    once = rope.rotate_at(x, pos - delta, d, layout=lay)
    assert np.max(np.abs(twice - once)) < 1e-5 * max(1.0, np.max(np.abs(x)))
    # the reset's rotation row turns the height and width bands by exactly zero
    assert np.all(c[0, 22:] == 1.0) and np.all(s[0, 22:] == 0.0)


def test_3d_scores_depend_on_coordinate_differences_only():
    # q.k after rotation is unchanged when both tokens move by the same number of
    # frames (relative-position property of each band)
    d, S, W = 64, 20, 5
    lay = _layout(d, S, W, 12, 10)
    rng = np.random.default_rng(4)
    q = rng.standard_normal((30, d)).astype(np.float64)
    k = rng.standard_normal((30, d)).astype(np.float64)
    pq = rng.integers(0, 400, size=30)
    pk = rng.integers(0, 400, size=30)
    def score(shift):
        rq = rope.rotate_at(q.astype(np.float32), pq + shift, d, layout=lay).astype(np.float64)
        rk = rope.rotate_at(k.astype(np.float32), pk + shift, d, layout=lay).astype(np.float64)
        return np.sum(rq * rk, axis=-1)
    assert np.max(np.abs(score(0) - score(37 * S))) < 1e-4
    # a shift that is not a whole number of frames moves the spatial coordinates
    assert np.max(np.abs(score(0) - score(3))) > 1e-2
