"""Pins for the two oracle schemes against each other and against closed forms.

The pages' central claim is that doing RoPE and FP8 once at write time, with a
ring buffer and one delta rotation per reset, reproduces the naive per-call
upkeep.  Before any reset that is an identity (same codes, same order); after a
reset the delta-rotated codes must sit within one e4m3 step of a fresh
rotation at the new positions, the step taken at the larger magnitude of the
element's RoPE pair.
"""
import math

import numpy as np
import pytest

from kv_cache_gb300 import synthetic
from oracle import e4m3, rope
from oracle.schemes import (NaiveWindow, WriteTimeRing, chunk_amax_k, chunk_amax_v,
                            dequantise_f64, quantise, scale_inv)


def _chunk(role, idx, T, H, d, outliers=False):
    return synthetic.bf16_to_f32(synthetic.chunk(role, idx, T, H, d, outliers))


def _logical(ring, arr):
    idx = (ring.head - ring.count + np.arange(ring.count)) % ring.R
    return arr[:, idx]


def _pair_ulp_diff(a_codes, b_codes):
    """|decode(a) - decode(b)| in units of the e4m3 step at max(|b0|, |b1|) of b's pair."""
    a = e4m3.decode(a_codes)
    b = e4m3.decode(b_codes)
    mag = np.maximum(np.abs(b[..., 0::2]), np.abs(b[..., 1::2]))
    mag = np.repeat(mag, 2, axis=-1)
    return np.abs(a - b) / e4m3.ulp_at(mag)


def _pair_norm_ulp_diff(a_codes, b_codes):
    """|decode(a) - decode(b)| in units of the e4m3 step at the norm of b's pair.

    A RoPE pair is a 2-D vector; a rotation keeps its norm and moves its larger
    element anywhere between norm / sqrt(2) and norm, so the norm is the one
    magnitude the cached pair and a fresh rotation of it share."""
    a = e4m3.decode(a_codes)
    b = e4m3.decode(b_codes)
    norm = np.sqrt(b[..., 0::2] ** 2 + b[..., 1::2] ** 2)
    return np.abs(a - b) / e4m3.ulp_at(np.repeat(norm, 2, axis=-1))


def test_amax_k_is_largest_pair_norm_bruteforce():
    x = _chunk("k", 0, 5, 2, 8, outliers=True)
    got = chunk_amax_k(x)
    for h in range(2):
        best = 0.0
        for t in range(5):
            for i in range(4):
                best = max(best, math.hypot(float(x[t, h, 2 * i]), float(x[t, h, 2 * i + 1])))
        assert abs(got[h] - best) <= 1e-6 * best
    assert np.all(chunk_amax_v(x) == np.abs(x).max(axis=(0, 2)))


def test_amax_k_rotation_invariant():
    x = _chunk("k", 1, 64, 4, 128, outliers=True)
    xr = rope.rotate_at(x, np.arange(30000, 30064), 128)
    assert np.allclose(chunk_amax_k(xr), chunk_amax_k(x), rtol=1e-6, atol=0)


def test_quantise_error_within_half_step():
    x = _chunk("v", 2, 32, 2, 64, outliers=True)
    amax = chunk_amax_v(x)
    scale, inv = scale_inv(amax)
    codes = quantise(x, inv[None, :, None])
    back = dequantise_f64(codes, scale[None, :, None])
    y = x.astype(np.float64) * inv[None, :, None].astype(np.float64)   # value in code units
    err = np.abs(back / scale[None, :, None] - y)
    assert np.all(err <= 0.5 * e4m3.ulp_at(np.abs(y)) * (1 + 1e-6) + 1e-12)
    # the largest element maps to (almost) 448 and nothing saturates beyond it
    assert np.max(e4m3.decode(codes)) <= 448.0 and np.max(np.abs(e4m3.decode(codes))) >= 416.0


def test_scale_inv_zero_amax():
    s, i = scale_inv(np.array([0.0, 448.0, 3.5], np.float32))
    assert s[0] == 1 and i[0] == 1 and s[1] == 1 and i[1] == 1
    assert s[2] == np.float32(3.5) / np.float32(448) and i[2] == np.float32(448) / np.float32(3.5)


@pytest.mark.parametrize("R,T,H,d", [(96, 32, 2, 64), (100, 32, 2, 64), (37, 8, 1, 16)])
def test_writetime_equals_naive_before_reset(R, T, H, d):
    naive = NaiveWindow(R, H, d)
    ring = WriteTimeRing(R, H, d)
    for w in range(2 * R // T + 3):
        k = _chunk("k", w, T, H, d, outliers=True)
        v = _chunk("v", w, T, H, d, outliers=True)
        naive.write(k, v)
        ring.write(k, v)
        k8, v8, ks, vs = naive.cache_codes()
        assert np.array_equal(_logical(ring, ring.k8), k8.transpose(1, 0, 2))
        assert np.array_equal(_logical(ring, ring.v8), v8.transpose(1, 0, 2))
        if w % 3 == 0:
            q = _chunk("q", w, T, H, d)
            a = naive.attend(q)
            b = ring.attend(q)
            assert np.max(np.abs(a - b)) < 1e-12


@pytest.mark.parametrize("R,T,H,d", [(96, 32, 2, 64), (100, 32, 2, 64), (8, 8, 1, 16)])
def test_rewrite_passes_writetime_equals_naive(R, T, H, d):
    # the two schemes hold the same codes after every denoise pass, including the
    # passes that replace the latest chunk, and attend alike
    naive = NaiveWindow(R, H, d)
    ring = WriteTimeRing(R, H, d)
    for w in range(2 * R // T + 2):
        for p in range(4):
            k = _chunk("k", 40 * w + p, T, H, d, outliers=p == 2)
            v = _chunk("v", 40 * w + p, T, H, d, outliers=p == 3)
            if p == 0:
                naive.write(k, v)
                ring.write(k, v)
            else:
                naive.rewrite(k, v)
                ring.rewrite(k, v)
            k8, v8, _, _ = naive.cache_codes()
            assert np.array_equal(_logical(ring, ring.k8), k8.transpose(1, 0, 2))
            assert np.array_equal(_logical(ring, ring.v8), v8.transpose(1, 0, 2))
        q = _chunk("q", w, T, H, d)
        assert np.max(np.abs(naive.attend(q) - ring.attend(q))) < 1e-12


@pytest.mark.parametrize("R,T,H,d", [(96, 32, 2, 64), (100, 32, 2, 64)])
def test_rebase_within_one_pair_step_of_fresh_rotation(R, T, H, d):
    naive = NaiveWindow(R, H, d)
    ring = WriteTimeRing(R, H, d)
    worst = 0.0
    for s in range(100):
        if s > 0 and s % 42 == 0:
            v_before = ring.v8.copy()
            k_before = ring.k8.copy()
            assert ring.rebase() == naive.rebase()
            assert np.array_equal(ring.v8, v_before)          # V untouched
            assert np.mean(ring.k8 != k_before) > 0.5          # K really rotated
            k8, v8, _, _ = naive.cache_codes()
            diff = _pair_ulp_diff(_logical(ring, ring.k8), k8.transpose(1, 0, 2))
            worst = max(worst, float(diff.max()))
            assert np.array_equal(_logical(ring, ring.v8), v8.transpose(1, 0, 2))
        k = _chunk("k", s, T, H, d, outliers=True)
        v = _chunk("v", s, T, H, d, outliers=True)
        naive.write(k, v)
        ring.write(k, v)
    # one step of the pair's larger element; measured by the element's own step
    # the worst case is hundreds of steps, since the rotation moves the large
    # partner's rounding error into the small one
    assert worst == 1.0


def test_rebase_within_one_pair_step_at_production_deltas():
    """d = 128, the production ring (5,788 slots, 757-token chunks) and its reset
    deltas: the first reset (before step 42's write) moves the window by
    42 x 757 - 5,788 = 26,006 positions, every later one by 42 x 757 = 31,794.
    Two heads keep the run short; the deltas and the rotation angles are the
    production ones.  Every delta-rotated code is within one e4m3 step of a
    fresh rotation at the new positions, the step taken at the pair's norm.
    Taken at the fresh pair's larger element instead, a handful of the 1.48 M
    codes per reset are two steps apart: there the rotation has moved the larger
    element one binade below the norm, while the cached codes still carry the
    rounding of the pair before the rotation."""
    R, T, H, d = 5788, 757, 2, 128
    naive = NaiveWindow(R, H, d)
    ring = WriteTimeRing(R, H, d)
    deltas = []
    for s in range(85):
        if s > 0 and s % 42 == 0:
            deltas.append(ring.rebase())
            assert naive.rebase() == deltas[-1]
            k8, _, _, _ = naive.cache_codes()
            fresh = k8.transpose(1, 0, 2)
            got = _logical(ring, ring.k8)
            assert _pair_norm_ulp_diff(got, fresh).max() == 1.0, s
            by_larger = _pair_ulp_diff(got, fresh)
            assert by_larger.max() <= 2.0 and np.mean(by_larger <= 1.0) >= 0.99999, s
            assert np.mean(got == fresh) > 0.6, s
        k = _chunk("k", 3000 + s, T, H, d, outliers=True)
        v = _chunk("v", 3000 + s, T, H, d, outliers=True)
        naive.write(k, v)
        ring.write(k, v)
    assert deltas == [26006, 31794]


def test_attention_nearly_unchanged_by_a_reset():
    """RoPE scores depend only on position differences, and a reset shifts the
    positions of the cached K and of the next Q together, so the same queries
    attend alike before and after it: only the FP8 roundings of Q and of the
    rotated K differ (measured ~4 % mean relative change on Gaussian data),
    while shifting one side alone decorrelates the result (~100 %)."""
    R, T, H, d = 96, 32, 2, 64
    ring = WriteTimeRing(R, H, d)
    for w in range(7):
        ring.write(_chunk("k", w, T, H, d), _chunk("v", w, T, H, d))
    q = _chunk("q", 3, T, H, d)
    before = ring.attend(q)
    assert ring.rebase() == 7 * T - R
    after = ring.attend(q)
    assert np.abs(after - before).sum() / np.abs(before).sum() < 0.25


def test_rebase_after_partial_fill_and_twice():
    R, T, H, d = 64, 10, 1, 16
    ring = WriteTimeRing(R, H, d)
    naive = NaiveWindow(R, H, d)
    for w in range(3):                    # count = 30 < R
        k = _chunk("k", 50 + w, T, H, d)
        ring.write(k, k); naive.write(k, k)
    assert ring.rebase() == 0             # next_pos == count: nothing to rotate
    assert ring.next_pos == 30
    for w in range(9):
        k = _chunk("k", 60 + w, T, H, d)
        ring.write(k, k); naive.write(k, k)
    naive.rebase(); naive.rebase()
    d1 = ring.rebase(); d2 = ring.rebase()
    assert d1 == 120 - 64 and d2 == 0
    k8, _, _, _ = naive.cache_codes()
    assert _pair_ulp_diff(_logical(ring, ring.k8), k8.transpose(1, 0, 2)).max() <= 1.0


def test_q_rows_reach_the_top_code_and_stay_within_half_a_step():
    # each (token, head) row of Q is scaled so that its largest rotated |value|
    # lands on the top code (448), and every dequantised value is within half an
    # e4m3 step of the rotated value (the RoPE routine is pinned on its own)
    from oracle import e4m3, rope
    from oracle.schemes import quantise_q, dequantised_q
    rng = np.random.default_rng(31)
    T, H, d = 40, 3, 64
    q = (rng.standard_normal((T, H, d)) * rng.choice([0.01, 1.0, 30.0], size=(T, H, 1))).astype(np.float32)
    q[5, 1] = 0.0                                           # an all-zero row
    pos = np.arange(100, 100 + T)
    codes, amax = quantise_q(q, pos, d, 10000.0)
    mags = np.abs(e4m3.decode(codes))
    top = mags.max(axis=2)
    assert top[5, 1] == 0.0 and amax[5, 1] == 0.0
    nz = np.ones((T, H), bool)
    nz[5, 1] = False
    assert np.all(top[nz] == 448.0)
    qr = rope.rotate_at(q, pos, d).astype(np.float64)
    deq = dequantised_q(q, pos, d, 10000.0)
    scale = (amax.astype(np.float64) / 448.0)[..., None]
    step = e4m3.ulp_at(np.abs(qr) / np.where(scale > 0, scale, 1.0)) * scale
    assert np.all(np.abs(deq - qr) <= 0.5 * step * (1 + 1e-6) + 1e-30)


def test_dequantisers_are_exact_products():
    # fl32(decode * scale) is the float32 rounding of the exact product, and the
    # float64 form is the exact product itself (two float32 factors)
    from fractions import Fraction
    from oracle import e4m3
    from oracle.schemes import dequantise_f32, dequantise_f64
    rng = np.random.default_rng(32)
    codes = rng.integers(0, 256, size=400).astype(np.uint8)
    codes = codes[(codes & 0x7F) != 0x7F]                   # no NaN codes
    scale = (rng.random(codes.shape) * 3 + 1e-3).astype(np.float32)
    exact = [Fraction(float(e4m3.decode(np.array([c]))[0])) * Fraction(float(s)) for c, s in zip(codes, scale)]
    f64 = dequantise_f64(codes, scale)
    assert all(Fraction(float(v)) == x for v, x in zip(f64, exact))
    f32 = dequantise_f32(codes, scale)
    assert all(np.float32(float(x)) == v for v, x in zip(f32, exact))
