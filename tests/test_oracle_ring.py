"""Pins for the oracle's ring bookkeeping: shifted-window order, closed forms, resets."""
import os

import numpy as np
import pytest

from oracle.schemes import NaiveWindow, WriteTimeRing

GOLDEN = os.path.join(os.path.dirname(__file__), "golden", "reset_schedule.txt")


def _zeros(T, H=1, d=2):
    return np.zeros((T, H, d), np.float32)


def _ring_logical(ring: WriteTimeRing, field):
    """Ring contents oldest-first: slots head-count .. head-1 (mod R)."""
    idx = (ring.head - ring.count + np.arange(ring.count)) % ring.R
    return field[idx]


@pytest.mark.parametrize("R,T", [(96, 32), (100, 32), (5788, 757), (7, 3), (16, 16), (10, 1)])
def test_logical_order_equals_shifted_window(R, T):
    ring = WriteTimeRing(R, 1, 2)
    naive = NaiveWindow(R, 1, 2)
    writes = max(6 * R // T + 3, 10)          # at least five wraps
    for w in range(writes):
        ring.write(_zeros(T), _zeros(T))
        naive.write(_zeros(T), _zeros(T))
        assert ring.count == naive.count == min((w + 1) * T, R)
        assert ring.head == ((w + 1) * T) % R
        assert ring.next_pos == naive.next_pos == (w + 1) * T
        assert np.array_equal(_ring_logical(ring, ring.pos), naive.pos)
        assert np.array_equal(_ring_logical(ring, ring.chunk), naive.chunk)
        # physical slot of logical token g is g mod R
        assert np.array_equal(naive.gidx % R, (ring.head - ring.count + np.arange(ring.count)) % R)


def _golden_rows():
    rows, maxpos = [], {}
    for line in open(GOLDEN):
        if not line.strip() or line.startswith("#"):
            continue
        f = line.split()
        if f[0] == "max_position":
            maxpos[f[1]] = int(f[2])
        else:
            rows.append((f[0], *map(int, f[1:])))
    return rows, maxpos


def test_reset_schedule_matches_golden():
    rows, maxpos = _golden_rows()
    assert len(rows) >= 5
    configs = {name: (R, T) for name, R, T, *_ in rows}
    for name, (R, T) in configs.items():
        want = {step: (npb, cnt, dl) for n, _, _, step, npb, cnt, dl in rows if n == name}
        last = max(want)
        ring = WriteTimeRing(R, 1, 2)
        naive = NaiveWindow(R, 1, 2)
        seen_max = -1
        for s in range(last + 1):
            if s > 0 and s % 42 == 0:
                before = (ring.next_pos, ring.count)
                d1 = ring.rebase()
                d2 = naive.rebase()
                assert d1 == d2
                if s in want:
                    assert (before[0], before[1], d1) == want[s], (name, s)
                assert ring.next_pos == ring.count
                assert np.array_equal(np.sort(ring.pos[ring.pos >= 0]), np.arange(ring.count))
            ring.write(_zeros(T), _zeros(T))
            naive.write(_zeros(T), _zeros(T))
            seen_max = max(seen_max, int(ring.pos.max()))
        if name in maxpos:
            assert seen_max == maxpos[name]


def test_each_token_rebased_at_most_once_production():
    R, T = 5788, 757
    ring = WriteTimeRing(R, 1, 2)
    times = {}
    for s in range(300):
        if s > 0 and s % 42 == 0:
            ring.rebase()
            for c in np.unique(ring.chunk[ring.chunk >= 0]):
                times[int(c)] = times.get(int(c), 0) + 1
        ring.write(_zeros(T), _zeros(T))
    assert max(times.values()) == 1
    # with fixed-size writes the window is the last R tokens, whose start sits
    # (-R) mod T = 268 tokens into a chunk: ceil(R / T) = 8 chunks are live
    lifetimes = []
    ring = WriteTimeRing(R, 1, 2)
    for w in range(60):
        ring.write(_zeros(T), _zeros(T))
        live = set(int(c) for c in np.unique(ring.chunk[ring.chunk >= 0]))
        lifetimes.append(len(live))
    assert max(lifetimes) == 8 and lifetimes[-1] == 8


def test_scale_frozen_through_eviction():
    R, T, H, d = 10, 4, 2, 4
    ring = WriteTimeRing(R, H, d)
    rng = np.random.default_rng(0)
    chunks = [rng.standard_normal((T, H, d)).astype(np.float32) * (w + 1) for w in range(4)]
    for c in chunks:
        ring.write(c, c)
    # chunks 0..3 start at slots 0, 4, 8, 2 (12 mod 10): chunk 2 wraps onto 0,1 and
    # chunk 3 takes 2..5, so chunk 0 is gone and chunk 1 keeps only slots 6, 7
    assert list(ring.chunk) == [2, 2, 3, 3, 3, 3, 1, 1, 2, 2]
    from oracle.schemes import chunk_amax_k
    assert np.all(ring.kamax[:, 6] == chunk_amax_k(chunks[1]))
    assert np.all(ring.kamax[:, 7] == chunk_amax_k(chunks[1]))


def test_reset_keeps_scales_and_rebases_positions_to_the_window():
    """A reset keeps every slot's frozen K and V scale and chunk id (scales are
    fixed once, at write) and rebases the window to positions 0 .. count - 1,
    oldest slot first (delta = next_pos - count)."""
    R, T, H, d = 10, 4, 2, 4
    ring = WriteTimeRing(R, H, d)
    rng = np.random.default_rng(1)
    for w in range(5):
        c = rng.standard_normal((T, H, d)).astype(np.float32) * (w + 1)
        ring.write(c, 2 * c)
    kam, vam, chunk = ring.kamax.copy(), ring.vamax.copy(), ring.chunk.copy()
    assert ring.rebase() == 20 - 10
    assert np.array_equal(ring.kamax, kam) and np.array_equal(ring.vamax, vam)
    assert np.array_equal(ring.chunk, chunk)
    assert list(_ring_logical(ring, ring.pos)) == list(range(10))
    assert ring.next_pos == ring.count == 10 and ring.last_pos == 6


def _ring_arrays(r: WriteTimeRing):
    return (r.k8, r.v8, r.kamax, r.vamax, r.pos, r.chunk)


def _ring_counters(r: WriteTimeRing):
    return (r.head, r.count, r.next_pos, r.writes, r.last_pos, r.last_n, r.resets)


@pytest.mark.parametrize("R,T,nw", [(10, 4, 3), (10, 4, 5), (12, 4, 3), (7, 7, 2), (300, 100, 4)])
def test_rewrite_equals_writing_that_chunk(R, T, nw):
    # history c_0..c_{nw-2}, then c_{nw-1} written and replaced by x over 3 passes:
    # the ring must equal the one that wrote x in c_{nw-1}'s place (nw = 3 at R = 10
    # straddles the ring's end; R = 12 ends on it; T = R overwrites everything)
    H, d = 2, 8
    rng = np.random.default_rng(R * 131 + T * 7 + nw)
    mk = lambda s: (rng.standard_normal((T, H, d)) * s).astype(np.float32)
    hist = [(mk(w + 1), mk(w + 2)) for w in range(nw)]
    passes = [(mk(3 + p), mk(0.5 + p)) for p in range(3)]
    a, b = WriteTimeRing(R, H, d), WriteTimeRing(R, H, d)
    for k, v in hist:
        a.write(k, v)
    for k, v in hist[:-1]:
        b.write(k, v)
    before = [x.copy() for x in _ring_arrays(a)]
    counters = _ring_counters(a)
    for k, v in passes:
        slots = a.rewrite(k, v)
        assert _ring_counters(a) == counters
    b.write(*passes[-1])
    assert list(slots) == list((b.head - T + np.arange(T)) % R)
    for x, y in zip(_ring_arrays(a), _ring_arrays(b)):
        assert np.array_equal(x, y)
    assert _ring_counters(a) == _ring_counters(b)
    # no slot outside the latest chunk moved
    others = np.ones(R, bool)
    others[slots] = False
    for i, (x, y) in enumerate(zip(before, _ring_arrays(a))):
        ax = 1 if i < 4 else 0                          # slot axis: [H][R](...), then [R]
        assert np.array_equal(np.compress(others, x, axis=ax), np.compress(others, y, axis=ax))


def test_rewrite_after_reset_uses_the_shifted_positions():
    # after a reset the latest chunk sits at count - T; a rewrite there must code x
    # exactly as a fresh ring that wrote x at that position
    R, T, H, d = 12, 4, 2, 8
    rng = np.random.default_rng(5)
    a = WriteTimeRing(R, H, d)
    for w in range(5):                                   # next_pos 20, count 12: delta 8
        a.write(rng.standard_normal((T, H, d)).astype(np.float32), rng.standard_normal((T, H, d)).astype(np.float32))
    assert a.rebase() == 8
    assert a.last_pos == R - T
    x = (rng.standard_normal((T, H, d)) * 3).astype(np.float32)
    y = rng.standard_normal((T, H, d)).astype(np.float32)
    slots = a.rewrite(x, y)
    assert list(a.pos[slots]) == list(range(R - T, R))
    b = WriteTimeRing(R, H, d)
    b.write(np.ones((R - T, H, d), np.float32), np.ones((R - T, H, d), np.float32))
    fresh = b.write(x, y)
    assert np.array_equal(a.k8[:, slots], b.k8[:, fresh])
    assert np.array_equal(a.v8[:, slots], b.v8[:, fresh])
    assert np.array_equal(a.kamax[:, slots], b.kamax[:, fresh])


def test_rewrite_needs_a_write_of_the_same_size():
    r = WriteTimeRing(8, 1, 2)
    with pytest.raises(AssertionError):
        r.rewrite(_zeros(4), _zeros(4))
    r.write(_zeros(4), _zeros(4))
    with pytest.raises(AssertionError):
        r.rewrite(_zeros(3), _zeros(3))


def test_3d_reset_rotates_only_the_time_band():
    # with the 3-D layout a reset is a whole number of frames: the codes of the
    # height and width bands stay as they are, the time band turns; the window's
    # time-band codes agree with a fresh write at the shifted frames within one
    # pair step (reading of the rebase for 1-D RoPE)
    from oracle.schemes import NaiveWindow
    R, T, H, d, S, W = 48, 12, 2, 64, 12, 4
    lay = (S, W, 12, 10)
    ring = WriteTimeRing(R, H, d, layout=lay)
    naive = NaiveWindow(R, H, d, layout=lay)
    rng = np.random.default_rng(9)
    for w in range(7):
        k = rng.standard_normal((T, H, d)).astype(np.float32)
        v = rng.standard_normal((T, H, d)).astype(np.float32)
        ring.write(k, v)
        naive.write(k, v)
    before = ring.k8.copy()
    assert ring.rebase() == naive.rebase() == 3 * T
    assert np.array_equal(ring.k8[..., 24:], before[..., 24:])
    assert np.mean(ring.k8[..., :24] != before[..., :24]) > 0.3
    k8, _, _, _ = naive.cache_codes()
    idx = (ring.head - ring.count + np.arange(ring.count)) % R
    # a whole-frame shift leaves height and width as they were: those codes equal a
    # fresh rotation at the shifted positions exactly
    assert np.array_equal(ring.k8[:, idx, 24:], k8.transpose(1, 0, 2)[..., 24:])
    from oracle import e4m3
    a = e4m3.decode(ring.k8[:, idx])
    b = e4m3.decode(k8.transpose(1, 0, 2))
    big = np.maximum(np.abs(a), np.abs(b))
    pair_big = np.maximum(big[..., 0::2], big[..., 1::2])
    step = e4m3.ulp_at(np.repeat(pair_big, 2, axis=-1))
    assert np.max(np.abs(a - b) / step) <= 1.0
