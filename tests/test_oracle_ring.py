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
