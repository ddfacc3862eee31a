"""GPU parity: the CUDA path through the C ABI against the CPU oracle on the same seeded inputs.

Bars: ring indices, positions and chunk ids bit-exact; FP8 K/V codes identical on
>= 99.9% of elements and never more than one e4m3 step apart; chunk amax exact;
attention max-abs <= 2e-2 and mean relative error <= 5e-3 against the oracle's
float64 attention over its own (identical) dequantised cache.
"""
import numpy as np
import pytest

from kv_cache_gb300 import kvring as kv
from oracle.schemes import WriteTimeRing
from tests._lib import ensure_built
from tests.gpu_util import (assert_attention_close, assert_codes_match, chunk_pair, to_dev)

pytestmark = pytest.mark.gpu


@pytest.fixture(scope="module", autouse=True)
def _lib():
    ensure_built()


def _check_cache(ring, layer, o: WriteTimeRing, min_identical=0.999):
    snap = ring.snapshot(layer)
    st = ring.state(layer)
    assert (st["head"], st["count"], st["next_pos"], st["writes"]) == (o.head, o.count, o.next_pos, o.writes)
    assert np.array_equal(snap["pos"].astype(np.int64), o.pos)
    assert np.array_equal(snap["chunk"].astype(np.int64), o.chunk)
    valid = o.pos >= 0
    assert np.array_equal(snap["kamax"][:, valid], o.kamax[:, valid])
    assert np.array_equal(snap["vamax"][:, valid], o.vamax[:, valid])
    fk = assert_codes_match(snap["k"][:, valid], o.k8[:, valid], min_identical, "K codes")
    fv = assert_codes_match(snap["v"][:, valid], o.v8[:, valid], min_identical, "V codes")
    return fk, fv


@pytest.mark.parametrize("R,T,H,d,outliers", [(96, 32, 2, 64, False), (100, 32, 2, 64, True),
                                               (300, 100, 3, 128, True), (16, 16, 1, 128, False)])
def test_write_small(R, T, H, d, outliers):
    ring = kv.KVRing(1, H, d, R, T, max_position=4096)
    o = WriteTimeRing(R, H, d)
    for w in range(2 * R // T + 3):
        kb, kf = chunk_pair("k", w, T, H, d, outliers)
        vb, vf = chunk_pair("v", w, T, H, d, outliers)
        ring.write(0, to_dev(kb), to_dev(vb))
        o.write(kf, vf)
        fk, fv = _check_cache(ring, 0, o)
        assert fk == 1.0 and fv == 1.0


def test_write_production_shape():
    R, T, H, d = 5788, 757, 16, 128
    ring = kv.KVRing(1, H, d, R, T, max_position=8192)
    o = WriteTimeRing(R, H, d)
    for w in range(9):                       # fills, then wraps (the 9th write straddles the end)
        kb, kf = chunk_pair("k", w, T, H, d, True)
        vb, vf = chunk_pair("v", w, T, H, d, True)
        ring.write(0, to_dev(kb), to_dev(vb))
        o.write(kf, vf)
    fk, fv = _check_cache(ring, 0, o)
    assert fk == 1.0 and fv == 1.0


@pytest.mark.parametrize("R,T,H,d,writes", [(300, 290, 3, 128, 5), (4100, 2048, 2, 128, 4), (2100, 2048, 1, 64, 3),
                                             (61, 50, 2, 64, 6)])
def test_write_long_chunks(R, T, H, d, writes):
    """Chunks of more than R - 16 tokens (their end wraps into the 16-slot group of
    their first slot) and of 2,048 tokens (17 groups per CTA of a cluster of 8):
    codes and amax bit-exact with the oracle after every write."""
    ring = kv.KVRing(1, H, d, R, T, max_position=T * (writes + 1))
    o = WriteTimeRing(R, H, d)
    for w in range(writes):
        kb, kf = chunk_pair("k", 300 + w, T, H, d, True)
        vb, vf = chunk_pair("v", 300 + w, T, H, d, True)
        ring.write(0, to_dev(kb), to_dev(vb))
        o.write(kf, vf)
        fk, fv = _check_cache(ring, 0, o)
        assert fk == 1.0 and fv == 1.0, f"write {w}: {fk}, {fv}"
    assert ring.check_device() == kv.KVRING_OK


@pytest.mark.parametrize("d", [64, 128])
def test_write_whole_ring_chunks_from_mid_group(d):
    """Chunks as long as the ring (T = R = 2,048) written from a slot inside a
    16-slot group: the chunk's last tokens land in its first slot's group, before
    its first token.  Bit-exact with the oracle after each write."""
    R = T = 2048
    H = 2
    ring = kv.KVRing(1, H, d, R, T, max_position=4 * T)
    o = WriteTimeRing(R, H, d)
    for w, n in enumerate([5, T, 21, T, T]):
        kb, kf = chunk_pair("k", 600 + w, T, H, d, True)
        vb, vf = chunk_pair("v", 600 + w, T, H, d, True)
        ring.write(0, to_dev(kb[:n]), to_dev(vb[:n]))
        o.write(kf[:n], vf[:n])
        fk, fv = _check_cache(ring, 0, o)
        assert fk == 1.0 and fv == 1.0, f"write {w} ({n} tokens): {fk}, {fv}"
    assert ring.check_device() == kv.KVRING_OK


def test_write_and_attend_at_the_head_limit():
    """256 heads (the library's limit): the write's 4,096 CTAs (a cluster of 8 per
    head and K|V) and the attention's grid, codes bit-exact, attention in tolerance."""
    R, T, H, d = 160, 48, 256, 64
    ring = kv.KVRing(1, H, d, R, T, max_position=4096)
    o = WriteTimeRing(R, H, d)
    for w in range(5):                       # fills and wraps
        kb, kf = chunk_pair("k", 500 + w, T, H, d, True)
        vb, vf = chunk_pair("v", 500 + w, T, H, d, True)
        ring.write(0, to_dev(kb), to_dev(vb))
        o.write(kf, vf)
        fk, fv = _check_cache(ring, 0, o)
        assert fk == 1.0 and fv == 1.0
    qb, qf = chunk_pair("q", 505, T, H, d, True)
    heads = np.array([0, 77, 128, 255])
    out = ring.attend(0, to_dev(qb)).cpu().numpy()
    assert_attention_close(out[:, heads], o.attend(qf, heads=heads), "256 heads")
    assert ring.check_device() == kv.KVRING_OK


# (600, 150, 2, 64): as the ring fills, 2, 3, 4 and 3 KV splits, merged as clusters
@pytest.mark.parametrize("R,T,H,d", [(96, 32, 2, 64), (100, 32, 2, 64), (300, 100, 2, 128), (600, 150, 2, 64)])
def test_attend_small(R, T, H, d):
    ring = kv.KVRing(1, H, d, R, T, max_position=4096)
    o = WriteTimeRing(R, H, d)
    for w in range(2 * R // T + 2):
        kb, kf = chunk_pair("k", w, T, H, d, True)
        vb, vf = chunk_pair("v", w, T, H, d, True)
        ring.write(0, to_dev(kb), to_dev(vb))
        o.write(kf, vf)
        qb, qf = chunk_pair("q", w, T, H, d, True)
        out = ring.attend(0, to_dev(qb)).cpu().numpy()
        assert_attention_close(out, o.attend(qf), f"write {w}")


def test_attend_warmup_partial_ring():
    # count < R: slots past count are never written and must be masked
    R, T, H, d = 1000, 130, 2, 128
    ring = kv.KVRing(1, H, d, R, T)
    o = WriteTimeRing(R, H, d)
    for w in range(3):
        kb, kf = chunk_pair("k", 100 + w, T, H, d)
        vb, vf = chunk_pair("v", 100 + w, T, H, d)
        ring.write(0, to_dev(kb), to_dev(vb))
        o.write(kf, vf)
        qb, qf = chunk_pair("q", 100 + w, T, H, d)
        assert_attention_close(ring.attend(0, to_dev(qb)).cpu().numpy(), o.attend(qf))


def test_attend_production_sampled():
    R, T, H, d = 5788, 757, 16, 128
    ring = kv.KVRing(1, H, d, R, T, max_position=8192)
    o = WriteTimeRing(R, H, d)
    for w in range(9):
        kb, kf = chunk_pair("k", w, T, H, d, True)
        vb, vf = chunk_pair("v", w, T, H, d, True)
        ring.write(0, to_dev(kb), to_dev(vb))
        o.write(kf, vf)
    qb, qf = chunk_pair("q", 9, T, H, d, True)
    out = ring.attend(0, to_dev(qb)).cpu().numpy()
    rng = np.random.default_rng(7)
    heads = np.array([0, 5, 10, 15])
    rows = np.unique(np.concatenate([rng.choice(T, 60, replace=False), [0, 127, 128, 640, 756]]))
    ref = o.attend(qf, heads=heads, rows=rows)
    assert_attention_close(out[np.ix_(rows, heads)], ref, "production sample")


def test_step_sequence_with_resets_tiny():
    """100 steps of the tiny case: write, 4 attends, resets at 42 and 84."""
    L, R, T, H, d = 2, 96, 32, 2, 64
    ring = kv.KVRing(L, H, d, R, T, max_position=R + 42 * T)
    oracles = [WriteTimeRing(R, H, d) for _ in range(L)]
    for s in range(100):
        if s > 0 and s % 42 == 0:
            ring.rebase()
            for o in oracles:
                o.rebase()
            for l in range(L):
                _check_cache(ring, l, oracles[l])
        for l in range(L):
            kb, kf = chunk_pair("k", s * L + l, T, H, d, True)
            vb, vf = chunk_pair("v", s * L + l, T, H, d, True)
            ring.write(l, to_dev(kb), to_dev(vb))
            oracles[l].write(kf, vf)
            for p in range(4):
                qb, qf = chunk_pair("q", (s * L + l) * 4 + p, T, H, d)
                out = ring.attend(l, to_dev(qb))
                if s % 7 == 0 or s in (41, 42, 43, 84, 85, 99):
                    assert_attention_close(out.cpu().numpy(), oracles[l].attend(qf), f"step {s} layer {l}")
        if s % 10 == 0 or s in (41, 42, 43, 83, 84, 85, 99):
            for l in range(L):
                _check_cache(ring, l, oracles[l])


def test_rebase_many_layers_production_heads():
    """Rebase over several layers at production head shape; bytes bit-exact with the oracle."""
    L, R, T, H, d = 3, 5788, 757, 16, 128
    ring = kv.KVRing(L, H, d, R, T, max_position=R + 42 * T)
    oracles = [WriteTimeRing(R, H, d) for _ in range(L)]
    for w in range(9):
        for l in range(L):
            kb, kf = chunk_pair("k", 10 * w + l, T, H, d, True)
            vb, vf = chunk_pair("v", 10 * w + l, T, H, d, True)
            ring.write(l, to_dev(kb), to_dev(vb))
            oracles[l].write(kf, vf)
    ring.rebase()
    for o in oracles:
        o.rebase()
    for l in range(L):
        fk, fv = _check_cache(ring, l, oracles[l])
        assert fk == 1.0 and fv == 1.0


@pytest.mark.parametrize("R,T,H,d", [(96, 32, 2, 64), (100, 32, 2, 128), (300, 100, 3, 128), (40, 40, 1, 64)])
def test_rewrite_passes_small(R, T, H, d):
    """Four denoise passes per step: one write, then three rewrites of the same chunk."""
    ring = kv.KVRing(1, H, d, R, T, max_position=4096)
    o = WriteTimeRing(R, H, d)
    for w in range(2 * R // T + 2):
        for p in range(4):
            i = 4 * w + p
            kb, kf = chunk_pair("k", 500 + i, T, H, d, p % 2 == 1)
            vb, vf = chunk_pair("v", 500 + i, T, H, d, p % 2 == 1)
            if p == 0:
                ring.write(0, to_dev(kb), to_dev(vb))
                o.write(kf, vf)
            else:
                ring.rewrite(0, to_dev(kb), to_dev(vb))
                o.rewrite(kf, vf)
            fk, fv = _check_cache(ring, 0, o)
            assert fk == 1.0 and fv == 1.0
            qb, qf = chunk_pair("q", 500 + i, T, H, d, True)
            out = ring.attend(0, to_dev(qb)).cpu().numpy()
            assert_attention_close(out, o.attend(qf), f"write {w} pass {p}")


def test_rewrite_after_reset_production_sampled():
    """Production shape: the ring wraps, positions reset, then passes 1..3 rewrite the
    latest chunk at its shifted positions; cache bytes and sampled attention."""
    R, T, H, d = 5788, 757, 16, 128
    ring = kv.KVRing(1, H, d, R, T, max_position=R + 42 * T)
    o = WriteTimeRing(R, H, d)
    for w in range(9):
        kb, kf = chunk_pair("k", 700 + w, T, H, d, True)
        vb, vf = chunk_pair("v", 700 + w, T, H, d, True)
        ring.write(0, to_dev(kb), to_dev(vb))
        o.write(kf, vf)
    ring.rebase()
    assert o.rebase() > 0
    rng = np.random.default_rng(11)
    heads = np.array([0, 7, 15])
    rows = np.unique(np.concatenate([rng.choice(T, 40, replace=False), [0, 127, 128, 756]]))
    for p in range(1, 4):
        kb, kf = chunk_pair("k", 720 + p, T, H, d, True)
        vb, vf = chunk_pair("v", 720 + p, T, H, d, True)
        ring.rewrite(0, to_dev(kb), to_dev(vb))
        o.rewrite(kf, vf)
        qb, qf = chunk_pair("q", 720 + p, T, H, d, True)
        out = ring.attend(0, to_dev(qb)).cpu().numpy()
        assert_attention_close(out[np.ix_(rows, heads)], o.attend(qf, heads=heads, rows=rows), f"pass {p}")
    fk, fv = _check_cache(ring, 0, o)
    assert fk == 1.0 and fv == 1.0


def _check_naive(ring, layer, o, what=""):
    """FP8 cache of a naive-upkeep ring after a refresh against NaiveWindow.cache_codes()."""
    snap = ring.snapshot(layer)
    n = o.count
    k8, v8, _, _ = o.cache_codes()
    _, _, _, _, ka, va = o.chunk_scales()
    assert np.array_equal(snap["pos"][:n].astype(np.int64), o.pos), what
    assert np.array_equal(snap["kamax"][:, :n], ka.T), what
    assert np.array_equal(snap["vamax"][:, :n], va.T), what
    fk = assert_codes_match(snap["k"][:, :n], k8.transpose(1, 0, 2), 0.999, "naive K codes " + what)
    fv = assert_codes_match(snap["v"][:, :n], v8.transpose(1, 0, 2), 0.999, "naive V codes " + what)
    assert fk == 1.0 and fv == 1.0


@pytest.mark.parametrize("R,T,H,d", [(96, 32, 2, 64), (100, 32, 2, 128), (40, 40, 1, 64), (300, 100, 3, 128)])
def test_naive_upkeep_small(R, T, H, d):
    """Naive ring: shift on write, newest rows replaced on rewrite, positions reset;
    each refresh re-rotates and re-quantises the whole window exactly as the oracle."""
    from oracle.schemes import NaiveWindow
    ring = kv.KVRing(1, H, d, R, T, max_position=R + 8 * T, naive_upkeep=True)
    o = NaiveWindow(R, H, d)
    for s in range(2 * R // T + 6):
        if s > 0 and s % 8 == 0:
            ring.rebase()
            o.rebase()
        for p in range(2):
            i = 900 + 2 * s + p
            kb, kf = chunk_pair("k", i, T, H, d, True)
            vb, vf = chunk_pair("v", i, T, H, d, True)
            if p == 0:
                ring.write(0, to_dev(kb), to_dev(vb))
                o.write(kf, vf)
            else:
                ring.rewrite(0, to_dev(kb), to_dev(vb))
                o.rewrite(kf, vf)
            ring.naive_refresh(0)
            _check_naive(ring, 0, o, f"step {s} pass {p}")
            qb, qf = chunk_pair("q", i, T, H, d, True)
            assert_attention_close(ring.attend(0, to_dev(qb)).cpu().numpy(), o.attend(qf), f"step {s} pass {p}")


def test_naive_upkeep_production_sampled():
    """Production shape, naive ring: full window, a reset, refresh, then sampled attention."""
    from oracle.schemes import NaiveWindow
    R, T, H, d = 5788, 757, 16, 128
    ring = kv.KVRing(1, H, d, R, T, max_position=R + 42 * T, naive_upkeep=True)
    o = NaiveWindow(R, H, d)
    for w in range(9):
        kb, kf = chunk_pair("k", 950 + w, T, H, d, True)
        vb, vf = chunk_pair("v", 950 + w, T, H, d, True)
        ring.write(0, to_dev(kb), to_dev(vb))
        o.write(kf, vf)
    ring.rebase()
    assert o.rebase() > 0
    qb, qf = chunk_pair("q", 960, T, H, d, True)
    with pytest.raises(kv.KVRingError) as e:
        ring.attend(0, to_dev(qb))
    assert e.value.code == kv.KVRING_ESTATE
    ring.naive_refresh(0)
    _check_naive(ring, 0, o, "production")
    out = ring.attend(0, to_dev(qb)).cpu().numpy()
    rng = np.random.default_rng(13)
    heads = np.array([1, 8, 14])
    rows = np.unique(np.concatenate([rng.choice(T, 40, replace=False), [0, 128, 756]]))
    ref = o.attend(qf)[np.ix_(rows, heads)]
    assert_attention_close(out[np.ix_(rows, heads)], ref, "naive production")


def _layout_3d(d, S, W):
    ph = d // 6
    return (S, W, d // 2 - 2 * ph, ph)


@pytest.mark.parametrize("R,T,H,d", [(96, 24, 2, 64), (96, 36, 2, 128)])
def test_rope_3d_small(R, T, H, d):
    """3-D video RoPE (frames of 12 tokens, rows of 4): writes through wraps, attention,
    and resets by whole frames that turn only the time band."""
    S, W = 12, 4
    lay = _layout_3d(d, S, W)
    ring = kv.KVRing(1, H, d, R, T, max_position=R + 6 * T, rope_3d=lay)
    o = WriteTimeRing(R, H, d, layout=lay)
    for s in range(14):
        if s > 0 and s % 6 == 0:
            before = ring.snapshot(0)["k"].copy()
            ring.rebase()
            o.rebase()
            fk, fv = _check_cache(ring, 0, o)
            assert fk == 1.0 and fv == 1.0
            after = ring.snapshot(0)["k"]
            assert np.array_equal(after[..., 2 * lay[2]:], before[..., 2 * lay[2]:])
        kb, kf = chunk_pair("k", 1100 + s, T, H, d, True)
        vb, vf = chunk_pair("v", 1100 + s, T, H, d, True)
        ring.write(0, to_dev(kb), to_dev(vb))
        o.write(kf, vf)
        fk, fv = _check_cache(ring, 0, o)
        assert fk == 1.0 and fv == 1.0
        qb, qf = chunk_pair("q", 1100 + s, T, H, d, True)
        assert_attention_close(ring.attend(0, to_dev(qb)).cpu().numpy(), o.attend(qf), f"3-D step {s}")


def test_rope_3d_naive_refresh():
    """Naive ring with 3-D RoPE: every refresh equals the oracle's re-rotation."""
    from oracle.schemes import NaiveWindow
    R, T, H, d, S, W = 96, 24, 2, 128, 12, 4
    lay = _layout_3d(d, S, W)
    ring = kv.KVRing(1, H, d, R, T, max_position=R + 6 * T, naive_upkeep=True, rope_3d=lay)
    o = NaiveWindow(R, H, d, layout=lay)
    for s in range(12):
        if s > 0 and s % 6 == 0:
            ring.rebase()
            o.rebase()
        kb, kf = chunk_pair("k", 1200 + s, T, H, d, True)
        vb, vf = chunk_pair("v", 1200 + s, T, H, d, True)
        ring.write(0, to_dev(kb), to_dev(vb))
        o.write(kf, vf)
        ring.naive_refresh(0)
        _check_naive(ring, 0, o, f"3-D step {s}")


def test_rope_3d_production_frames_sampled():
    """Frames of 11 x 17 = 187 tokens, 4 frames per chunk (748 tokens), a 31-frame ring
    (5,797 slots), 16 heads x 128: fill, reset, then cache bytes and sampled attention."""
    S, W, H, d = 187, 17, 16, 128
    T, R = 4 * S, 31 * S
    lay = _layout_3d(d, S, W)
    ring = kv.KVRing(1, H, d, R, T, max_position=R + 42 * T, rope_3d=lay)
    o = WriteTimeRing(R, H, d, layout=lay)
    for w in range(9):
        kb, kf = chunk_pair("k", 1300 + w, T, H, d, True)
        vb, vf = chunk_pair("v", 1300 + w, T, H, d, True)
        ring.write(0, to_dev(kb), to_dev(vb))
        o.write(kf, vf)
    ring.rebase()
    assert o.rebase() % S == 0
    fk, fv = _check_cache(ring, 0, o)
    assert fk == 1.0 and fv == 1.0
    qb, qf = chunk_pair("q", 1310, T, H, d, True)
    out = ring.attend(0, to_dev(qb)).cpu().numpy()
    rng = np.random.default_rng(17)
    heads = np.array([2, 9, 15])
    rows = np.unique(np.concatenate([rng.choice(T, 40, replace=False), [0, 186, 187, 747]]))
    assert_attention_close(out[np.ix_(rows, heads)], o.attend(qf, heads=heads, rows=rows), "3-D production")


def test_edge_sizes():
    # T = 1, T = R (whole ring in one write), then a write that wraps mid-group
    R, H, d = 40, 1, 64
    ring = kv.KVRing(1, H, d, R, R, max_position=4096)
    o = WriteTimeRing(R, H, d)
    for w, T in enumerate([1, 40, 3, 17, 40, 1, 23]):
        kb, kf = chunk_pair("k", 200 + w, T, H, d, True)
        vb, vf = chunk_pair("v", 200 + w, T, H, d, True)
        ring.write(0, to_dev(kb), to_dev(vb))
        o.write(kf, vf)
        fk, fv = _check_cache(ring, 0, o)
        assert fk == 1.0 and fv == 1.0
        qb, qf = chunk_pair("q", 200 + w, T, H, d)
        assert_attention_close(ring.attend(0, to_dev(qb)).cpu().numpy(), o.attend(qf), f"T={T}")


def test_state_errors_on_device_ring():
    ring = kv.KVRing(1, 2, 64, 96, 32)
    qb, _ = chunk_pair("q", 0, 32, 2, 64)
    with pytest.raises(kv.KVRingError) as e:
        ring.attend(0, to_dev(qb))
    assert e.value.code == kv.KVRING_ESTATE
    kb, _ = chunk_pair("k", 0, 32, 2, 64)
    ring.write(0, to_dev(kb), to_dev(kb))
    qb16, _ = chunk_pair("q", 0, 16, 2, 64)
    with pytest.raises(kv.KVRingError) as e:
        ring.attend(0, to_dev(qb16))
    assert e.value.code == kv.KVRING_ESTATE
    assert ring.check_device() == kv.KVRING_OK
