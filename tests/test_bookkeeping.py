"""Host ring bookkeeping of the C library (host-only rings) against the oracle, bit-exact,
plus argument and state checks.  No GPU needed."""
import numpy as np
import pytest

from kv_cache_gb300 import kvring as kv
from oracle.schemes import WriteTimeRing
from tests._lib import ensure_built


@pytest.fixture(scope="module", autouse=True)
def _lib():
    ensure_built()


def _ring(L, H, d, R, T, max_position=0):
    return kv.KVRing(L, H, d, R, T, max_position=max_position, host_only=True)


def _compare(ring, layer, o: WriteTimeRing):
    st = ring.state(layer)
    assert st["head"] == o.head
    assert st["count"] == o.count
    assert st["next_pos"] == o.next_pos
    assert st["writes"] == o.writes
    assert st["last_write_pos"] == o.last_pos
    assert st["last_write_tokens"] == o.last_n
    snap = ring.snapshot(layer, cache=False)
    assert np.array_equal(snap["pos"].astype(np.int64), o.pos)
    assert np.array_equal(snap["chunk"].astype(np.int64), o.chunk)


@pytest.mark.parametrize("R,T,steps", [(96, 32, 100), (100, 32, 100), (5788, 757, 130), (7, 7, 50), (10, 3, 60)])
def test_schedule_matches_oracle(R, T, steps):
    ring = _ring(2, 1, 64, R, T, max_position=R + 42 * T)
    o = WriteTimeRing(R, 1, 2)
    for s in range(steps):
        if s > 0 and s % 42 == 0:
            ring.rebase()
            o.rebase()
            _compare(ring, 0, o)
        ring.write(0, None, None, n_tokens=T)
        ring.write(1, None, None, n_tokens=T)
        o.write(np.zeros((T, 1, 2), np.float32), np.zeros((T, 1, 2), np.float32))
        _compare(ring, 0, o)
        _compare(ring, 1, o)
    assert ring.state(0)["resets"] == o.resets


def test_variable_chunk_sizes_and_per_layer_delta():
    R = 50
    ring = _ring(2, 1, 64, R, 20, max_position=1000)
    oracles = [WriteTimeRing(R, 1, 2), WriteTimeRing(R, 1, 2)]
    sizes = [[5, 20, 1, 17, 13, 20, 2, 9], [20, 20, 20, 3, 7, 11, 19, 1]]
    for w in range(len(sizes[0])):
        for l in range(2):
            n = sizes[l][w]
            ring.write(l, None, None, n_tokens=n)
            oracles[l].write(np.zeros((n, 1, 2), np.float32), np.zeros((n, 1, 2), np.float32))
    ring.rebase()
    for l in range(2):
        oracles[l].rebase()
        _compare(ring, l, oracles[l])


def test_errors_leave_state_unchanged():
    ring = _ring(1, 2, 64, 96, 32, max_position=200)
    before = ring.state(0)
    with pytest.raises(kv.KVRingError) as e:
        kv.kvring_write(ring.handle, 0, None, None, 33, 2, 64)
    assert e.value.code == kv.KVRING_EINVAL and "max_tokens_per_write" in e.value.message
    with pytest.raises(kv.KVRingError) as e:
        kv.kvring_write(ring.handle, 1, None, None, 8, 2, 64)
    assert e.value.code == kv.KVRING_EINVAL and "layer" in e.value.message
    with pytest.raises(kv.KVRingError) as e:
        kv.kvring_write(ring.handle, -1, None, None, 8, 2, 64)
    assert e.value.code == kv.KVRING_EINVAL
    assert ring.state(0) == before
    for _ in range(6):
        ring.write(0, None, None, n_tokens=32)       # next_pos = 192
    with pytest.raises(kv.KVRingError) as e:
        ring.write(0, None, None, n_tokens=9)          # 201 > 200
    assert e.value.code == kv.KVRING_ESTATE and "rebase" in e.value.message
    st = ring.state(0)
    ring.write(0, None, None, n_tokens=8)              # 200 == max_position is fine
    ring.rebase()
    assert ring.state(0)["next_pos"] == 96 and st["writes"] + 1 == ring.state(0)["writes"]
    ring.write(0, None, None, n_tokens=0)              # empty write is a no-op
    assert ring.state(0)["writes"] == st["writes"] + 1


def test_attend_needs_a_device_ring():
    ring = _ring(1, 1, 64, 16, 8)
    ring.write(0, None, None, n_tokens=8)
    lib = kv.load()
    rc = lib.kvring_attend(ring.handle, 0, None, 8, None, None)
    assert rc == kv.KVRING_EINVAL
    assert "host-only" in kv.kvring_last_error(ring.handle)


@pytest.mark.parametrize("field,value", [("num_layers", 0), ("num_layers", 257), ("num_heads", 0),
                                         ("head_dim", 96), ("capacity", 0), ("max_tokens_per_write", 0),
                                         ("max_tokens_per_write", 97), ("max_position", -1), ("flags", 8)])
def test_create_rejects_bad_config(field, value):
    cfg = kv.kvring_config(1, 2, 64, 96, 32, 0, 10000.0, kv.KVRING_FLAG_HOST_ONLY)
    setattr(cfg, field, value)
    with pytest.raises(kv.KVRingError) as e:
        kv.kvring_create(cfg)
    assert e.value.code == kv.KVRING_EINVAL
    assert kv.kvring_last_error(None)


def test_null_handles_are_rejected():
    lib = kv.load()
    assert lib.kvring_write(None, 0, None, None, 1, None) == kv.KVRING_EINVAL
    assert lib.kvring_rebase(None, None) == kv.KVRING_EINVAL
    assert lib.kvring_destroy(None) == kv.KVRING_OK
    assert lib.kvring_get_state(None, 0, None) == kv.KVRING_EINVAL


@pytest.mark.parametrize("R,T", [(96, 32), (100, 32), (5788, 757), (7, 7)])
def test_rewrite_passes_leave_the_schedule_unchanged(R, T):
    # one write and three rewrites per step, resets every 42 steps: the state
    # after each call equals the oracle's
    ring = _ring(1, 1, 64, R, T, max_position=R + 42 * T)
    o = WriteTimeRing(R, 1, 2)
    z = np.zeros((T, 1, 2), np.float32)
    for s in range(90):
        if s > 0 and s % 42 == 0:
            ring.rebase()
            o.rebase()
        ring.write(0, None, None, n_tokens=T)
        o.write(z, z)
        for _ in range(3):
            ring.rewrite(0, None, None, n_tokens=T)
            o.rewrite(z, z)
            _compare(ring, 0, o)


def test_rewrite_errors_leave_state_unchanged():
    ring = _ring(1, 2, 64, 96, 32, max_position=200)
    lib = kv.load()
    with pytest.raises(kv.KVRingError) as e:
        ring.rewrite(0, None, None, n_tokens=32)
    assert e.value.code == kv.KVRING_ESTATE and "before any write" in e.value.message
    ring.write(0, None, None, n_tokens=20)
    before = ring.state(0)
    for n in (19, 21, 0):
        with pytest.raises(kv.KVRingError) as e:
            ring.rewrite(0, None, None, n_tokens=n)
        assert e.value.code == kv.KVRING_ESTATE and "n_tokens" in e.value.message
    assert lib.kvring_write_ex(ring.handle, 0, None, None, 20, 0x2, None) == kv.KVRING_EINVAL
    assert "flag" in kv.kvring_last_error(ring.handle)
    assert ring.state(0) == before
    for _ in range(8):                          # next_pos = 180: a rewrite never checks max_position
        ring.write(0, None, None, n_tokens=20)
    ring.rewrite(0, None, None, n_tokens=20)
    assert ring.state(0)["next_pos"] == 180 and ring.state(0)["last_write_pos"] == 160
    assert lib.kvring_write_ex(ring.handle, 0, None, None, 21, 0, None) == kv.KVRING_ESTATE   # 201 > 200
    assert lib.kvring_write_ex(None, 0, None, None, 1, 1, None) == kv.KVRING_EINVAL


def _compare_naive(ring, layer, o):
    st = ring.state(layer)
    assert (st["count"], st["next_pos"], st["writes"]) == (o.count, o.next_pos, o.writes)
    assert (st["last_write_pos"], st["last_write_tokens"]) == (o.last_pos, o.last_n)
    snap = ring.snapshot(layer, cache=False)
    assert np.array_equal(snap["pos"][:o.count].astype(np.int64), o.pos)
    assert np.array_equal(snap["chunk"][:o.count].astype(np.int64), o.chunk)


@pytest.mark.parametrize("R,T", [(96, 32), (100, 32), (5788, 757), (7, 3)])
def test_naive_ring_rows_match_the_shifted_window(R, T):
    # a naive-upkeep ring keeps its rows in logical order: positions and chunk ids
    # equal the oracle's shifted window through writes, rewrites and resets
    from oracle.schemes import NaiveWindow
    ring = kv.KVRing(1, 1, 64, R, T, max_position=R + 42 * T, host_only=True, naive_upkeep=True)
    o = NaiveWindow(R, 1, 2)
    z = np.zeros((T, 1, 2), np.float32)
    for s in range(90):
        if s > 0 and s % 42 == 0:
            ring.rebase()
            o.rebase()
            _compare_naive(ring, 0, o)
        ring.write(0, None, None, n_tokens=T)
        o.write(z, z)
        _compare_naive(ring, 0, o)
        if s % 5 == 0:
            ring.rewrite(0, None, None, n_tokens=T)
            o.rewrite(z, z)
            _compare_naive(ring, 0, o)
        ring.naive_refresh(0)


def test_naive_refresh_errors():
    ring = kv.KVRing(1, 1, 64, 16, 8, host_only=True, naive_upkeep=True)
    with pytest.raises(kv.KVRingError) as e:
        ring.naive_refresh(0)
    assert e.value.code == kv.KVRING_ESTATE
    with pytest.raises(kv.KVRingError) as e:
        ring.naive_refresh(1)
    assert e.value.code == kv.KVRING_EINVAL
    plain = kv.KVRing(1, 1, 64, 16, 8, host_only=True)
    plain.write(0, None, None, n_tokens=8)
    with pytest.raises(kv.KVRingError) as e:
        plain.naive_refresh(0)
    assert e.value.code == kv.KVRING_EINVAL and "naive" in e.value.message


@pytest.mark.parametrize("S,W,pt,ph,R", [(0, 1, 0, 0, 96), (12, 5, 0, 0, 96), (12, 4, 0, 0, 100),
                                          (12, 4, 16, 16, 96), (12, 4, 0, 5, 96), (12, 4, 31, 1, 96)])
def test_create_rejects_bad_3d_layout(S, W, pt, ph, R):
    cfg = kv.kvring_config(1, 2, 64, R, 24, 0, 10000.0, kv.KVRING_FLAG_HOST_ONLY | kv.KVRING_FLAG_ROPE_3D,
                           S, W, pt, ph)
    with pytest.raises(kv.KVRingError) as e:
        kv.kvring_create(cfg)
    assert e.value.code == kv.KVRING_EINVAL and "3-D" in e.value.message


def test_3d_ring_writes_whole_frames_and_resets_by_frames():
    from oracle.schemes import WriteTimeRing
    S, R, T = 12, 96, 24
    ring = kv.KVRing(1, 1, 64, R, T, max_position=R + 42 * T, host_only=True, rope_3d=(S, 4, 0, 0))
    with pytest.raises(kv.KVRingError) as e:
        ring.write(0, None, None, n_tokens=13)
    assert e.value.code == kv.KVRING_EINVAL and "frames" in e.value.message
    o = WriteTimeRing(R, 1, 2)
    z = np.zeros((T, 1, 2), np.float32)
    for s in range(60):
        if s > 0 and s % 42 == 0:
            ring.rebase()
            assert o.rebase() % S == 0
        n = T if s % 3 else S
        ring.write(0, None, None, n_tokens=n)
        o.write(z[:n], z[:n])
        _compare(ring, 0, o)
