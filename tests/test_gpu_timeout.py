"""Bounded device waits: a K/V load that never comes makes the attention kernel give up
cleanly, report KVRING_ETIMEOUT through the error word, and leave the ring usable;
a chunk's rows that never come do the same in the write kernel.

The missing load is a testing aid of the library (kvring_debug_fault): the producer
warp leaves one tile's TMA copy out, so its consumers' waits run out after the short
limit given here.  No fault, trap or unbounded wait is involved.
"""
import numpy as np
import pytest

from kv_cache_gb300 import kvring as kv
from oracle.schemes import WriteTimeRing
from tests._lib import ensure_built
from tests.gpu_util import assert_attention_close, chunk_pair, to_dev

pytestmark = pytest.mark.gpu


@pytest.fixture(scope="module", autouse=True)
def _lib():
    ensure_built()


@pytest.mark.parametrize("R,T,H,d,skip", [(1000, 256, 2, 128, 1), (96, 32, 2, 64, 0)])
def test_missing_load_times_out_and_ring_recovers(R, T, H, d, skip):
    ring = kv.KVRing(1, H, d, R, T, max_position=8192)
    o = WriteTimeRing(R, H, d)
    for w in range(R // T + 1):
        kb, kf = chunk_pair("k", 300 + w, T, H, d, True)
        vb, vf = chunk_pair("v", 300 + w, T, H, d, True)
        ring.write(0, to_dev(kb), to_dev(vb))
        o.write(kf, vf)
    qb, qf = chunk_pair("q", 300, T, H, d, True)
    kv.kvring_debug_fault(ring.handle, skip, 20_000_000)       # 20 ms limit, tile `skip` never loaded
    ring.attend(0, to_dev(qb))
    assert ring.check_device() == kv.KVRING_ETIMEOUT
    msg = kv.kvring_last_error(ring.handle)
    assert "timed out" in msg and "attention" in msg
    # the fault applies to one call only; the cache was not touched
    assert ring.check_device() == kv.KVRING_OK
    for _ in range(2):
        out = ring.attend(0, to_dev(qb)).cpu().numpy()
        assert ring.check_device() == kv.KVRING_OK
        assert_attention_close(out, o.attend(qf), "after time-out")


@pytest.mark.parametrize("R,T,H,d,group", [(1000, 256, 2, 128, 3), (96, 32, 2, 64, 0)])
def test_missing_write_rows_time_out_and_ring_recovers(R, T, H, d, group):
    """The write kernel's bounded waits (kvring_debug_fault_write): one ring group's
    TMA copy is left out, the CTA waiting for it gives up after the short limit and
    reports KVRING_ETIMEOUT (kernel: write), its cluster still finishes; the same
    chunk written again over itself is bit-exact with the oracle."""
    ring = kv.KVRing(1, H, d, R, T, max_position=8192)
    o = WriteTimeRing(R, H, d)
    for w in range(R // T + 1):
        kb, kf = chunk_pair("k", 400 + w, T, H, d, True)
        vb, vf = chunk_pair("v", 400 + w, T, H, d, True)
        ring.write(0, to_dev(kb), to_dev(vb))
        o.write(kf, vf)
    assert ring.check_device() == kv.KVRING_OK
    head = ring.state(0)["head"]
    g = (head // 16 + group) % (-(-R // 16))             # a group the next chunk touches
    kb, kf = chunk_pair("k", 450, T, H, d, True)
    vb, vf = chunk_pair("v", 450, T, H, d, True)
    kdev, vdev = to_dev(kb), to_dev(vb)
    kv.kvring_debug_fault_write(ring.handle, g, 20_000_000)   # 20 ms limit, group g's rows never loaded
    ring.write(0, kdev, vdev)
    o.write(kf, vf)
    assert ring.check_device() == kv.KVRING_ETIMEOUT
    msg = kv.kvring_last_error(ring.handle)
    assert "timed out" in msg and "write" in msg
    assert ring.check_device() == kv.KVRING_OK            # the fault applied to one call only
    ring.rewrite(0, kdev, vdev)                           # the same chunk over itself
    assert ring.check_device() == kv.KVRING_OK
    snap = ring.snapshot(0)
    valid = o.pos >= 0
    assert np.array_equal(snap["kamax"][:, valid], o.kamax[:, valid])
    assert np.array_equal(snap["vamax"][:, valid], o.vamax[:, valid])
    assert np.array_equal(snap["k"][:, valid], o.k8[:, valid])
    assert np.array_equal(snap["v"][:, valid], o.v8[:, valid])
    qb, qf = chunk_pair("q", 450, T, H, d, True)
    assert_attention_close(ring.attend(0, to_dev(qb)).cpu().numpy(), o.attend(qf), "after the write's time-out")
