"""Bounded device waits: a K/V load that never comes makes the attention kernel give up
cleanly, report KVRING_ETIMEOUT through the error word, and leave the ring usable.

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
