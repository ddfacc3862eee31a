"""The allocation-free attention entry point against the oracle and the ring's own call.

kvring_attend_noalloc is for callers that may not allocate device memory because
their own arena owns all of it: they hold the FP8 cache themselves and the call
prepares the queries inside the attention kernel, keeping nothing between calls.
Here a ring is filled through the normal API (and the same chunks go into the
CPU oracle), its cache is copied into caller-owned tensors in the documented
layouts, and two calls in a row of the allocation-free entry point must agree,
within the attention tolerance of the parity tests, with the oracle's float64
attention over the same cache and queries, and with kvring_attend.  A large call
is followed by a much smaller one without an error word.  This file is collected
last on purpose.
"""
import numpy as np
import pytest
import torch

from kv_cache_gb300 import kvring as kv
from oracle import rope as oracle_rope
from oracle.schemes import WriteTimeRing
from tests._lib import ensure_built
from tests.gpu_util import assert_attention_close, chunk_pair, to_dev

pytestmark = pytest.mark.gpu


@pytest.fixture(scope="module", autouse=True)
def _lib():
    ensure_built()


def _filled(R, T, H, d, writes, seed):
    """A device ring and the oracle ring after the same writes."""
    ring = kv.KVRing(1, H, d, R, T, max_position=8192)
    o = WriteTimeRing(R, H, d)
    for w in range(writes):
        kb, kf = chunk_pair("k", seed + w, T, H, d, True)
        vb, vf = chunk_pair("v", seed + w, T, H, d, True)
        ring.write(0, to_dev(kb), to_dev(vb))
        o.write(kf, vf)
    return ring, o


def _caller_owned_cache(ring, R, H, d, npos):
    """Copy layer 0 of a ring into CUDA tensors in the entry point's layouts."""
    snap = ring.snapshot(0)
    Rp = (R + 127) // 128 * 128
    k8 = np.zeros((H, Rp, d), np.uint8)
    k8[:, :R] = snap["k"]
    vt8 = np.zeros((H, d, Rp), np.uint8)
    vt8[:, :, :R] = snap["v"].transpose(0, 2, 1)
    ka = np.zeros((H, Rp), np.float32)
    ka[:, :R] = snap["kamax"]
    va = np.zeros((H, Rp), np.float32)
    va[:, :R] = snap["vamax"]
    c, s = oracle_rope.angle_table(np.arange(npos), d)
    rope = np.stack([c, s], axis=-1).astype(np.float32)          # [npos][d/2][2]
    dev = lambda a: torch.from_numpy(np.ascontiguousarray(a)).cuda()
    return dev(k8), dev(vt8), dev(ka), dev(va), dev(rope)


def _noalloc(cache, st, q, err):
    k8, vt8, ka, va, rope = cache
    out = torch.full(tuple(q.shape), float("nan"), dtype=torch.float32, device="cuda")
    kv.kvring_attend_noalloc(k8, vt8, ka, va, rope, st["last_write_pos"], q, out, st["count"], err=err)
    torch.cuda.synchronize()
    return out.cpu().numpy()


@pytest.mark.parametrize("R,T,H,d,writes", [(5788, 757, 16, 128, 9), (96, 32, 2, 64, 5), (300, 130, 3, 128, 2)])
def test_noalloc_matches_oracle_and_ring_attention_twice(R, T, H, d, writes):
    ring, o = _filled(R, T, H, d, writes, 700)
    st = ring.state(0)
    cache = _caller_owned_cache(ring, R, H, d, st["next_pos"] + 1)
    err = torch.zeros(4, dtype=torch.int32, device="cuda")
    rng = np.random.default_rng(5)
    heads = np.arange(H) if H <= 4 else np.array([0, 5, 10, 15])
    rows = np.arange(T) if T <= 200 else np.unique(np.concatenate([rng.choice(T, 60, replace=False), [0, 255, 256, T - 1]]))
    for call in range(2):
        qb, qf = chunk_pair("q", 800 + call, T, H, d, True)
        q = to_dev(qb)
        out = _noalloc(cache, st, q, err)
        assert int(err[0]) == 0
        assert_attention_close(out[np.ix_(rows, heads)], o.attend(qf, heads=heads, rows=rows), f"call {call} vs oracle")
        assert_attention_close(out, ring.attend(0, q).cpu().numpy(), f"call {call} vs kvring_attend")
    ring.close()


def test_noalloc_small_call_after_a_large_call_without_error_word():
    # 32 heads x 512 queries, then 2 heads x 32 queries, both with err=None (the
    # library's own error word)
    big_ring, big_o = _filled(1024, 512, 32, 64, 2, 900)
    big_st = big_ring.state(0)
    big_cache = _caller_owned_cache(big_ring, 1024, 32, 64, big_st["next_pos"] + 1)
    small_ring, small_o = _filled(96, 32, 2, 64, 5, 950)
    small_st = small_ring.state(0)
    small_cache = _caller_owned_cache(small_ring, 96, 2, 64, small_st["next_pos"] + 1)
    qb_big, qf_big = chunk_pair("q", 910, 512, 32, 64, True)
    qb_small, qf_small = chunk_pair("q", 960, 32, 2, 64, True)
    for _ in range(2):
        out_big = _noalloc(big_cache, big_st, to_dev(qb_big), None)
        heads, rows = np.array([0, 13, 31]), np.array([0, 1, 127, 128, 300, 511])
        assert_attention_close(out_big[np.ix_(rows, heads)], big_o.attend(qf_big, heads=heads, rows=rows), "large call")
        out_small = _noalloc(small_cache, small_st, to_dev(qb_small), None)
        assert_attention_close(out_small, small_o.attend(qf_small), "small call after a large one")
        assert_attention_close(out_small, small_ring.attend(0, to_dev(qb_small)).cpu().numpy(), "vs kvring_attend")
    big_ring.close()
    small_ring.close()


def test_noalloc_64_heads_300_queries():
    # 64 heads x 300 queries (padded: 64 x 512 query rows), d = 64
    R, T, H, d = 512, 300, 64, 64
    ring, o = _filled(R, T, H, d, 2, 990)
    st = ring.state(0)
    cache = _caller_owned_cache(ring, R, H, d, st["next_pos"] + 1)
    qb, qf = chunk_pair("q", 991, T, H, d, True)
    err = torch.zeros(4, dtype=torch.int32, device="cuda")
    out = _noalloc(cache, st, to_dev(qb), err)
    assert int(err[0]) == 0
    heads, rows = np.array([0, 31, 63]), np.array([0, 1, 127, 128, 255, 256, 299])
    assert_attention_close(out[np.ix_(rows, heads)], o.attend(qf, heads=heads, rows=rows), "64 heads vs oracle")
    assert_attention_close(out, ring.attend(0, to_dev(qb)).cpu().numpy(), "64 heads vs kvring_attend")
    ring.close()
