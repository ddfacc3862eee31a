"""The allocation-free attention entry point against the oracle and the ring's own call.

kvring_attend_noalloc is for callers that may not allocate device memory because
their own arena owns all of it: they hold the FP8 cache themselves and the call
uses only a fixed scratch array inside the library.  Here a ring is filled
through the normal API (and the same chunks go into the CPU oracle), its cache
is copied into caller-owned tensors in the documented layouts, and two calls in
a row of the allocation-free entry point must agree, within the attention
tolerance of the parity tests, with the oracle's float64 attention over the
same cache and queries, and with kvring_attend.  A call that fills the whole
scratch is followed by a much smaller one without an error word, so the second
runs on scratch left behind by the first.  This file is collected last on purpose.
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


def test_noalloc_small_call_after_a_full_scratch_call_without_error_word():
    # 32 heads x 512 queries fill the 16,384 scratch rows; then 2 heads x 32 queries
    # with err=None (the library's own error word) read only rows they wrote
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
        assert_attention_close(out_big[np.ix_(rows, heads)], big_o.attend(qf_big, heads=heads, rows=rows), "full scratch")
        out_small = _noalloc(small_cache, small_st, to_dev(qb_small), None)
        assert_attention_close(out_small, small_o.attend(qf_small), "small call after a full one")
        assert_attention_close(out_small, small_ring.attend(0, to_dev(qb_small)).cpu().numpy(), "vs kvring_attend")
    big_ring.close()
    small_ring.close()


def test_noalloc_rejects_sizes_beyond_its_scratch():
    H, d, Rp, n = 64, 128, 256, 300          # 64 heads x 512 padded rows > 16,384
    k8 = torch.zeros((H, Rp, d), dtype=torch.uint8, device="cuda")
    vt8 = torch.zeros((H, d, Rp), dtype=torch.uint8, device="cuda")
    ka = torch.zeros((H, Rp), dtype=torch.float32, device="cuda")
    rope = torch.zeros((n, d // 2, 2), dtype=torch.float32, device="cuda")
    q = torch.zeros((n, H, d), dtype=torch.bfloat16, device="cuda")
    out = torch.zeros((n, H, d), dtype=torch.float32, device="cuda")
    with pytest.raises(kv.KVRingError) as e:
        kv.kvring_attend_noalloc(k8, vt8, ka, ka, rope, 0, q, out, 128)
    assert e.value.code == kv.KVRING_EINVAL and "scratch" in e.value.message
