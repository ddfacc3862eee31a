"""The allocation-free attention entry point against the ring's own attention call.

kvring_attend_noalloc is for callers that may not allocate device memory because
their own arena owns all of it: they hold the FP8 cache themselves and the call
uses only a fixed scratch array inside the library.  Here a ring is filled
through the normal API, its cache is copied into caller-owned tensors in the
documented layouts, and two calls in a row of the allocation-free entry point
must agree with kvring_attend on the same queries within the attention
tolerance of the parity tests.  This file is collected last on purpose.
"""
import numpy as np
import pytest
import torch

from kv_cache_gb300 import kvring as kv
from oracle import rope as oracle_rope
from tests._lib import ensure_built
from tests.gpu_util import assert_attention_close, chunk_pair, to_dev

pytestmark = pytest.mark.gpu


@pytest.fixture(scope="module", autouse=True)
def _lib():
    ensure_built()


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


@pytest.mark.parametrize("R,T,H,d,writes", [(5788, 757, 16, 128, 9), (96, 32, 2, 64, 5), (300, 130, 3, 128, 2)])
def test_noalloc_matches_ring_attention_twice(R, T, H, d, writes):
    ring = kv.KVRing(1, H, d, R, T, max_position=8192)
    for w in range(writes):
        kb, _ = chunk_pair("k", 700 + w, T, H, d, True)
        vb, _ = chunk_pair("v", 700 + w, T, H, d, True)
        ring.write(0, to_dev(kb), to_dev(vb))
    st = ring.state(0)
    k8, vt8, ka, va, rope = _caller_owned_cache(ring, R, H, d, st["next_pos"] + 1)
    err = torch.zeros(4, dtype=torch.int32, device="cuda")
    for call in range(2):
        qb, _ = chunk_pair("q", 800 + call, T, H, d, True)
        q = to_dev(qb)
        ref = ring.attend(0, q).cpu().numpy()
        out = torch.full((T, H, d), float("nan"), dtype=torch.float32, device="cuda")
        kv.kvring_attend_noalloc(k8, vt8, ka, va, rope, st["last_write_pos"], q, out, st["count"], err=err)
        torch.cuda.synchronize()
        assert int(err[0]) == 0
        assert_attention_close(out.cpu().numpy(), ref, f"call {call}")


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
