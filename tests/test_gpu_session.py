"""A long session at the unsharded width: 64 heads x 128, 1,000 steps, resets every 42.

The cache must not drift: at steps 1, 42, 43, 500 and 999 the FP8 bytes of both
blocks equal the oracle's and attention of 4 heads x 64 query rows stays within
tolerance.  The oracle does not replay 1,000 steps at 64 heads: the ring holds
the newest 7 chunks and part of an eighth (5,788 = 7 x 757 + 489), and a reset
inside the last ten steps only turns chunks written inside them, so an oracle
ring whose bookkeeping is taken from a bookkeeping-only oracle ring (1 head,
d = 2, every step) and which replays the last ten steps with data holds the
same cache.
"""
import copy
from collections import deque

import numpy as np
import pytest

from kv_cache_gb300 import kvring as kv
from kv_cache_gb300 import synthetic
from oracle.schemes import WriteTimeRing
from tests._lib import ensure_built
from tests.gpu_util import assert_attention_close, assert_codes_match

pytestmark = pytest.mark.gpu

L, H, d, R, T, RE, STEPS, REPLAY = 2, 64, 128, 5788, 757, 42, 1000, 10
CHECKS = (1, 42, 43, 500, 999)


@pytest.fixture(scope="module", autouse=True)
def _lib():
    ensure_built()


def _bookkeeping(dst: WriteTimeRing, src: WriteTimeRing):
    for f in ("head", "count", "next_pos", "writes", "resets", "last_pos", "last_n"):
        setattr(dst, f, getattr(src, f))
    dst.pos = src.pos.copy()
    dst.chunk = src.chunk.copy()


def test_session_64_heads_no_drift():
    import torch
    pool_bits = {r: [synthetic.chunk(r, i, T, H, d, outliers=True) for i in range(synthetic.POOL)] for r in "kvq"}
    pool_dev = {r: [torch.from_numpy(b.view(np.int16)).view(torch.bfloat16).cuda() for b in pool_bits[r]]
                for r in pool_bits}
    f32 = synthetic.bf16_to_f32
    ring = kv.KVRing(L, H, d, R, T, max_position=R + RE * T)
    tiny = WriteTimeRing(R, 1, 2)
    z = np.zeros((T, 1, 2), np.float32)
    before = deque(maxlen=REPLAY)      # the bookkeeping ring before each of the last REPLAY steps
    out = torch.empty((T, H, d), dtype=torch.float32, device="cuda")
    rng = np.random.default_rng(21)
    heads = np.array([0, 21, 42, 63])
    rows = np.unique(np.concatenate([rng.choice(T, 60, replace=False), [0, 255, 256, 756]]))
    for s in range(STEPS):
        before.append(copy.deepcopy(tiny))
        if s > 0 and s % RE == 0:
            ring.rebase()
            tiny.rebase()
        for l in range(L):
            i = synthetic.pool_index(s, l, 4, L)
            ring.write(l, pool_dev["k"][i], pool_dev["v"][i])
        tiny.write(z, z)
        for l in range(L):
            for p in range(4):
                ring.attend(l, pool_dev["q"][synthetic.pool_index(s, l, p, L)], out)
        if s not in CHECKS:
            continue
        assert ring.check_device() == kv.KVRING_OK
        first = s - len(before) + 1
        for l in range(L):
            o = WriteTimeRing(R, H, d)
            _bookkeeping(o, before[0])
            for t in range(first, s + 1):
                if t > 0 and t % RE == 0:
                    o.rebase()
                i = synthetic.pool_index(t, l, 4, L)
                o.write(f32(pool_bits["k"][i]), f32(pool_bits["v"][i]))
            st = ring.state(l)
            assert (st["head"], st["count"], st["next_pos"], st["writes"]) == (o.head, o.count, o.next_pos, o.writes)
            snap = ring.snapshot(l)
            valid = o.pos >= 0
            assert np.array_equal(snap["pos"].astype(np.int64), o.pos)
            assert np.array_equal(snap["kamax"][:, valid], o.kamax[:, valid])
            fk = assert_codes_match(snap["k"][:, valid], o.k8[:, valid], 0.999, f"K step {s} block {l}")
            fv = assert_codes_match(snap["v"][:, valid], o.v8[:, valid], 0.999, f"V step {s} block {l}")
            assert fk == 1.0 and fv == 1.0, f"step {s} block {l}"
            # attention of the step's last pass, sampled
            qi = synthetic.pool_index(s, l, 3, L)
            ring.attend(l, pool_dev["q"][qi], out)
            ref = o.attend(f32(pool_bits["q"][qi]), heads=heads, rows=rows)
            assert_attention_close(out.cpu().numpy()[np.ix_(rows, heads)], ref, f"step {s} block {l}")
