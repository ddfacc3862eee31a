"""Argument checks of the allocation-free attention entry point, on the CPU.

Every bad argument must be refused before anything is launched: by the binding
(dtypes, shapes, devices, the error word) and, for what raw pointers still
carry (the RoPE table's row count, the scratch limit, alignment), by the
library itself, which returns KVRING_EINVAL before its first CUDA call.
"""
import ctypes

import pytest
import torch

from kv_cache_gb300 import kvring as kv
from tests._lib import ensure_built

H, d, Rp, n_q, q_pos0 = 2, 64, 128, 32, 96


def _args(**over):
    a = dict(k8=torch.zeros((H, Rp, d), dtype=torch.uint8), vt8=torch.zeros((H, d, Rp), dtype=torch.uint8),
             kamax=torch.zeros((H, Rp)), vamax=torch.zeros((H, Rp)), rope=torch.zeros((q_pos0 + n_q, d // 2, 2)),
             q_pos0=q_pos0, q=torch.zeros((n_q, H, d), dtype=torch.bfloat16), out=torch.zeros((n_q, H, d)),
             count=100, err=torch.zeros(4, dtype=torch.int32))
    a.update(over)
    return a


def test_valid_arguments_pass():
    assert kv.noalloc_arg_error(**_args(), device="cpu") is None
    assert kv.noalloc_arg_error(**_args(err=None), device="cpu") is None


@pytest.mark.parametrize("over,needle", [
    (dict(rope=torch.zeros((q_pos0 + n_q - 1, d // 2, 2))), "rope has"),      # one row short
    (dict(q_pos0=-1), "rope has"),
    (dict(rope=torch.zeros((200, d // 2, 2), dtype=torch.float64)), "rope must be"),
    (dict(rope=torch.zeros((200, d, 2))), "rope must be"),
    (dict(k8=torch.zeros((H, Rp, d), dtype=torch.int8)), "k8 must be torch.uint8"),
    (dict(vt8=torch.zeros((H, Rp, d), dtype=torch.uint8)), "vt8 must have shape"),
    (dict(kamax=torch.zeros((H, Rp), dtype=torch.float16)), "kamax must be torch.float32"),
    (dict(vamax=torch.zeros((H, Rp + 1))), "vamax must have shape"),
    (dict(q=torch.zeros((n_q, H, d), dtype=torch.float16)), "q must be torch.bfloat16"),
    (dict(out=torch.zeros((n_q, H, d), dtype=torch.bfloat16)), "out must be torch.float32"),
    (dict(out=torch.zeros((n_q, H, 2 * d))[..., ::2]), "out must be contiguous"),
    (dict(err=torch.zeros(3, dtype=torch.int32)), "err must be"),
    (dict(err=torch.zeros(4, dtype=torch.int64)), "err must be"),
    (dict(count=0), "count must be"),
    (dict(count=Rp + 1), "count must be"),
])
def test_bad_argument_is_named(over, needle):
    msg = kv.noalloc_arg_error(**_args(**over), device="cpu")
    assert msg is not None and needle in msg, msg


def test_tensors_on_another_device_are_refused():
    # every tensor is on the CPU while the call would run on a CUDA device
    msg = kv.noalloc_arg_error(**_args(), device="cuda:0")
    assert msg is not None and "the call runs on cuda:0" in msg


def test_binding_raises_before_the_library_is_called():
    with pytest.raises(ValueError):
        kv.kvring_attend_noalloc(**{k: v for k, v in _args(count=0).items()})


def _raw_call(lib, rope_rows, q_pos0_, n_q_, heads=H, slots=Rp, count=100, align=256):
    p = ctypes.c_void_p(1 << 20)                 # never dereferenced: the checks come first
    odd = ctypes.c_void_p((1 << 20) + 8) if align != 256 else p
    return lib.kvring_attend_noalloc(p, p, p, p, p, rope_rows, q_pos0_, odd, n_q_, heads, d, slots, count,
                                     p, None, None)


def test_library_refuses_before_any_cuda_call():
    lib = ensure_built()
    rc = _raw_call(lib, rope_rows=q_pos0 + n_q - 1, q_pos0_=q_pos0, n_q_=n_q)
    assert rc == kv.KVRING_EINVAL and "rope has" in kv.kvring_last_error(None)
    rc = _raw_call(lib, rope_rows=10, q_pos0_=2 ** 40, n_q_=n_q)
    assert rc == kv.KVRING_EINVAL and "rope has" in kv.kvring_last_error(None)
    rc = _raw_call(lib, rope_rows=10 ** 6, q_pos0_=0, n_q_=300, heads=64)        # 64 x 512 rows > 16,384
    assert rc == kv.KVRING_EINVAL and "scratch" in kv.kvring_last_error(None)
    rc = _raw_call(lib, rope_rows=10 ** 6, q_pos0_=0, n_q_=n_q, align=8)         # q not 16-byte aligned
    assert rc == kv.KVRING_EINVAL and "aligned" in kv.kvring_last_error(None)
    rc = _raw_call(lib, rope_rows=10 ** 6, q_pos0_=0, n_q_=n_q, count=0)
    assert rc == kv.KVRING_EINVAL
