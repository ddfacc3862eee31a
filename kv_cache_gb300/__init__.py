"""GB300-native write-time KV cache for streaming video DiT attention.

The compute path lives in ``libkvring.so`` (C ABI in ``include/kvring.h``,
kernels in ``csrc/``); ``kvring`` is the ctypes binding with the same names.
Build with ``python -m kv_cache_gb300.build``.
"""
from .kvring import (KVRING_EINVAL, KVRING_ENODEV, KVRING_ENOMEM, KVRING_ECUDA, KVRING_ESTATE,  # noqa: F401
                     KVRING_ETIMEOUT, KVRING_OK, KVRing, KVRingError, kvring_attend, kvring_attend_noalloc, kvring_check_device,
                     kvring_config, kvring_create, kvring_debug_fault, kvring_destroy, kvring_get_state,
                     kvring_last_error, kvring_launch_count, kvring_rebase, kvring_snapshot, kvring_state, kvring_write,
                     kvring_write_ex, KVRING_WRITE_REWRITE, KVRING_FLAG_NAIVE_UPKEEP, kvring_naive_refresh, KVRING_FLAG_ROPE_3D)
