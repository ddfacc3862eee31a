"""Thin Python binding of libkvring.so (ctypes).  Argument marshalling only.

Every function has the name of the C entry point it calls and the same
arguments, with torch tensors in place of raw device pointers and a torch
stream (default: the current stream) in place of ``cudaStream_t``.  A non-zero
status raises :class:`KVRingError` carrying the code and the library's message.
Nothing here computes any part of the cache path: the library's kernels do.
If the shared library is missing, loading raises; there is no fallback.
"""
from __future__ import annotations

import ctypes
import os
from typing import Optional

import numpy as np

PKG = os.path.dirname(os.path.abspath(__file__))
ROOT = os.path.dirname(PKG)
LIB_PATH = os.path.join(PKG, "libkvring.so")
HEADER = os.path.join(ROOT, "include", "kvring.h")

KVRING_OK = 0
KVRING_EINVAL = -1
KVRING_ENOMEM = -2
KVRING_ECUDA = -3
KVRING_ESTATE = -4
KVRING_ETIMEOUT = -5
KVRING_ENODEV = -6
KVRING_FLAG_HOST_ONLY = 0x1
KVRING_FLAG_NAIVE_UPKEEP = 0x2
KVRING_FLAG_ROPE_3D = 0x4
KVRING_MAX_LAYERS = 256

ERROR_NAMES = {0: "OK", -1: "EINVAL", -2: "ENOMEM", -3: "ECUDA", -4: "ESTATE", -5: "ETIMEOUT", -6: "ENODEV"}


class kvring_config(ctypes.Structure):
    _fields_ = [
        ("num_layers", ctypes.c_int32),
        ("num_heads", ctypes.c_int32),
        ("head_dim", ctypes.c_int32),
        ("capacity", ctypes.c_int32),
        ("max_tokens_per_write", ctypes.c_int32),
        ("max_position", ctypes.c_int32),
        ("rope_theta", ctypes.c_float),
        ("flags", ctypes.c_uint32),
        ("frame_tokens", ctypes.c_int32),
        ("frame_width", ctypes.c_int32),
        ("rope_pairs_t", ctypes.c_int32),
        ("rope_pairs_h", ctypes.c_int32),
    ]


class kvring_state(ctypes.Structure):
    _fields_ = [
        ("head", ctypes.c_int64),
        ("count", ctypes.c_int64),
        ("next_pos", ctypes.c_int64),
        ("writes", ctypes.c_int64),
        ("resets", ctypes.c_int64),
        ("last_write_pos", ctypes.c_int64),
        ("last_write_tokens", ctypes.c_int64),
    ]

    def as_dict(self) -> dict:
        return {name: int(getattr(self, name)) for name, _ in self._fields_}


class KVRingError(RuntimeError):
    def __init__(self, code: int, message: str):
        super().__init__(f"kvring {ERROR_NAMES.get(code, code)}: {message}")
        self.code = code
        self.message = message


_lib: Optional[ctypes.CDLL] = None

_P = ctypes.c_void_p
_SIGNATURES = {
    "kvring_create": (ctypes.c_int, [ctypes.POINTER(kvring_config), ctypes.POINTER(_P)]),
    "kvring_destroy": (ctypes.c_int, [_P]),
    "kvring_write": (ctypes.c_int, [_P, ctypes.c_int32, _P, _P, ctypes.c_int32, _P]),
    "kvring_write_ex": (ctypes.c_int, [_P, ctypes.c_int32, _P, _P, ctypes.c_int32, ctypes.c_uint32, _P]),
    "kvring_attend": (ctypes.c_int, [_P, ctypes.c_int32, _P, ctypes.c_int32, _P, _P]),
    "kvring_rebase": (ctypes.c_int, [_P, _P]),
    "kvring_naive_refresh": (ctypes.c_int, [_P, ctypes.c_int32, _P]),
    "kvring_get_state": (ctypes.c_int, [_P, ctypes.c_int32, ctypes.POINTER(kvring_state)]),
    "kvring_snapshot": (ctypes.c_int, [_P, ctypes.c_int32, _P, _P, _P, _P, _P, _P, _P]),
    "kvring_snapshot_q": (ctypes.c_int, [_P, _P, _P, _P]),
    "kvring_check_device": (ctypes.c_int, [_P, _P]),
    "kvring_last_error": (ctypes.c_char_p, [_P]),
    "kvring_debug_fault": (ctypes.c_int, [_P, ctypes.c_int32, ctypes.c_int64]),
    "kvring_debug_fault_write": (ctypes.c_int, [_P, ctypes.c_int32, ctypes.c_int64]),
    "kvring_launch_count": (ctypes.c_int, [_P, ctypes.POINTER(ctypes.c_uint64)]),
    "kvring_attend_noalloc": (ctypes.c_int, [_P, _P, _P, _P, _P, ctypes.c_int64, ctypes.c_int64, _P, ctypes.c_int32,
                                             ctypes.c_int32, ctypes.c_int32, ctypes.c_int32, ctypes.c_int32, _P, _P,
                                             _P]),
}


def load(path: str = LIB_PATH) -> ctypes.CDLL:
    """Load libkvring.so once (raises OSError if it has not been built)."""
    global _lib
    if _lib is not None:
        return _lib
    if not os.path.exists(path):
        raise OSError(f"{path} is missing: run `python -m kv_cache_gb300.build` first")
    lib = ctypes.CDLL(path)
    for name, (res, args) in _SIGNATURES.items():
        fn = getattr(lib, name)
        fn.restype = res
        fn.argtypes = args
    _lib = lib
    return lib


def _check(rc: int, ring) -> None:
    if rc != KVRING_OK:
        msg = load().kvring_last_error(ring)
        raise KVRingError(rc, msg.decode() if msg else "")


def _stream(stream) -> int:
    if stream is None:
        import torch
        return torch.cuda.current_stream().cuda_stream
    if isinstance(stream, int):
        return stream
    return stream.cuda_stream


def _dev_bf16(t, n: int, H: int, d: int, name: str) -> int:
    import torch
    if not isinstance(t, torch.Tensor):
        raise TypeError(f"{name} must be a torch tensor")
    if t.dtype != torch.bfloat16 or not t.is_cuda or not t.is_contiguous():
        raise ValueError(f"{name} must be a contiguous CUDA bfloat16 tensor")
    if tuple(t.shape) != (n, H, d):
        raise ValueError(f"{name} must have shape ({n}, {H}, {d}), got {tuple(t.shape)}")
    return t.data_ptr()


def kvring_create(cfg: kvring_config):
    """Returns the opaque handle (a ctypes void pointer value)."""
    lib = load()
    h = _P()
    rc = lib.kvring_create(ctypes.byref(cfg), ctypes.byref(h))
    _check(rc, None)
    return h.value


def kvring_destroy(ring) -> None:
    _check(load().kvring_destroy(ring), None)


def kvring_write(ring, layer: int, k, v, n_tokens: int, H: int, d: int, stream=None) -> None:
    kp = _dev_bf16(k, n_tokens, H, d, "k") if k is not None else None
    vp = _dev_bf16(v, n_tokens, H, d, "v") if v is not None else None
    s = _stream(stream) if (k is not None or v is not None) else 0
    _check(load().kvring_write(ring, layer, kp, vp, n_tokens, s), ring)


KVRING_WRITE_REWRITE = 0x1


def kvring_write_ex(ring, layer: int, k, v, n_tokens: int, flags: int, H: int, d: int, stream=None) -> None:
    kp = _dev_bf16(k, n_tokens, H, d, "k") if k is not None else None
    vp = _dev_bf16(v, n_tokens, H, d, "v") if v is not None else None
    s = _stream(stream) if (k is not None or v is not None) else 0
    _check(load().kvring_write_ex(ring, layer, kp, vp, n_tokens, flags, s), ring)


def kvring_attend(ring, layer: int, q, n_q: int, out, H: int, d: int, stream=None) -> None:
    import torch
    qp = _dev_bf16(q, n_q, H, d, "q")
    if out.dtype != torch.float32 or not out.is_cuda or not out.is_contiguous() or tuple(out.shape) != (n_q, H, d):
        raise ValueError(f"out must be a contiguous CUDA float32 tensor of shape ({n_q}, {H}, {d})")
    _check(load().kvring_attend(ring, layer, qp, n_q, out.data_ptr(), _stream(stream)), ring)


def kvring_naive_refresh(ring, layer: int, stream=None, host_only: bool = False) -> None:
    _check(load().kvring_naive_refresh(ring, layer, 0 if host_only else _stream(stream)), ring)


def kvring_rebase(ring, stream=None, host_only: bool = False) -> None:
    _check(load().kvring_rebase(ring, 0 if host_only else _stream(stream)), ring)


def kvring_get_state(ring, layer: int) -> dict:
    st = kvring_state()
    _check(load().kvring_get_state(ring, layer, ctypes.byref(st)), ring)
    return st.as_dict()


def kvring_snapshot(ring, layer: int, H: int, R: int, d: int, stream=None, cache: bool = True) -> dict:
    """Synchronous copy of one layer to new numpy arrays."""
    k = np.zeros((H, R, d), np.uint8) if cache else None
    v = np.zeros((H, R, d), np.uint8) if cache else None
    ka = np.zeros((H, R), np.float32) if cache else None
    va = np.zeros((H, R), np.float32) if cache else None
    pos = np.zeros(R, np.int32)
    chunk = np.zeros(R, np.int32)
    ptr = lambda a: a.ctypes.data if a is not None else None
    s = _stream(stream) if cache else 0
    _check(load().kvring_snapshot(ring, layer, ptr(k), ptr(v), ptr(ka), ptr(va), ptr(pos), ptr(chunk), s), ring)
    return {"k": k, "v": v, "kamax": ka, "vamax": va, "pos": pos, "chunk": chunk}


def kvring_snapshot_q(ring, n_q: int, H: int, d: int, stream=None) -> dict:
    """Synchronous copy of the latest attention call's e4m3 Q codes [H, n_q, d] and row amax [H, n_q]."""
    q8 = np.zeros((H, n_q, d), np.uint8)
    qamax = np.zeros((H, n_q), np.float32)
    _check(load().kvring_snapshot_q(ring, q8.ctypes.data, qamax.ctypes.data, _stream(stream)), ring)
    return {"q8": q8, "qamax": qamax}


def kvring_check_device(ring, stream=None) -> int:
    """KVRING_OK or KVRING_ETIMEOUT (returned, not raised); other codes raise."""
    rc = load().kvring_check_device(ring, _stream(stream))
    if rc not in (KVRING_OK, KVRING_ETIMEOUT):
        _check(rc, ring)
    return rc


def kvring_last_error(ring) -> str:
    msg = load().kvring_last_error(ring)
    return msg.decode() if msg else ""


def kvring_launch_count(ring) -> int:
    n = ctypes.c_uint64()
    _check(load().kvring_launch_count(ring, ctypes.byref(n)), ring)
    return int(n.value)


def kvring_debug_fault(ring, skip_tile: int, timeout_ns: int) -> None:
    _check(load().kvring_debug_fault(ring, skip_tile, timeout_ns), ring)


def kvring_debug_fault_write(ring, skip_group: int, timeout_ns: int) -> None:
    _check(load().kvring_debug_fault_write(ring, skip_group, timeout_ns), ring)


def noalloc_arg_error(k8, vt8, kamax, vamax, rope, q_pos0: int, q, out, count: int, err=None, device=None):
    """The first problem with kvring_attend_noalloc's arguments, or None.

    Checks every tensor's dtype, shape, contiguity and device (``device``: the
    device the call will run on, by default the current CUDA device), that the
    RoPE table has the rows the queries read, and that ``err`` is None or int32
    with at least 4 elements.  The library repeats the checks it can make on raw
    pointers (row counts, sizes, alignment); dtypes and devices only this layer sees.
    """
    import torch
    if device is None:
        if not torch.cuda.is_available():
            return "no CUDA device is available"
        device = torch.device("cuda", torch.cuda.current_device())
    device = torch.device(device)
    if not isinstance(q, torch.Tensor) or q.dim() != 3:
        return "q must be a tensor of shape (n_q, H, d)"
    n_q, H, d = (int(x) for x in q.shape)
    if not isinstance(k8, torch.Tensor) or k8.dim() != 3:
        return "k8 must be a tensor of shape (H, slots_padded, d)"
    slots_padded = int(k8.shape[1])
    spec = (("q", q, torch.bfloat16, (n_q, H, d)), ("k8", k8, torch.uint8, (H, slots_padded, d)),
            ("vt8", vt8, torch.uint8, (H, d, slots_padded)), ("kamax", kamax, torch.float32, (H, slots_padded)),
            ("vamax", vamax, torch.float32, (H, slots_padded)), ("out", out, torch.float32, (n_q, H, d)))
    for name, t, dtype, shape in spec:
        if not isinstance(t, torch.Tensor):
            return f"{name} must be a torch tensor"
        if t.dtype != dtype:
            return f"{name} must be {dtype}, got {t.dtype}"
        if tuple(t.shape) != shape:
            return f"{name} must have shape {shape}, got {tuple(t.shape)}"
        if not t.is_contiguous():
            return f"{name} must be contiguous"
        if t.device != device:
            return f"{name} is on {t.device}, the call runs on {device}"
    if not isinstance(rope, torch.Tensor) or rope.dtype != torch.float32 or rope.dim() != 3 \
            or tuple(rope.shape[1:]) != (d // 2, 2) or not rope.is_contiguous():
        return f"rope must be a contiguous float32 tensor of shape (rows, {d // 2}, 2)"
    if rope.device != device:
        return f"rope is on {rope.device}, the call runs on {device}"
    if int(q_pos0) < 0 or int(rope.shape[0]) < int(q_pos0) + n_q:
        return f"rope has {int(rope.shape[0])} rows; queries at positions {int(q_pos0)}..{int(q_pos0) + n_q - 1} need more"
    if not 1 <= int(count) <= slots_padded:
        return f"count must be in [1, {slots_padded}]"
    if err is not None:
        if not isinstance(err, torch.Tensor) or err.dtype != torch.int32 or err.numel() < 4 or not err.is_contiguous():
            return "err must be None or a contiguous int32 tensor of at least 4 elements"
        if err.device != device:
            return f"err is on {err.device}, the call runs on {device}"
    return None


def kvring_attend_noalloc(k8, vt8, kamax, vamax, rope, q_pos0: int, q, out, count: int, err=None,
                          stream=None) -> None:
    """Attention over a caller-held one-layer cache without any device allocation.

    k8 uint8 [H, slots_padded, d], vt8 uint8 [H, d, slots_padded], kamax/vamax
    float32 [H, slots_padded], rope float32 [rows, d/2, 2] with rows >= q_pos0 + n_q,
    q bf16 [n_q, H, d], out float32 [n_q, H, d], err int32 [>= 4] (zero before the
    call; it keeps the first time-out) or None -- all CUDA tensors the caller owns,
    on the current device (include/kvring.h has the layouts and the fixed scratch
    limit).  Bad arguments raise ValueError before anything is launched.
    """
    msg = noalloc_arg_error(k8, vt8, kamax, vamax, rope, q_pos0, q, out, count, err)
    if msg is not None:
        raise ValueError(msg)
    n_q, H, d = (int(x) for x in q.shape)
    slots_padded = int(k8.shape[1])
    rc = load().kvring_attend_noalloc(k8.data_ptr(), vt8.data_ptr(), kamax.data_ptr(), vamax.data_ptr(),
                                      rope.data_ptr(), int(rope.shape[0]), int(q_pos0), q.data_ptr(), n_q, H, d,
                                      slots_padded, int(count), out.data_ptr(),
                                      err.data_ptr() if err is not None else None, _stream(stream))
    _check(rc, None)


class KVRing:
    """Owning wrapper: one ring set of `num_layers` rings."""

    def __init__(self, num_layers: int, num_heads: int, head_dim: int, capacity: int,
                 max_tokens_per_write: int, max_position: int = 0, rope_theta: float = 10000.0,
                 host_only: bool = False, naive_upkeep: bool = False, rope_3d=None):
        """rope_3d: None (1-D RoPE) or (frame_tokens, frame_width, pairs_t, pairs_h); pairs 0, 0 = default split."""
        flags = (KVRING_FLAG_HOST_ONLY if host_only else 0) | (KVRING_FLAG_NAIVE_UPKEEP if naive_upkeep else 0)
        S, W, pt, ph = rope_3d if rope_3d is not None else (0, 0, 0, 0)
        if rope_3d is not None:
            flags |= KVRING_FLAG_ROPE_3D
        self.cfg = kvring_config(num_layers, num_heads, head_dim, capacity, max_tokens_per_write,
                                 max_position, rope_theta, flags, S, W, pt, ph)
        self.L, self.H, self.d, self.R = num_layers, num_heads, head_dim, capacity
        self.host_only = host_only
        self._last_nq = 0
        self.handle = kvring_create(self.cfg)

    def close(self) -> None:
        if self.handle:
            kvring_destroy(self.handle)
            self.handle = None

    def __del__(self):
        try:
            self.close()
        except Exception:
            pass

    def __enter__(self):
        return self

    def __exit__(self, *exc):
        self.close()

    def write(self, layer: int, k, v, n_tokens: Optional[int] = None, stream=None) -> None:
        n = k.shape[0] if n_tokens is None else n_tokens
        kvring_write(self.handle, layer, k, v, n, self.H, self.d, stream)

    def rewrite(self, layer: int, k, v, n_tokens: Optional[int] = None, stream=None) -> None:
        """Replace the latest chunk of ``layer`` with new K, V (next denoise pass)."""
        n = k.shape[0] if n_tokens is None else n_tokens
        kvring_write_ex(self.handle, layer, k, v, n, KVRING_WRITE_REWRITE, self.H, self.d, stream)

    def attend(self, layer: int, q, out=None, stream=None):
        import torch
        if out is None:
            out = torch.empty((q.shape[0], self.H, self.d), dtype=torch.float32, device=q.device)
        kvring_attend(self.handle, layer, q, q.shape[0], out, self.H, self.d, stream)
        self._last_nq = int(q.shape[0])
        return out

    def rebase(self, stream=None) -> None:
        kvring_rebase(self.handle, stream, host_only=self.host_only)

    def naive_refresh(self, layer: int, stream=None) -> None:
        """Naive-upkeep rings: re-rotate and re-quantise the layer's whole window."""
        kvring_naive_refresh(self.handle, layer, stream, host_only=self.host_only)

    def state(self, layer: int) -> dict:
        return kvring_get_state(self.handle, layer)

    def snapshot(self, layer: int, stream=None, cache: bool = True) -> dict:
        return kvring_snapshot(self.handle, layer, self.H, self.R, self.d, stream, cache)

    def snapshot_q(self, stream=None) -> dict:
        """The latest attention call's prepared queries (e4m3 codes and row amax)."""
        return kvring_snapshot_q(self.handle, self._last_nq, self.H, self.d, stream)

    def check_device(self, stream=None) -> int:
        return kvring_check_device(self.handle, stream)

    def launch_count(self) -> int:
        return kvring_launch_count(self.handle)
