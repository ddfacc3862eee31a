"""Test helper: make sure libkvring.so exists (build it in-tree when missing)."""
import os

from kv_cache_gb300 import build as _build
from kv_cache_gb300 import kvring as _kv


def ensure_built():
    if not os.path.exists(_kv.LIB_PATH):
        _build.build()
    return _kv.load()
