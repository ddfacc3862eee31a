"""The C ABI library loads and exports every entry point include/kvring.h declares."""
import ctypes
import re

from kv_cache_gb300 import kvring as kv
from tests._lib import ensure_built


def _declared():
    text = open(kv.HEADER).read()
    text = re.sub(r"/\*.*?\*/", "", text, flags=re.S)
    return sorted(set(re.findall(r"\b(kvring_[a-z_]+)\s*\(", text)))


def test_header_declares_the_boundary():
    names = _declared()
    for required in ["kvring_create", "kvring_write", "kvring_attend", "kvring_rebase", "kvring_destroy",
                     "kvring_get_state", "kvring_snapshot", "kvring_last_error", "kvring_check_device"]:
        assert required in names


def test_library_exports_every_declared_symbol():
    lib = ensure_built()
    for name in _declared():
        assert hasattr(lib, name), name
    # the binding wraps each one under the same name
    for name in _declared():
        assert hasattr(kv, name), name


def test_struct_layouts_match_header():
    ensure_built()
    assert ctypes.sizeof(kv.kvring_config) == 12 * 4
    assert ctypes.sizeof(kv.kvring_state) == 7 * 8
