"""The C-ABI library (CPU checks, no GPU): it loads, exports every entry point declared
in include/oscar.h, and validates configurations / sizes its device block without CUDA."""
import ctypes
import os
import re

import pytest

ROOT = os.path.dirname(os.path.dirname(os.path.abspath(__file__)))


@pytest.fixture(scope="module")
def lib():
    from int2_rotated_kv_rotate_gb300 import build, _native

    build.build()
    return _native.lib()


def declared_functions():
    text = open(os.path.join(ROOT, "include", "oscar.h")).read()
    text = re.sub(r"/\*.*?\*/", "", text, flags=re.S)
    return sorted(set(re.findall(r"\b(oscar_[a-z0-9_]+)\s*\(", text)))


def test_every_declared_symbol_is_exported(lib):
    names = declared_functions()
    assert len(names) >= 20
    from int2_rotated_kv_rotate_gb300 import _native

    for n in names:
        assert hasattr(lib, n), f"{n} not exported"
        assert n in _native.EXPORTS, f"{n} has no binding"
    assert sorted(_native.EXPORTS) == names


def cfg(**kw):
    from int2_rotated_kv_rotate_gb300._native import oscar_config

    base = dict(format=0, head_dim=128, n_q_heads=32, n_kv_heads=8, group=128, page=64, n_sink=4, window=128,
                n_layers=2, max_requests=4, max_pages=100, max_pages_per_request=50)
    base.update(kw)
    return oscar_config(*[base[f] for f, _ in oscar_config._fields_])


def test_device_bytes_and_invalid_configs(lib):
    c = cfg()
    n = lib.oscar_cache_device_bytes(ctypes.byref(c))
    # INT2 pools: per (layer, page, kv-head) 4096 B codes + 512 B scale/zero (g128)
    assert n >= 2 * 100 * 8 * (4096 + 512)
    c32 = cfg(group=32)
    n32 = lib.oscar_cache_device_bytes(ctypes.byref(c32))
    assert n32 - n >= 2 * 100 * 8 * (2048 - 512) - 4096  # g32 scale/zero: 2 KB per page-head
    bf = cfg(format=1)
    nb = lib.oscar_cache_device_bytes(ctypes.byref(bf))
    assert nb >= 2 * 100 * 8 * 32768
    for bad in (dict(head_dim=64), dict(page=32), dict(group=64), dict(n_q_heads=24), dict(n_q_heads=16),
                dict(window=100), dict(window=2048), dict(n_sink=65), dict(n_layers=0), dict(max_pages=0),
                dict(format=3)):
        c = cfg(**bad)
        assert lib.oscar_cache_device_bytes(ctypes.byref(c)) == 0, bad
        assert lib.oscar_last_error()


def test_null_handles_are_rejected(lib):
    assert lib.oscar_commit_append(None) == 1
    assert lib.oscar_decode_workspace_bytes(None) == 0
    lib.oscar_decode_workspace_max_bytes.restype = ctypes.c_size_t
    assert lib.oscar_decode_workspace_max_bytes(None) == 0
    s = ctypes.c_int()
    assert lib.oscar_request_alloc(None, ctypes.byref(s)) == 1
