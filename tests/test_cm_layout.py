"""Channel-major value pages (format OSCAR_FORMAT_INT2_CM), host side, no GPU.

The reader that rebuilds token-major 32-byte rows from a channel-major value block
(KVCache._cm_rows, which the GPU parity tests use to compare stored codes with the
oracle's rows) is checked against a block packed here, bit by bit, from the layout the C
header states: word 128 b + c holds channel c of tokens 16 b .. 16 b + 15, token
16 b + 8 h + f at bit 16 h + 2 f.  The configuration rules of the format go through the
library's own validation.
"""
import ctypes
import types

import numpy as np
import pytest
import torch

import oracle
from int2_rotated_kv_rotate_gb300.cache import KVCache


def cm_block(codes: np.ndarray) -> np.ndarray:
    """codes [64 tokens][128 channels] -> 512 little-endian uint32 words."""
    blk = np.zeros(512, dtype=np.uint32)
    for tok in range(64):
        b, h, f = tok // 16, (tok // 8) % 2, tok % 8
        for c in range(128):
            blk[128 * b + c] |= np.uint32(int(codes[tok, c]) << (16 * h + 2 * f))
    return blk


@pytest.mark.parametrize("seed", [1, 2])
def test_channel_major_rows_rebuild_the_token_rows(seed):
    rng = np.random.default_rng(seed)
    codes = rng.integers(0, 4, size=(64, 128)).astype(np.uint8)
    off = 4096  # the block somewhere inside a byte pool
    mem = torch.zeros(off + 2048 + 512, dtype=torch.uint8)
    mem[off:off + 2048] = torch.from_numpy(cm_block(codes).view(np.uint8).copy())
    fake = types.SimpleNamespace(mem=mem)
    t = torch.tensor(rng.permutation(64)[:40], dtype=torch.long)  # any positions, any order
    rows = KVCache._cm_rows(fake, torch.full((t.numel(),), off, dtype=torch.long), t).numpy()
    expect = np.stack([oracle.pack_row(codes[i]) for i in t.tolist()])
    assert np.array_equal(rows, expect)
    # a single changed code shows up in exactly its token's row
    codes2 = codes.copy()
    codes2[37, 101] ^= 2
    mem[off:off + 2048] = torch.from_numpy(cm_block(codes2).view(np.uint8).copy())
    rows2 = KVCache._cm_rows(fake, torch.full((64,), off, dtype=torch.long), torch.arange(64)).numpy()
    diff = np.nonzero((rows2 != np.stack([oracle.pack_row(codes[i]) for i in range(64)])).any(axis=1))[0]
    assert diff.tolist() == [37]


@pytest.fixture(scope="module")
def lib():
    from int2_rotated_kv_rotate_gb300 import build, _native

    build.build()
    return _native.lib()


def cfg(**kw):
    from int2_rotated_kv_rotate_gb300._native import oscar_config

    base = dict(format=2, head_dim=128, n_q_heads=32, n_kv_heads=8, group=128, page=64, n_sink=4, window=128,
                n_layers=2, max_requests=4, max_pages=100, max_pages_per_request=50)
    base.update(kw)
    return oscar_config(*[base[f] for f, _ in oscar_config._fields_])


def test_channel_major_configurations(lib):
    tm = cfg(format=0)
    same = lib.oscar_cache_device_bytes(ctypes.byref(tm))
    for ok in (dict(), dict(n_q_heads=64), dict(group=32)):  # GQA 4 / 8 at g128, GQA 4 at g32
        c = cfg(**ok)
        n = lib.oscar_cache_device_bytes(ctypes.byref(c))
        assert n > 0, ok
        if not ok:
            assert n == same  # the same pools, another order inside the value block
    bad = cfg(n_q_heads=64, group=32)  # GQA 8 at g32: no kernel
    assert lib.oscar_cache_device_bytes(ctypes.byref(bad)) == 0
    assert b"INT2_CM" in lib.oscar_last_error()
