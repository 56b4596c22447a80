"""The C-ABI library builds, loads and exports what include/pkv.h declares.

CPU only: every call here is rejected by host-side argument checks (or is a
size query) before any CUDA runtime call, so no GPU is needed.
"""

import ctypes
import os
import re

import pytest

from paged_kv_decode_05_gb300 import binding as B
from paged_kv_decode_05_gb300.build import build

INCLUDE = os.path.join(os.path.dirname(os.path.dirname(__file__)), "include")
HEADERS = sorted(os.path.join(INCLUDE, f) for f in os.listdir(INCLUDE) if f.endswith(".h"))


@pytest.fixture(scope="module")
def lib():
    build()
    return B.lib()


def declared_functions():
    text = "".join(open(h).read() for h in HEADERS)
    text = re.sub(r"/\*.*?\*/", "", text, flags=re.S)
    return sorted(set(re.findall(r"\b(pkv_[a-z0-9_]+)\s*\(", text)))


def test_every_declared_symbol_is_exported(lib):
    names = declared_functions()
    assert len(names) >= 8
    for n in names:
        assert hasattr(lib, n), n
    assert sorted(B.exported_symbols()) == names


def test_status_strings(lib):
    for code, name in B.STATUS.items():
        assert B.pkv_status_string(code).startswith(name)
    assert B.pkv_status_string(99) == "PKV_ERR_UNKNOWN"


def desc(nb=8, bs=16, h=2, d=128, dt=B.PKV_BF16):
    return B.CacheDesc(nb, bs, h, d, dt)


def test_append_host_validation(lib):
    P = ctypes.c_void_p
    fake = 0x100000  # never dereferenced: each call fails its host checks first
    d = desc()
    assert lib.pkv_append(fake, fake, B.PKV_BF16, 4, fake, fake, fake, None, None, None, None, 0,
                          None, None) == 1
    assert lib.pkv_append(None, fake, B.PKV_BF16, 4, fake, fake, fake, None, None,
                          ctypes.byref(d), None, 0, None, None) == 1
    assert lib.pkv_append(fake + 8, fake, B.PKV_BF16, 4, fake, fake, fake, None, None,
                          ctypes.byref(d), None, 0, None, None) == 1        # misaligned
    assert lib.pkv_append(fake, fake, B.PKV_F16, 4, fake, fake, fake, None, None,
                          ctypes.byref(d), None, 0, None, None) == 1        # dtype mismatch
    assert lib.pkv_append(fake, fake, B.PKV_BF16, -1, fake, fake, fake, None, None,
                          ctypes.byref(d), None, 0, None, None) == 1
    assert lib.pkv_append(fake, fake, B.PKV_BF16, 0, fake, fake, fake, None, None,
                          ctypes.byref(d), None, 0, None, None) == 0        # nothing to do
    d96 = desc(d=96)
    assert lib.pkv_append(fake, fake, B.PKV_BF16, 4, fake, fake, fake, None, None,
                          ctypes.byref(d96), None, 0, None, None) == 2
    d8 = desc(dt=B.PKV_I8)
    need = lib.pkv_append_workspace_size(ctypes.byref(d8))
    assert need == 80 * 8 * 2          # 80 bytes per (block, kv head) tile
    assert lib.pkv_append(fake, fake, B.PKV_BF16, 4, fake, fake, fake, fake, fake,
                          ctypes.byref(d8), fake, need - 4, None, None) == 3  # workspace
    assert lib.pkv_append(fake, fake, B.PKV_BF16, 4, fake, fake, fake, None, fake,
                          ctypes.byref(d8), fake, need, None, None) == 1      # no k_scales
    assert lib.pkv_append_workspace_size(ctypes.byref(d)) == 0
    del P


def _decode(lib, fn, q_dtype=B.PKV_BF16, d=None, batch=4, hq=8, ws=None, ws_bytes=1 << 30,
            parts=64, q=0x100000):
    fake = 0x100000
    d = d or desc()
    return getattr(lib, fn)(q, q_dtype, fake, fake, None, None, ctypes.byref(d), fake, 4, fake,
                            batch, hq, 0.125, fake, fake if ws is None else ws, ws_bytes, parts,
                            None, None)


def test_decode_host_validation(lib):
    for fn in ("pkv_decode_attn", "pkv_decode_split"):
        assert _decode(lib, fn, hq=7) == 1                       # hq % hkv
        assert _decode(lib, fn, hq=32) == 2                      # group 16 not built
        assert _decode(lib, fn, d=desc(d=80)) == 2
        assert _decode(lib, fn, d=desc(bs=32)) == 2
        assert _decode(lib, fn, q_dtype=B.PKV_F16) == 1          # q != kv 16-bit type
        assert _decode(lib, fn, batch=9000) == 2
        assert _decode(lib, fn, batch=0) == 0
        assert _decode(lib, fn, q=None) == 1
        assert _decode(lib, fn, q=0x100008) == 1                 # misaligned q
        assert _decode(lib, fn, ws_bytes=16) == 3                # workspace too small
        assert _decode(lib, fn, ws=0x100080) == 3                # workspace not 256-aligned
        assert _decode(lib, fn, d=desc(dt=B.PKV_I8)) == 1        # int8 without scales
    assert lib.pkv_decode_combine(ctypes.byref(desc()), 4, 8, B.PKV_BF16, 0x100000, 0x100000,
                                  16, 64, None) == 3


def test_workspace_size_formula(lib):
    d = desc(nb=100, h=8, d=128)
    got = lib.pkv_decode_workspace_size(256, 32, ctypes.byref(d), 1824)
    slots = 256 * 8 + 1824
    a = lambda x: (x + 255) // 256 * 256  # noqa: E731
    assert got == a(4 * 257) + a(slots * 4 * 2 * 4) + a(slots * 4 * 128 * 4)
    assert lib.pkv_decode_workspace_size(256, 12, ctypes.byref(d), 64) == 0  # unsupported group
    assert lib.pkv_decode_workspace_size(256, 128, ctypes.byref(d), 64) == 0  # group 16
    g8 = lib.pkv_decode_workspace_size(256, 64, ctypes.byref(d), 1216)        # group 8
    slots = 256 * 8 + 1216
    assert g8 == a(4 * 257) + a(slots * 8 * 2 * 4) + a(slots * 8 * 128 * 4)


def test_multiquery_and_copy_blocks_host_validation(lib):
    fake = 0x100000
    d = desc(nb=64, h=2, d=128)

    def mq(q_dtype=B.PKV_BF16, dd=None, batch=4, hq=8, max_q=5, ws=fake, ws_bytes=1 << 30,
           parts=16):
        return lib.pkv_multiquery_attn(fake, q_dtype, fake, max_q, fake, fake, scales, scales,
                                       ctypes.byref(dd or d), fake, 4, fake, batch, hq, 0.125,
                                       fake, ws, ws_bytes, parts, None, None)
    scales = None
    assert mq(hq=7) == 1                         # heads not a multiple of kv heads
    assert mq(hq=32) == 2                        # group 16 not built
    assert mq(max_q=0) == 1
    assert mq(q_dtype=B.PKV_F16) == 1            # q dtype must match a 16-bit cache
    assert mq(q_dtype=B.PKV_I8) == 1             # q is never INT8
    assert mq(dd=desc(dt=B.PKV_I8)) == 1         # INT8 caches need their scales
    assert mq(dd=desc(d=96)) == 2
    assert mq(batch=5000) == 2
    assert mq(batch=0) == 0
    assert mq(ws_bytes=64) == 3
    assert mq(ws=fake + 128) == 3                # workspace not 256-aligned
    # size query agrees with the layout: 20 rows (5 queries x group 4) take
    # the short-run kernel's tile of 24 rows, one tile per (sequence, kv head)
    dd = desc(nb=64, h=2, d=128)
    slots = 4 * 2 * 1 + 16
    a = lambda x: (x + 255) // 256 * 256  # noqa: E731
    assert lib.pkv_multiquery_workspace_size(4, 8, 5, ctypes.byref(dd), 16) == \
        a(4 * 5) + a(slots * 24 * 2 * 4) + a(slots * 24 * 128 * 4)
    # 28 rows (7 queries x group 4): the mma.sync kernel's 32-row tile
    assert lib.pkv_multiquery_workspace_size(4, 8, 7, ctypes.byref(dd), 16) == \
        a(4 * 5) + a(slots * 32 * 2 * 4) + a(slots * 32 * 128 * 4)
    # block copy
    assert lib.pkv_copy_blocks(fake, fake, None, None, ctypes.byref(d), fake, fake, 0, None,
                               None) == 0
    assert lib.pkv_copy_blocks(fake, fake, None, None, ctypes.byref(d), fake, fake, -1, None,
                               None) == 1
    assert lib.pkv_copy_blocks(fake, fake, None, None, ctypes.byref(desc(dt=B.PKV_I8)), fake, fake,
                               3, None, None) == 1   # INT8 needs scales
    assert lib.pkv_copy_blocks(fake + 4, fake, None, None, ctypes.byref(d), fake, fake, 3, None,
                               None) == 1            # misaligned cache


def test_decode_step_host_validation(lib):
    fake = 0x100000
    d = desc()

    def step(dd=None, k_new=fake, run_combine=1, batch=4, hq=8, scales=None):
        return lib.pkv_decode_step(fake, B.PKV_BF16, k_new, fake, fake, fake, scales, scales,
                                   ctypes.byref(dd or d), fake, 4, fake, batch, hq, 0.125, fake,
                                   fake, 1 << 30, 64, run_combine, None, None)
    assert step(dd=desc(dt=B.PKV_I8)) == 1       # INT8 caches need their scales
    assert step(dd=desc(dt=B.PKV_I8), scales=fake + 2) == 1   # misaligned scales
    assert step(run_combine=2) == 1
    assert step(k_new=None) == 1
    assert step(k_new=fake + 8) == 1             # the new rows are bulk-copied: 16-byte aligned
    assert step(hq=7) == 1
    assert step(batch=0) == 0
    assert lib.pkv_decode_step(fake, B.PKV_BF16, fake, fake, fake, fake, None, None, None, fake, 4,
                               fake, 4, 8, 0.125, fake, fake, 1 << 30, 64, 1, None, None) == 1
