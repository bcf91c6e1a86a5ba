"""The C-ABI library without a GPU: it loads, exports every entry point the
header declares, and rejects bad arguments on the host before any CUDA call."""
import ctypes
import os
import re

import numpy as np
import pytest

import paged_kv_cache_190_gb300 as pa

ROOT = os.path.dirname(os.path.dirname(os.path.abspath(__file__)))


def _declared_functions():
    text = open(os.path.join(ROOT, "include", "pa.h")).read()
    text = re.sub(r"/\*.*?\*/", "", text, flags=re.S)
    names = set(re.findall(r"\b(pa_[a-z0-9_]+)\s*\(", text))
    return names


def test_library_exports_every_declared_symbol():
    lib = pa.library()
    declared = _declared_functions()
    assert declared == set(pa.EXPORTED_SYMBOLS)
    for name in sorted(declared):
        assert hasattr(lib, name), name


def test_error_strings():
    for code in range(0, -8, -1):
        s = pa.pa_get_error_string(code)
        assert s and s != "unknown status", code
    assert pa.pa_get_error_string(-99) == "unknown status"


def _decode_raw(**over):
    lib = pa.library()
    buf = (ctypes.c_uint8 * 4096)()
    base = ctypes.addressof(buf)
    aligned = (base + 255) & ~255
    args = dict(out=aligned, q=aligned, k=aligned, v=aligned, bt=aligned, cl=aligned, scale=1.0,
                hkv=8, b=2, hq=32, d=128, bs=16, nb=64, mbps=8, maxlen=100, dtype=1, chunk=0,
                ws=aligned, wsb=1 << 30, errs=None, stream=None)
    args.update(over)
    return lib.pa_decode(args["out"], args["q"], args["k"], args["v"], args["bt"], args["cl"],
                         args["scale"], args["hkv"], args["b"], args["hq"], args["d"], args["bs"],
                         args["nb"], args["mbps"], args["maxlen"], args["dtype"], args["chunk"],
                         args["ws"], args["wsb"], args["errs"], args["stream"])


@pytest.mark.parametrize("over,status", [
    (dict(dtype=7), -2),
    (dict(d=96), -2),
    (dict(bs=8), -2),
    (dict(hq=30), -1),            # not a multiple of the kv heads
    (dict(hq=24), -2),            # group of 3
    (dict(hkv=0), -1),
    (dict(b=-1), -1),
    (dict(maxlen=8 * 16 + 1), -1),  # longer than a table row holds
    (dict(out=None), -1),
    (dict(bt=None), -1),
    (dict(q=12345), -1),          # misaligned
    (dict(b=0), 0),               # nothing to do
])
def test_decode_host_checks(over, status):
    assert _decode_raw(**over) == status


def test_cache_ops_host_checks():
    lib = pa.library()
    buf = (ctypes.c_uint8 * 1024)()
    p = (ctypes.addressof(buf) + 255) & ~255
    # reshape: unsupported head_dim, negative tokens, misaligned, empty
    assert lib.pa_reshape_and_cache(p, p, p, p, p, 4, 8, 96, 16, 64, 1, None, None) == -2
    assert lib.pa_reshape_and_cache(p, p, p, p, p, -1, 8, 128, 16, 64, 1, None, None) == -1
    assert lib.pa_reshape_and_cache(p + 4, p, p, p, p, 4, 8, 128, 16, 64, 1, None, None) == -1
    assert lib.pa_reshape_and_cache(p, p, p, p, p, 0, 8, 128, 16, 64, 1, None, None) == 0
    # copy_blocks: block size not a multiple of 16, empty list
    assert lib.pa_copy_blocks(p, p, p, 3, 40, 64, None, None) == -1
    assert lib.pa_copy_blocks(p, p, p, 0, 4096, 64, None, None) == 0
    assert lib.pa_copy_blocks(None, p, p, 2, 4096, 64, None, None) == -1


def test_workspace_size_with_explicit_chunk_is_monotone():
    s1 = pa.pa_decode_workspace_size(4, 32, 8, 128, 16, 1000, 64)
    s2 = pa.pa_decode_workspace_size(4, 32, 8, 128, 16, 2000, 64)
    s3 = pa.pa_decode_workspace_size(4, 32, 8, 128, 16, 2000, 128)
    assert 0 < s1 < s2 and s3 < s2
    # chunk must be a multiple of 16 and of the block size, at most 128 pages
    assert pa.pa_decode_workspace_size(4, 32, 8, 128, 32, 2000, 48) == 0
    assert pa.pa_decode_workspace_size(4, 32, 8, 128, 16, 2000, 2048) > 0
    assert pa.pa_decode_workspace_size(4, 32, 8, 128, 16, 2000, 4096) == 0
    assert pa.pa_decode_workspace_size(4, 32, 8, 128, 32, 8000, 4096) > 0
    assert pa.pa_decode_workspace_size(4, 32, 8, 128, 32, 8000, 8192) == 0


def test_cascade_host_checks():
    """pa_decode_cascade refuses bad group arguments on the host; its workspace
    covers the decode's and grows with the groups."""
    lib = pa.library()
    buf = (ctypes.c_uint8 * 4096)()
    p = (ctypes.addressof(buf) + 255) & ~255

    def call(num_groups=2, gs=p, sl=p, hq=32, b=4, d=128, bs=16):
        return lib.pa_decode_cascade(p, p, p, p, p, p, gs, sl, num_groups, 1.0, 8, b, hq, d, bs,
                                     64, 8, 100, 64, p, 1 << 30, None, None)
    assert call(num_groups=0) == -1                 # at least one group
    assert call(num_groups=5) == -1                 # more groups than sequences
    assert call(gs=None) == -1
    assert call(sl=None) == -1
    assert call(d=96) == -2
    assert call(bs=8) == -2
    assert call(hq=16 * 8) == -2                    # 16 query heads per kv head
    assert call(b=0, num_groups=0) == 0             # nothing to do
    dec = pa.pa_decode_workspace_size(4, 32, 8, 128, 16, 2000, 64)
    c1 = pa.pa_decode_cascade_workspace_size(4, 1, 32, 8, 128, 16, 2000, 64)
    c2 = pa.pa_decode_cascade_workspace_size(4, 3, 32, 8, 128, 16, 2000, 64)
    assert dec < c1 <= c2
    assert lib.pa_decode_cascade_workspace_size(4, 0, 32, 8, 128, 16, 2000, 64) == 0
    assert lib.pa_decode_cascade_workspace_size(4, 1, 32, 8, 128, 32, 2000, 48) == 0  # 1.5 pages
