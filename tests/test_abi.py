"""The C ABI: the library builds, loads, exports every function include/mla_decode.h
declares, and rejects bad host-side arguments before touching the GPU (so these
run without one)."""
import ctypes
import os
import re

import pytest

from mla_decode_attention_03_gb300 import build

HEADER = os.path.join(os.path.dirname(os.path.dirname(os.path.abspath(__file__))), "include",
                      "mla_decode.h")

FAKE = 1 << 20  # a 16-byte aligned non-null address; never dereferenced by rejected calls


@pytest.fixture(scope="module")
def lib():
    path = build.build()
    return ctypes.CDLL(str(path))


def declared_functions():
    text = open(HEADER, encoding="utf-8").read()
    text = re.sub(r"/\*.*?\*/", "", text, flags=re.S)
    return sorted(set(re.findall(r"\b(mla_[a-z_]+)\s*\(", text)))


def test_header_declares_the_entry_points():
    assert declared_functions() == sorted([
        "mla_status_string", "mla_num_parts", "mla_metadata_ints", "mla_workspace_bytes",
        "mla_get_metadata", "mla_decode_with_kvcache", "mla_decode_splitkv", "mla_combine_splits",
        "mla_decode_with_kvcache_static", "mla_write_cache", "mla_copy_blocks"])


def test_every_declared_symbol_is_exported(lib):
    for name in declared_functions():
        assert hasattr(lib, name), name


def _decode(lib, **kw):
    a = dict(q=FAKE, b=2, s_q=1, h_q=128, d=576, kcache=FAKE, num_blocks=10, block_size=64, h_kv=1,
             stride=576, block_table=FAKE, max_blocks=4, seqlens=FAKE, dv=512, metadata=FAKE,
             num_parts=4, num_splits=FAKE, scale=576 ** -0.5, causal=0, out=FAKE, lse=FAKE,
             workspace=FAKE, workspace_bytes=1 << 40, status=FAKE, stream=None)
    a.update(kw)
    f = lib.mla_decode_with_kvcache
    f.restype = ctypes.c_int32
    P, I, I64, SZ, F = ctypes.c_void_p, ctypes.c_int, ctypes.c_int64, ctypes.c_size_t, ctypes.c_float
    f.argtypes = [P, I, I, I, I, P, I64, I, I, I, P, I, P, I, P, I, P, F, I, P, P, P, SZ, P, P]
    return f(a["q"], a["b"], a["s_q"], a["h_q"], a["d"], a["kcache"], a["num_blocks"], a["block_size"],
             a["h_kv"], a["stride"], a["block_table"], a["max_blocks"], a["seqlens"], a["dv"],
             a["metadata"], a["num_parts"], a["num_splits"], a["scale"], a["causal"], a["out"],
             a["lse"], a["workspace"], a["workspace_bytes"], a["status"], a["stream"])


@pytest.mark.parametrize("kw,code", [
    (dict(d=512), -2), (dict(dv=256), -2), (dict(block_size=32), -2), (dict(h_q=256), -2),
    (dict(h_q=100, h_kv=3), -1), (dict(b=0), -1), (dict(s_q=0), -1), (dict(stride=500), -1),
    (dict(stride=580), -3), (dict(q=FAKE + 8), -3), (dict(out=FAKE + 2), -3),
    (dict(kcache=FAKE + 4), -3), (dict(workspace_bytes=16), -1), (dict(causal=2), -1),
    (dict(scale=float("nan")), -1), (dict(scale=0.0), -1), (dict(scale=-0.04), -1),
    (dict(num_parts=0), -1), (dict(q=0), -1),
    (dict(num_blocks=1 << 26), -1),
])
def test_decode_rejects_bad_arguments(lib, kw, code):
    assert _decode(lib, **kw) == code


def test_metadata_rejects_bad_arguments(lib):
    f = lib.mla_get_metadata
    f.restype = ctypes.c_int32
    f.argtypes = [ctypes.c_void_p, ctypes.c_int, ctypes.c_int, ctypes.c_void_p, ctypes.c_void_p,
                  ctypes.c_void_p, ctypes.c_void_p]
    assert f(FAKE, 0, 4, FAKE, FAKE, FAKE, None) == -1
    assert f(FAKE, 16385, 4, FAKE, FAKE, FAKE, None) == -1
    assert f(FAKE, 8, 0, FAKE, FAKE, FAKE, None) == -1
    assert f(None, 8, 4, FAKE, FAKE, FAKE, None) == -1


def test_sizes_and_strings(lib):
    lib.mla_workspace_bytes.restype = ctypes.c_size_t
    lib.mla_workspace_bytes.argtypes = [ctypes.c_int] * 4
    lib.mla_metadata_ints.restype = ctypes.c_size_t
    lib.mla_metadata_ints.argtypes = [ctypes.c_int]
    lib.mla_status_string.restype = ctypes.c_char_p
    lib.mla_status_string.argtypes = [ctypes.c_int32]
    # (b + parts) slots x rows x 512 bf16, then (b + parts) x rows fp32 lse, each 256-byte aligned
    o = (128 + 76) * 128 * 512 * 2
    l = (128 + 76) * 128 * 4
    assert lib.mla_workspace_bytes(128, 1, 128, 76) == o + ((l + 255) // 256) * 256
    assert lib.mla_workspace_bytes(0, 1, 128, 76) == 0
    assert lib.mla_metadata_ints(76) == 76 * 8
    for code in (0, -1, -2, -3, -4, -5, -6, -7, -8):
        assert lib.mla_status_string(code).startswith(b"MLA_")
    assert lib.mla_status_string(12345) == b"MLA: unknown status"
