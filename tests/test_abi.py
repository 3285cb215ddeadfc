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
        "mla_decode_with_kvcache_static", "mla_write_cache", "mla_copy_blocks",
        "mla_host_pipeline_create", "mla_host_pipeline_destroy", "mla_host_chunks",
        "mla_host_scratch_bytes", "mla_decode_host", "mla_selftest_wait_timeout"])


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
    # (b + parts) slots x rows x 512 fp32, then (b + parts) x rows fp32 lse, each 256-byte aligned
    o = (128 + 76) * 128 * 512 * 4
    l = (128 + 76) * 128 * 4
    assert lib.mla_workspace_bytes(128, 1, 128, 76) == o + ((l + 255) // 256) * 256
    assert lib.mla_workspace_bytes(0, 1, 128, 76) == 0
    assert lib.mla_metadata_ints(76) == 76 * 8
    for code in (0, -1, -2, -3, -4, -5, -6, -7, -8):
        assert lib.mla_status_string(code).startswith(b"MLA_")
    assert lib.mla_status_string(12345) == b"MLA: unknown status"


# ------------------------------------------------------------ host-buffer pipeline (host logic only)
MAX_CHUNKS = 8


def _chunks(lib, seqlens, chunks):
    f = lib.mla_host_chunks
    f.restype = ctypes.c_int
    f.argtypes = [ctypes.c_void_p, ctypes.c_int, ctypes.c_int, ctypes.c_void_p]
    sl = (ctypes.c_int32 * max(1, len(seqlens)))(*seqlens)
    bounds = (ctypes.c_int32 * (MAX_CHUNKS + 1))()
    n = f(ctypes.addressof(sl), len(seqlens), chunks, ctypes.addressof(bounds))
    return n, list(bounds[: n + 1]) if n > 0 else []


def _cost(L):
    return -(-max(L, 0) // 64) + 1


def _check_cut(seqlens, n, bounds):
    b = len(seqlens)
    assert bounds[0] == 0 and bounds[-1] == b and len(bounds) == n + 1
    assert all(x < y for x, y in zip(bounds, bounds[1:])), bounds  # no empty run
    costs = [_cost(L) for L in seqlens]
    total = sum(costs)
    prefix = [0]
    for c in costs:
        prefix.append(prefix[-1] + c)
    halves = n if n <= 2 else 2 * n - 2  # shares 1, 2, ..., 2, 1 in halves
    for k in range(1, n):
        e = bounds[k]
        before = k if n <= 2 else 2 * k - 1
        target = -(-total * before // halves)
        lo, hi = bounds[k - 1] + 1, b - (n - k)
        if lo < e < hi:
            # an unclamped bound is the first sequence where the running cost
            # reaches its share of the total (end runs half a middle run)
            assert prefix[e] >= target and prefix[e - 1] < target, (k, e, target)


@pytest.mark.parametrize("seqlens,chunks,want_n", [
    ([4096] * 128, 4, 4), ([4096] * 128, 1, 1), ([4096] * 128, 8, 8),
    ([4096] * 128, 100, 8), ([100, 200, 300], 8, 3), ([0, 0, 0, 0], 2, 2), ([5], 3, 1),
    ([65536, 65536] + [300] * 62, 4, 4), ([65536, 65536] + [300] * 62, 0, 1),
    ([256] * 16, 0, 1), ([4096] * 16, 0, 1), ([4096] * 32, 0, 1), ([4096] * 64, 0, 1),
    ([4096] * 128, 0, 3), ([8192] * 128, 0, 3),
    ([-5, 70, 1, 4096], 2, 2),
])
def test_host_chunks_cut(lib, seqlens, chunks, want_n):
    n, bounds = _chunks(lib, seqlens, chunks)
    assert n == want_n
    _check_cut(seqlens, n, bounds)


def test_host_chunks_uniform_batch_end_runs_half(lib):
    # 128 equal sequences: two runs split evenly; with more, the first and the
    # last run hold half as many sequences as each middle run
    assert _chunks(lib, [4096] * 128, 2)[1] == [0, 64, 128]
    assert _chunks(lib, [4096] * 128, 3)[1] == [0, 32, 96, 128]
    assert _chunks(lib, [4096] * 128, 5)[1] == [0, 16, 48, 80, 112, 128]


def test_host_chunks_random_batches(lib):
    import random
    rng = random.Random(7)
    for _ in range(300):
        b = rng.randint(1, 40)
        seqlens = [rng.choice([0, 1, 63, 64, 65, rng.randint(0, 20000)]) for _ in range(b)]
        chunks = rng.randint(-1, 10)
        n, bounds = _chunks(lib, seqlens, chunks)
        pages = sum(-(-max(L, 0) // 64) for L in seqlens)
        want = min(max(1, min(3, (pages + 1400) // 2800)) if chunks <= 0 else min(chunks, MAX_CHUNKS), b)
        assert n == want
        _check_cut(seqlens, n, bounds)


def test_host_chunks_rejects_bad_arguments(lib):
    f = lib.mla_host_chunks
    f.restype = ctypes.c_int
    f.argtypes = [ctypes.c_void_p, ctypes.c_int, ctypes.c_int, ctypes.c_void_p]
    assert f(FAKE, 0, 2, FAKE) == -1
    assert f(None, 4, 2, FAKE) == -1
    assert f(FAKE, 4, 2, None) == -1


def test_host_scratch_bytes(lib):
    f = lib.mla_host_scratch_bytes
    f.restype = ctypes.c_size_t
    f.argtypes = [ctypes.c_int] * 5
    lib.mla_workspace_bytes.restype = ctypes.c_size_t
    lib.mla_workspace_bytes.argtypes = [ctypes.c_int] * 4
    up = lambda x: (x + 255) // 256 * 256
    b, s_q, h_q, mb, parts = 128, 1, 128, 64, 76
    rows = b * s_q * h_q
    want = (up(rows * 576 * 2) + up(rows * 512 * 2) + up(rows * 4) + up(b * mb * 4) + up(b * 4)
            + MAX_CHUNKS * up(parts * 8 * 4) + MAX_CHUNKS * up((b + 1) * 4)
            + lib.mla_workspace_bytes(b, s_q, h_q, parts))
    assert f(b, s_q, h_q, mb, parts) == want
    assert f(0, 1, 128, 64, 76) == 0 and f(1, 1, 128, 0, 76) == 0 and f(1, 1, 128, 64, 0) == 0


def test_host_decode_checks_lengths_on_the_host(lib):
    """Lengths outside [0, max_blocks*64] are rejected before any CUDA call
    (the pipeline pointer is never dereferenced on that path); a length at the
    limit passes the check and only then needs the GPU (MLA_ERR_CUDA here)."""
    f = lib.mla_decode_host
    P, I, I64, SZ, F = ctypes.c_void_p, ctypes.c_int, ctypes.c_int64, ctypes.c_size_t, ctypes.c_float
    f.restype = ctypes.c_int32
    f.argtypes = [P, P, I, I, I, I, P, I64, I, I, I, P, I, P, I, I, F, I, P, P, I, P, SZ, P, P]

    def call(seqlens):
        sl = (ctypes.c_int32 * len(seqlens))(*seqlens)
        return f(FAKE, FAKE, len(seqlens), 1, 128, 576, FAKE, 10, 64, 1, 576, FAKE, 4, ctypes.addressof(sl),
                 512, 4, 0.04, 0, FAKE, FAKE, 0, FAKE, 1 << 40, FAKE, None)

    assert call([256, -1]) == -1
    assert call([257, 5]) == -1
    assert call([256, 0, 17]) == -4


def test_host_decode_rejects_null_pipeline(lib):
    f = lib.mla_decode_host
    P, I, I64, SZ, F = ctypes.c_void_p, ctypes.c_int, ctypes.c_int64, ctypes.c_size_t, ctypes.c_float
    f.restype = ctypes.c_int32
    f.argtypes = [P, P, I, I, I, I, P, I64, I, I, I, P, I, P, I, I, F, I, P, P, I, P, SZ, P, P]
    args = [None, FAKE, 2, 1, 128, 576, FAKE, 10, 64, 1, 576, FAKE, 4, FAKE, 512, 4, 0.04, 0, FAKE, FAKE, 0,
            FAKE, 1 << 40, FAKE, None]
    assert f(*args) == -1
    lib.mla_host_pipeline_destroy.restype = ctypes.c_int32
    lib.mla_host_pipeline_destroy.argtypes = [P]
    assert lib.mla_host_pipeline_destroy(None) == 0
    lib.mla_host_pipeline_create.restype = ctypes.c_int32
    lib.mla_host_pipeline_create.argtypes = [P]
    assert lib.mla_host_pipeline_create(None) == -1


def test_binding_fails_loudly_without_the_library(monkeypatch, tmp_path):
    """No CPU fallback: with the CUDA library missing, the binding raises
    instead of computing anything."""
    import torch

    from mla_decode_attention_03_gb300 import ops
    monkeypatch.setattr(ops, "LIB_PATH", tmp_path / "libmla_decode.so")
    monkeypatch.setattr(ops, "_lib", None)
    with pytest.raises(ops.MLAError, match="missing"):
        ops.load_library()
    with pytest.raises(ops.MLAError):
        ops.workspace_bytes(1, 1, 128, 4)
    with pytest.raises(ops.MLAError):
        ops.host_chunks(torch.tensor([64, 128], dtype=torch.int32))


# ------------------------------------------------------------ binding argument checks (no GPU reached)
def _io(b=4, s_q=1, h_q=128, mb=8):
    import torch
    return dict(q=torch.empty((b, s_q, h_q, 576), dtype=torch.bfloat16),
                block_table=torch.empty((b, mb), dtype=torch.int32),
                cache_seqlens=torch.empty((b,), dtype=torch.int32),
                out=torch.empty((b, s_q, h_q, 512), dtype=torch.bfloat16),
                lse=torch.empty((b, h_q, s_q), dtype=torch.float32))


@pytest.mark.parametrize("b,s_q,h_q,mb", [(128, 1, 128, 64), (128, 2, 128, 100), (6, 1, 128, 64), (1, 1, 16, 4),
                                          (16, 1, 16, 64), (9, 2, 128, 48), (6, 1, 64, 16)])
def test_check_io_accepts_the_shapes_the_library_is_called_with(b, s_q, h_q, mb):
    from mla_decode_attention_03_gb300 import ops
    a = _io(b, s_q, h_q, mb)
    ops._check_io(**a)
    ops._check_io(a["q"], a["block_table"], a["cache_seqlens"], None, None)


def test_check_io_refuses_what_would_be_read_or_written_out_of_bounds():
    import torch

    from mla_decode_attention_03_gb300 import ops
    bad = [
        ("block_table", torch.empty((3, 8), dtype=torch.int32)),        # fewer rows than sequences
        ("block_table", torch.empty((4, 8), dtype=torch.int64)),
        ("block_table", torch.empty((32,), dtype=torch.int32)),
        ("cache_seqlens", torch.empty((3,), dtype=torch.int32)),
        ("cache_seqlens", torch.empty((4, 1), dtype=torch.int32)),
        ("cache_seqlens", torch.empty((4,), dtype=torch.int64)),
        ("out", torch.empty((4, 1, 64, 512), dtype=torch.bfloat16)),    # too small
        ("out", torch.empty((4, 1, 128, 512), dtype=torch.float16)),
        ("out", torch.empty((4, 1, 512, 128), dtype=torch.bfloat16).transpose(2, 3)),  # not contiguous
        ("lse", torch.empty((4, 1, 128), dtype=torch.float32)),         # [b, s_q, h_q] instead of [b, h_q, s_q]
        ("lse", torch.empty((4, 128, 1), dtype=torch.float64)),
    ]
    for name, t in bad:
        a = _io()
        a[name] = t
        with pytest.raises(ops.MLAError):
            ops._check_io(**a)
    a = _io()
    a["q"] = a["q"][0]
    with pytest.raises(ops.MLAError):
        ops._check_io(**a)


def test_combine_and_copy_blocks_refuse_bad_shapes_before_the_library():
    import torch

    from mla_decode_attention_03_gb300 import ops
    a = _io()
    ns = torch.empty((5,), dtype=torch.int32)
    ws = torch.empty((1 << 20,), dtype=torch.uint8)
    with pytest.raises(ops.MLAError):
        ops.combine_splits(ns, ws, 4, a["out"], torch.empty((4, 1, 128), dtype=torch.float32))
    with pytest.raises(ops.MLAError):
        ops.combine_splits(torch.empty((4,), dtype=torch.int32), ws, 4, a["out"], a["lse"])
    with pytest.raises(ops.MLAError):
        ops.combine_splits(ns, torch.empty((16,), dtype=torch.uint8), 4, a["out"], a["lse"])
    with pytest.raises(ops.MLAError):
        ops.combine_splits(ns, ws, 4, a["out"][..., :256], a["lse"])
    cache = torch.empty((4, 64, 1, 576), dtype=torch.bfloat16)
    with pytest.raises(ops.MLAError, match="num_pairs, 2"):
        ops.copy_blocks([cache], torch.tensor([0, 1, 2, 3]))
