"""fp64 CPU oracle for MLA decode over a paged latent KV cache.

TEST INFRASTRUCTURE ONLY: imported by the tests, by the package smoke check
and by the benchmark's CPU-baseline and reference legs.  The product path (the
CUDA library and its Python binding) never imports, links or calls anything
here, and nothing here imports the product.

The arithmetic lives in ``mla_oracle.c`` (plain C, fp64); this module compiles
it with gcc on first use and marshals NumPy arrays into it.  What it computes is
the definition of ``flash_mla_with_kvcache`` as exercised by the compare_a
benchmark of the PAI FlashMLA tutorial (section 4, "不同 MLA 实现的简易性能比较"),
read through the paged cache layout of vLLM PR #12676: see the header of
``mla_oracle.c`` for the formula and the readings taken where the pages are
silent.

Parity status: pinned (tests/test_oracle.py).
"""
from __future__ import annotations

import ctypes
import os
import subprocess
from pathlib import Path

import numpy as np

_HERE = Path(__file__).resolve().parent
_SRC = _HERE / "mla_oracle.c"
_BUILD = _HERE / "_build"
_LIB_PATH = _BUILD / "libmla_oracle.so"
_lib = None

# Planted mistakes understood by the C code (used only by the pin tests).
MUTATIONS = {
    "drop_last_token": 1,
    "causal_off_by_one": 2,
    "v_offset": 3,
    "no_scale": 4,
    "ignore_block_table": 5,
    "lse_base2": 6,
    "head_group": 7,
    "rope_dropped": 8,
}


def build(force: bool = False) -> Path:
    """Compile the oracle into oracle/_build/libmla_oracle.so (gcc, fp64, no FMA contraction)."""
    _BUILD.mkdir(exist_ok=True)
    if force or not _LIB_PATH.exists() or _LIB_PATH.stat().st_mtime < _SRC.stat().st_mtime:
        tmp = _LIB_PATH.with_suffix(f".{os.getpid()}.tmp")
        subprocess.check_call([
            "gcc", "-O2", "-std=c11", "-fPIC", "-shared", "-pthread",
            "-ffp-contract=off", str(_SRC), "-o", str(tmp), "-lm",
        ])
        os.replace(tmp, _LIB_PATH)
    return _LIB_PATH


def _load():
    global _lib
    if _lib is None:
        lib = ctypes.CDLL(str(build()))
        fn = lib.mla_oracle_rows_mutant
        fn.restype = ctypes.c_int
        P = ctypes.c_void_p
        fn.argtypes = [P, ctypes.c_int, ctypes.c_int, ctypes.c_int, ctypes.c_int,
                       P, ctypes.c_int64, ctypes.c_int, ctypes.c_int, ctypes.c_int,
                       P, ctypes.c_int, P, ctypes.c_int, ctypes.c_double, ctypes.c_int,
                       P, ctypes.c_int64, P, P, ctypes.c_int, ctypes.c_int]
        _lib = lib
    return _lib


def host_threads() -> int:
    """Host cores this process may run on."""
    try:
        return len(os.sched_getaffinity(0))
    except AttributeError:  # pragma: no cover
        return os.cpu_count() or 1


def decode_rows(q_bits, kcache_bits, block_table, cache_seqlens, rows, *, dv=512,
                softmax_scale, causal=False, threads=None, mutation=0):
    """Oracle values for selected output rows.

    q_bits:       uint16 [b, s_q, h_q, d]   bf16 bit patterns, contiguous
    kcache_bits:  uint16 [num_blocks, block_size, h_kv, stride]  (stride >= d;
                  elements past d are padding and never read)
    block_table:  int32 [b, max_blocks_per_seq]
    cache_seqlens:int32 [b]
    rows:         int32 [n, 3] of (i, j, h)
    Returns (out float64 [n, dv], lse float64 [n]); lse is a natural log.
    """
    lib = _load()
    q = np.ascontiguousarray(q_bits, dtype=np.uint16)
    kc = np.ascontiguousarray(kcache_bits, dtype=np.uint16)
    bt = np.ascontiguousarray(block_table, dtype=np.int32)
    sl = np.ascontiguousarray(cache_seqlens, dtype=np.int32)
    rows = np.ascontiguousarray(rows, dtype=np.int32).reshape(-1, 3)
    b, s_q, h_q, d = q.shape
    num_blocks, block_size, h_kv, stride = kc.shape
    assert bt.ndim == 2 and bt.shape[0] == b and sl.shape == (b,)
    n = rows.shape[0]
    out = np.zeros((n, dv), dtype=np.float64)
    lse = np.zeros((n,), dtype=np.float64)
    threads = host_threads() if threads is None else int(threads)
    rc = lib.mla_oracle_rows_mutant(
        q.ctypes.data, b, s_q, h_q, d, kc.ctypes.data, num_blocks, block_size, h_kv, stride,
        bt.ctypes.data, bt.shape[1], sl.ctypes.data, dv, float(softmax_scale), int(bool(causal)),
        rows.ctypes.data, n, out.ctypes.data, lse.ctypes.data, threads, int(mutation))
    if rc != 0:
        raise ValueError(f"oracle rejected its inputs (code {rc})")
    return out, lse


def all_rows(b: int, s_q: int, h_q: int) -> np.ndarray:
    """Every (i, j, h) triple, in the order of out[b, s_q, h_q]."""
    i, j, h = np.meshgrid(np.arange(b), np.arange(s_q), np.arange(h_q), indexing="ij")
    return np.stack([i.ravel(), j.ravel(), h.ravel()], axis=1).astype(np.int32)


def decode(q_bits, kcache_bits, block_table, cache_seqlens, *, dv=512, softmax_scale,
           causal=False, threads=None, mutation=0):
    """Full oracle output: out float64 [b, s_q, h_q, dv], lse float64 [b, h_q, s_q]."""
    b, s_q, h_q, _ = q_bits.shape
    out, lse = decode_rows(q_bits, kcache_bits, block_table, cache_seqlens,
                           all_rows(b, s_q, h_q), dv=dv, softmax_scale=softmax_scale,
                           causal=causal, threads=threads, mutation=mutation)
    return out.reshape(b, s_q, h_q, dv), lse.reshape(b, s_q, h_q).transpose(0, 2, 1).copy()
