"""CPU oracle for the two cache-maintenance operations next to MLA decode.

TEST INFRASTRUCTURE ONLY (see oracle/__init__.py): the product path never
imports this module.

* write_cache: puts new tokens into the paged latent cache -- entry
  (page, slot) = (s // block_size, s % block_size) for slot id s =
  slot_mapping[t] receives the 512 latent values kv_c[t] followed by the 64
  rope values k_pe[t]; negative slot ids are skipped (padding tokens).  The
  entry layout is that of the cache the decode reads: 576 meaningful elements
  per entry at a stride of 576, or 640 for the 256-byte aligned layout of vLLM
  PR #12676 ("Mem align KV caches for CUDA devices"); the pad is not touched.
* copy_blocks: the copy_blocks_mla operation that PR adds
  (`copy_blocks_mla(kv_caches, block_mapping)`): for every layer's cache and
  every (src, dst) pair, page dst becomes a copy of page src (the whole page,
  pad included).  Every source is read before any destination is written.

Both are plain NumPy over uint16 bf16 bit patterns (copies are exact).
Parity status: pinned by tests/test_cache_ops.py (read-back, untouched entries,
and a round trip through the decode oracle).
"""
from __future__ import annotations

import numpy as np

LATENT, ROPE = 512, 64


def write_cache(kcache_bits: np.ndarray, kv_c_bits: np.ndarray, k_pe_bits: np.ndarray,
                slot_mapping: np.ndarray) -> np.ndarray:
    """kcache_bits uint16 [num_blocks, block_size, 1, stride] (returned updated copy),
    kv_c_bits uint16 [T, 512], k_pe_bits uint16 [T, 64], slot_mapping int64 [T]."""
    out = kcache_bits.copy()
    num_blocks, block_size = out.shape[0], out.shape[1]
    for t, s in enumerate(np.asarray(slot_mapping, dtype=np.int64)):
        if s < 0:
            continue
        if s >= num_blocks * block_size:
            raise ValueError(f"slot {s} outside the cache")
        page, slot = divmod(int(s), block_size)
        out[page, slot, 0, :LATENT] = kv_c_bits[t]
        out[page, slot, 0, LATENT:LATENT + ROPE] = k_pe_bits[t]
    return out


def copy_blocks(kcaches_bits: list, block_mapping: np.ndarray) -> list:
    """kcaches_bits: list (one per layer) of uint16 [num_blocks, block_size, 1, stride];
    block_mapping int64 [n, 2] of (src, dst).  Returns updated copies."""
    out = []
    pairs = np.asarray(block_mapping, dtype=np.int64).reshape(-1, 2)
    for cache in kcaches_bits:
        snapshot = cache.copy()
        upd = cache.copy()
        for src, dst in pairs:
            upd[dst] = snapshot[src]
        out.append(upd)
    return out
