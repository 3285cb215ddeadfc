"""Seeded synthetic inputs for MLA decode over a paged latent KV cache.

This module only draws random numbers and lays them out; it holds none of the
attention arithmetic.  The CUDA path and the fp64 oracle both take their inputs
from here, so they see the same bytes.

The shapes follow the FlashMLA benchmark driven by the PAI tutorial
("云上玩转DeepSeek系列之五", section 4, compare_a): q[b, s_q, h_q, d] and a cache
of 64-token pages blocked_k[num_blocks, 64, h_kv, d] with d = 576 and dv = 512,
a block_table of int32 page ids and per-sequence cache_seqlens.  An entry may
be padded to 640 elements (the 256-byte aligned layout of vLLM PR #12676,
"Mem align KV caches for CUDA devices"); the pad is zero-filled as in that PR's
zeroed cache allocation, unless a test asks for poison.

Recipe (all draws from numpy's PCG64 `default_rng(seed)`, in this order):
  1. cache_seqlens, when the workload draws them;
  2. q ~ N(0, 1), rounded to bf16;
  3. the page permutation, when the workload permutes pages;
  4. cache entries ~ N(0, 1), rounded to bf16, drawn page by page;
  5. the "peaky" token slots, when asked (their whole entry is multiplied by 4,
     which is exact in bf16);
  6. poison for unused slots and the pad, when asked (finite +-1e4).
Pages are allocated only for the tokens a sequence holds; block_table entries
past a sequence's last page are -1 and must never be read.
"""
from __future__ import annotations

from dataclasses import dataclass, field

import numpy as np
import torch

D_QK = 576       # latent 512 + rope 64
D_V = 512
BLOCK_SIZE = 64
POISON = 1.0e4

# The five workloads, with the parameters their names stand for.
WORKLOADS = {
    "tiny": dict(b=1, s_q=1, h_q=16, h_kv=1, stride=576, causal=False),
    "v2lite": dict(b=16, s_q=1, h_q=16, h_kv=1, stride=640, causal=False),
    "bench": dict(b=128, s_q=1, h_q=128, h_kv=1, stride=576, causal=False),
    "mtp": dict(b=128, s_q=2, h_q=128, h_kv=1, stride=640, causal=True),
    "skewed": dict(b=64, s_q=1, h_q=128, h_kv=1, stride=640, causal=False),
}


@dataclass
class Workload:
    name: str
    q: torch.Tensor              # bf16 [b, s_q, h_q, 576]
    kcache_alloc: torch.Tensor   # bf16 [num_blocks, 64, h_kv, stride] (whole allocation)
    block_table: torch.Tensor    # int32 [b, max_blocks_per_seq]
    cache_seqlens: torch.Tensor  # int32 [b]
    s_q: int
    h_q: int
    h_kv: int
    stride: int
    causal: bool
    softmax_scale: float = D_QK ** -0.5
    dv: int = D_V
    extra: dict = field(default_factory=dict)

    @property
    def b(self) -> int:
        return self.q.shape[0]

    @property
    def kcache(self) -> torch.Tensor:
        """The [num_blocks, 64, h_kv, 576] view of the (possibly padded) allocation."""
        return self.kcache_alloc[..., :D_QK]

    @property
    def num_blocks(self) -> int:
        return self.kcache_alloc.shape[0]

    def numpy_bits(self):
        """(q, kcache_alloc) as uint16 bf16 bit patterns, for the oracle."""
        qb = self.q.contiguous().view(torch.int16).numpy().view(np.uint16)
        kb = self.kcache_alloc.contiguous().view(torch.int16).numpy().view(np.uint16)
        return qb, kb


def _bf16_normal(rng: np.random.Generator, shape) -> torch.Tensor:
    x = rng.standard_normal(shape, dtype=np.float32)
    return torch.from_numpy(x).to(torch.bfloat16)


def make(b: int, s_q: int, h_q: int, h_kv: int, cache_seqlens, *, stride: int = 576,
         causal: bool = False, seed: int = 0, permute: bool = True, peaky_frac: float = 0.0,
         poison: bool = False, width_pages: int | None = None, name: str = "custom",
         softmax_scale: float = D_QK ** -0.5) -> Workload:
    """General generator.  `cache_seqlens` is a sequence of ints or a callable
    taking the rng and returning them (so that they are drawn first)."""
    rng = np.random.default_rng(seed)
    if callable(cache_seqlens):
        cache_seqlens = cache_seqlens(rng)
    seqlens = np.asarray(cache_seqlens, dtype=np.int64).reshape(b)
    assert (seqlens >= 0).all()
    n_pages = (seqlens + BLOCK_SIZE - 1) // BLOCK_SIZE
    if width_pages is None:
        # the benchmark pads the longest sequence to a multiple of 256 tokens
        max_pad = int(-(-max(int(seqlens.max()), 1) // 256) * 256)
        width_pages = max_pad // BLOCK_SIZE
    assert int(n_pages.max(initial=0)) <= width_pages
    num_blocks = max(int(n_pages.sum()), 1)

    q = _bf16_normal(rng, (b, s_q, h_q, D_QK))

    ids = rng.permutation(num_blocks) if permute else np.arange(num_blocks)
    table = np.full((b, width_pages), -1, dtype=np.int32)
    pos = 0
    for i in range(b):
        table[i, : n_pages[i]] = ids[pos: pos + n_pages[i]]
        pos += int(n_pages[i])

    kc = torch.zeros((num_blocks, BLOCK_SIZE, h_kv, stride), dtype=torch.bfloat16)
    chunk = max(1, (1 << 24) // (BLOCK_SIZE * h_kv * D_QK))
    for p0 in range(0, num_blocks, chunk):
        p1 = min(num_blocks, p0 + chunk)
        kc[p0:p1, :, :, :D_QK] = _bf16_normal(rng, (p1 - p0, BLOCK_SIZE, h_kv, D_QK))

    extra = {}
    if peaky_frac > 0.0:
        n_slots = num_blocks * BLOCK_SIZE
        hot = rng.choice(n_slots, size=max(1, int(round(peaky_frac * n_slots))), replace=False)
        flat = kc.view(n_slots, h_kv, stride)
        flat[torch.from_numpy(np.sort(hot))] *= 4
        extra["peaky_slots"] = np.sort(hot)

    if poison:
        sign = torch.from_numpy(np.where(rng.random((num_blocks, BLOCK_SIZE)) < 0.5, -1.0, 1.0)
                                .astype(np.float32)).to(torch.bfloat16)
        if stride > D_QK:
            kc[..., D_QK:] = (POISON * sign)[:, :, None, None]
        for i in range(b):
            L = int(seqlens[i])
            if L % BLOCK_SIZE:
                page = int(table[i, L // BLOCK_SIZE])
                kc[page, L % BLOCK_SIZE:, :, :] = (POISON * sign[page, L % BLOCK_SIZE:])[:, None, None]

    return Workload(name=name, q=q, kcache_alloc=kc, block_table=torch.from_numpy(table),
                    cache_seqlens=torch.from_numpy(seqlens.astype(np.int32)), s_q=s_q, h_q=h_q,
                    h_kv=h_kv, stride=stride, causal=causal, softmax_scale=softmax_scale,
                    extra=extra)


def named(name: str, *, seed: int = 0, stride: int | None = None, poison: bool = False) -> Workload:
    """One of the five named workloads:

    tiny    b=1,   s_q=1, h_q=16,  L=[256],                     stride 576, pages in order
    v2lite  b=16,  s_q=1, h_q=16,  L ~ U{1024..4096},           stride 640, pages permuted
    bench   b=128, s_q=1, h_q=128, L = 4096 for all,            stride 576 (or 640), in order
    mtp     b=128, s_q=2, h_q=128, causal, L = clip(round(N(4096, 1024)), 256, 8192),
                                                                stride 640, pages permuted
    skewed  b=64,  s_q=1, h_q=128, L = [65536, 65536] + 62 x U{64..1024}, stride 640,
            pages permuted, 1% of token slots scaled by 4
    All with h_kv = 1, d = 576, dv = 512, 64-token pages, scale 576**-0.5.
    """
    p = dict(WORKLOADS[name])
    if stride is not None:
        p["stride"] = stride
    b = p.pop("b")
    s_q, h_q, h_kv = p.pop("s_q"), p.pop("h_q"), p.pop("h_kv")
    if name == "tiny":
        return make(b, s_q, h_q, h_kv, [256], seed=seed, permute=False, poison=poison,
                    name=name, **p)
    if name == "v2lite":
        return make(b, s_q, h_q, h_kv, lambda r: r.integers(1024, 4096, size=b, endpoint=True),
                    seed=seed, permute=True, poison=poison, name=name, **p)
    if name == "bench":
        return make(b, s_q, h_q, h_kv, [4096] * b, seed=seed, permute=False, poison=poison,
                    name=name, **p)
    if name == "mtp":
        return make(b, s_q, h_q, h_kv,
                    lambda r: np.clip(np.round(r.normal(4096.0, 1024.0, size=b)), 256, 8192),
                    seed=seed, permute=True, poison=poison, name=name, **p)
    if name == "skewed":
        return make(b, s_q, h_q, h_kv,
                    lambda r: np.concatenate([[65536, 65536],
                                              r.integers(64, 1024, size=b - 2, endpoint=True)]),
                    seed=seed, permute=True, peaky_frac=0.01, poison=poison, name=name, **p)
    raise KeyError(name)
