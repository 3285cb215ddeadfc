"""Cache maintenance next to the decode: writing new tokens into the paged
latent cache and copy_blocks_mla (vLLM PR #12676).

CPU: the oracle's two operations are pinned by read-back, by what they must
leave untouched, and by a round trip through the decode oracle (attention over
tokens written into a permuted paged cache equals attention over the same
tokens laid out directly).  GPU: the CUDA kernels must equal the oracle bit for
bit (they only move bytes).
"""
import numpy as np
import pytest
import torch

import oracle
from oracle import cache_ops
from mla_decode_attention_03_gb300 import workloads as W

RNG = np.random.default_rng(77)


def _bits(shape):
    x = torch.from_numpy(RNG.standard_normal(shape, dtype=np.float32)).to(torch.bfloat16)
    return x.view(torch.int16).numpy().view(np.uint16)


def _case(num_blocks=6, stride=640, tokens=200):
    kc = _bits((num_blocks, 64, 1, stride))
    kv_c, k_pe = _bits((tokens, 512)), _bits((tokens, 64))
    slots = RNG.choice(num_blocks * 64, size=tokens, replace=False).astype(np.int64)
    slots[RNG.random(tokens) < 0.1] = -1  # padding tokens
    return kc, kv_c, k_pe, slots


def test_write_cache_reads_back_and_leaves_the_rest():
    kc, kv_c, k_pe, slots = _case()
    out = cache_ops.write_cache(kc, kv_c, k_pe, slots)
    written = np.zeros(kc.shape[:2], bool)
    for t, s in enumerate(slots):
        if s < 0:
            continue
        p, o = divmod(int(s), 64)
        assert np.array_equal(out[p, o, 0, :512], kv_c[t])
        assert np.array_equal(out[p, o, 0, 512:576], k_pe[t])
        written[p, o] = True
    assert np.array_equal(out[~written], kc[~written])       # other entries untouched
    assert np.array_equal(out[..., 576:], kc[..., 576:])     # the pad is never written


def test_write_cache_then_decode_equals_direct_layout():
    # 130 tokens of one sequence written into randomly chosen physical pages
    T, nb = 130, 5
    kv_c, k_pe = _bits((T, 512)), _bits((T, 64))
    pages = RNG.permutation(nb)[:3]
    slots = np.array([pages[t // 64] * 64 + t % 64 for t in range(T)], dtype=np.int64)
    kc = cache_ops.write_cache(np.zeros((nb, 64, 1, 640), np.uint16), kv_c, k_pe, slots)
    q = _bits((1, 1, 4, 576))
    bt = np.full((1, 4), -1, np.int32)
    bt[0, :3] = pages
    o1, l1 = oracle.decode(q, kc, bt, np.array([T], np.int32), softmax_scale=576 ** -0.5)
    direct = np.zeros((3, 64, 1, 576), np.uint16)
    direct.reshape(192, 576)[:T] = np.concatenate([kv_c, k_pe], axis=1)
    o2, l2 = oracle.decode(q, direct, np.arange(4, dtype=np.int32)[None, :3].copy(),
                           np.array([T], np.int32), softmax_scale=576 ** -0.5)
    assert np.array_equal(o1, o2) and np.array_equal(l1, l2)


def test_copy_blocks_copies_sources_and_nothing_else():
    caches = [_bits((8, 64, 1, 640)) for _ in range(3)]
    mapping = np.array([[0, 5], [3, 1], [7, 6]], np.int64)
    out = cache_ops.copy_blocks(caches, mapping)
    for c, o in zip(caches, out):
        for s, d in mapping:
            assert np.array_equal(o[d], c[s])
        untouched = [p for p in range(8) if p not in mapping[:, 1]]
        assert np.array_equal(o[untouched], c[untouched])


def test_write_cache_rejects_slots_outside_the_cache():
    kc, kv_c, k_pe, slots = _case()
    slots[0] = kc.shape[0] * 64
    with pytest.raises(ValueError):
        cache_ops.write_cache(kc, kv_c, k_pe, slots)


# ------------------------------------------------------------------ GPU
@pytest.mark.gpu
@pytest.mark.parametrize("stride", [576, 640])
def test_gpu_write_cache_matches_oracle(stride):
    from mla_decode_attention_03_gb300 import ops
    kc, kv_c, k_pe, slots = _case(stride=stride, tokens=300, num_blocks=8)
    want = cache_ops.write_cache(kc, kv_c, k_pe, slots)
    alloc = torch.from_numpy(kc.view(np.int16)).cuda()
    # kv_c rows handed over with a padded row stride, as a slice of a wider buffer
    wide = torch.zeros((300, 640), dtype=torch.int16)
    wide[:, :512] = torch.from_numpy(kv_c.view(np.int16))
    kv = wide.cuda().view(torch.bfloat16)[:, :512]
    pe = torch.from_numpy(k_pe.view(np.int16)).cuda().view(torch.bfloat16)
    status = ops.new_status()
    ops.write_cache(kv, pe, torch.from_numpy(slots).cuda(), alloc.view(torch.bfloat16)[..., :576], status)
    torch.cuda.synchronize()
    ops.check_status(status)
    assert np.array_equal(alloc.cpu().numpy().view(np.uint16), want)


@pytest.mark.gpu
def test_gpu_copy_blocks_matches_oracle():
    from mla_decode_attention_03_gb300 import ops
    caches = [_bits((16, 64, 1, 640)) for _ in range(4)]
    mapping = np.array([[0, 9], [3, 1], [7, 6], [15, 2]], np.int64)
    want = cache_ops.copy_blocks(caches, mapping)
    dev = [torch.from_numpy(c.view(np.int16)).cuda() for c in caches]
    status = ops.new_status()
    ops.copy_blocks([d.view(torch.bfloat16)[..., :576] for d in dev], torch.from_numpy(mapping), status)
    torch.cuda.synchronize()
    ops.check_status(status)
    for d, w in zip(dev, want):
        assert np.array_equal(d.cpu().numpy().view(np.uint16), w)


@pytest.mark.gpu
def test_gpu_written_cache_decodes_like_the_oracle():
    """Tokens written by the kernel into a 640-stride cache, then decoded by the
    decode kernel, match the fp64 oracle on the written cache."""
    from mla_decode_attention_03_gb300 import ops
    from tests._gpu_helpers import all_rows, assert_matches, run_gpu
    T, nb = 700, 16
    kv_c, k_pe = _bits((T, 512)), _bits((T, 64))
    pages = RNG.permutation(nb)[:11]
    slots = np.array([pages[t // 64] * 64 + t % 64 for t in range(T)], dtype=np.int64)
    alloc = torch.zeros((nb, 64, 1, 640), dtype=torch.int16, device="cuda")
    ops.write_cache(torch.from_numpy(kv_c.view(np.int16)).cuda().view(torch.bfloat16),
                    torch.from_numpy(k_pe.view(np.int16)).cuda().view(torch.bfloat16),
                    torch.from_numpy(slots).cuda(), alloc.view(torch.bfloat16)[..., :576])
    torch.cuda.synchronize()
    bt = np.full((1, 11), -1, np.int32)
    bt[0] = pages
    w = W.Workload(name="written", q=W.make(1, 1, 128, 1, [1], seed=78).q,
                   kcache_alloc=alloc.cpu().view(torch.bfloat16), block_table=torch.from_numpy(bt),
                   cache_seqlens=torch.tensor([T], dtype=torch.int32), s_q=1, h_q=128, h_kv=1,
                   stride=640, causal=False)
    out, lse, _, _ = run_gpu(w, parts=3)
    assert_matches(w, out, lse, all_rows(w))
