"""GPU parity: the CUDA path through the C ABI against the fp64 oracle.

Every test compares every output row element by element: small shapes that
span several pages, ragged tails and the degenerate cases, and the five named
workloads at their full sizes in the launch configuration the benchmark times
(the recommended number of parts).
Tolerance: |d out| <= 1e-2 + 2e-2 |out_oracle| and |d lse| <= 1e-3.
"""
import zlib

import numpy as np
import pytest
import torch

from mla_decode_attention_03_gb300 import ops
from mla_decode_attention_03_gb300 import workloads as W
from tests._gpu_helpers import all_rows, assert_matches, run_gpu, sample_rows, to_device

pytestmark = pytest.mark.gpu

SMALL = [
    # id, b, s_q, h_q, h_kv, seqlens, stride, causal, parts
    ("ragged_tails", 5, 1, 128, 1, [1, 63, 64, 65, 700], 576, False, None),
    ("ragged_tails_split", 5, 1, 128, 1, [1, 63, 64, 65, 700], 576, False, 3),
    ("causal_two_tiles", 3, 2, 128, 1, [1, 2, 333], 640, True, None),
    ("causal_64_heads", 4, 2, 64, 1, [100, 200, 64, 5], 640, True, 2),
    ("kv_groups", 2, 1, 16, 2, [300, 17], 576, False, None),
    ("three_queries", 3, 3, 32, 1, [130, 3, 64], 576, True, 4),
    ("empty_sequences", 3, 1, 128, 1, [0, 100, 0], 640, False, None),
    ("long_split_many", 2, 1, 128, 1, [5000, 3000], 640, False, None),
    ("h16_many_short", 40, 1, 16, 1, "short", 576, False, None),
    # the last row tile only partly holds query positions (64 of 128 rows; 48
    # of 96 with 48 heads): only those rows are exchanged between the CTAs
    ("partial_last_tile", 3, 3, 64, 1, [100, 300, 65], 640, True, None),
    ("h48_partial_last_tile", 2, 3, 48, 1, [200, 77], 576, True, 3),
    # ~10 sequences per part: a segment boundary (Q staging, epilogue) every
    # few pages, and more sequences than the scheduler block has threads
    ("many_segments", 700, 1, 16, 1, "short", 640, False, None),
    ("many_segments_128_heads", 300, 1, 128, 1, "short", 576, False, None),
    # tiles of at most 16 rows (the 16-row kernel): query positions x heads
    # per KV head = 16, 12 and 4 rows; causal rows with nothing visible
    # (L=1, 2 with several positions); split sequences; four KV heads
    ("rows16_causal_two_positions", 3, 2, 8, 1, [1, 2, 333], 640, True, None),
    ("rows16_causal_four_positions_split", 3, 4, 4, 1, [65, 130, 7], 576, True, 3),
    ("rows12_causal_three_positions", 2, 3, 4, 1, [200, 64], 640, True, None),
    ("rows4_four_kv_heads_split", 2, 1, 16, 4, [150, 90], 576, False, 2),
]


@pytest.mark.parametrize("case", SMALL, ids=[c[0] for c in SMALL])
def test_small_all_rows(case):
    name, b, s_q, h_q, h_kv, sl, stride, causal, parts = case
    if sl == "short":
        sl = list(np.random.default_rng(3).integers(1, 200, size=b))
    w = W.make(b, s_q, h_q, h_kv, sl, stride=stride, causal=causal, seed=zlib.crc32(name.encode()) % 1000,
               poison=True)
    out, lse, _, _ = run_gpu(w, parts=parts)
    assert_matches(w, out, lse, all_rows(w))


@pytest.mark.parametrize("name", ["tiny", "v2lite"])
def test_named_small_all_rows(name):
    w = W.named(name)
    out, lse, _, _ = run_gpu(w)
    assert_matches(w, out, lse, all_rows(w))


@pytest.mark.parametrize("name,stride", [("bench", 576), ("bench", 640), ("mtp", None), ("skewed", None)])
def test_named_full_size_all_rows(name, stride):
    w = W.named(name, stride=stride)
    out, lse, _, nsplit = run_gpu(w)
    assert_matches(w, out, lse, all_rows(w))


# Behaviour tests run on both kernels: 128 heads per KV head (the 128-row
# cluster kernel) and 16 (the 16-row kernel; 8 heads when s_q = 2).
KERNEL_HEADS = [128, 16]


@pytest.mark.parametrize("h_q", KERNEL_HEADS)
def test_lazy_rescale_every_page(h_q):
    """The running max is moved (and O and the row sums rescaled) only when it
    grows by more than 8 log2 units (the 16-row kernel rescales on every page).  Here one key per page climbs by about 9.6
    log2 units over the previous page's (q has 4 in dim 0 for every head, the
    climbing key 40*(p+1) there), so the rescale runs on nearly every page of
    every row, while the other keys of earlier pages still carry weight that a
    wrong rescale factor would distort by 2^9.  Sequences are cut into several
    pieces so the merge of rescaled pieces is covered too."""
    lens = [6 * 64, 5 * 64 - 17, 7 * 64 + 3, 64]
    w = W.make(len(lens), 1, h_q, 1, lens, stride=640, seed=27)
    w.q[..., 0] = 4.0
    bt = w.block_table.numpy()
    for i, L in enumerate(lens):
        for p in range(-(-L // 64)):
            tok = (5 + 7 * p) % min(64, L - 64 * p)  # a visible slot of page p
            w.kcache_alloc[int(bt[i, p]), tok, 0, 0] = 40.0 * (p + 1)
    for parts in (None, 9):
        out, lse, _, _ = run_gpu(w, parts=parts)
        assert_matches(w, out, lse, all_rows(w))


@pytest.mark.parametrize("h_q", KERNEL_HEADS)
def test_negative_length_reported_and_treated_as_empty(h_q):
    """A negative cache_seqlens entry is outside the contract; the scheduler
    reports MLA_ERR_BAD_SEQLEN in the status word, the decode treats that
    sequence as empty (no page of it is read), and the context stays usable."""
    w = W.make(3, 1, h_q, 1, [200, 64, 300], seed=26)
    dev = to_device(w)
    sl = dev["cache_seqlens"].clone()
    sl[1] = -5
    status = ops.new_status()
    meta, nsplit = ops.get_mla_metadata(sl, 4, status)
    out, lse = ops.mla_decode_with_kvcache(dev["q"], dev["kcache"], dev["block_table"], sl, meta, nsplit,
                                           w.softmax_scale, False, status=status)
    torch.cuda.synchronize()
    assert int(status.item()) == -7
    assert torch.all(out[1] == 0) and torch.all(torch.isneginf(lse[1]))
    rows = all_rows(w)
    rows = rows[rows[:, 0] != 1]
    assert_matches(w, out, lse, rows)
    w_ok = W.make(1, 1, 16, 1, [64], seed=25)
    out, lse, _, _ = run_gpu(w_ok)
    assert_matches(w_ok, out, lse, all_rows(w_ok))


@pytest.mark.parametrize("h_q", KERNEL_HEADS)
def test_stride_576_and_640_identical(h_q):
    w640 = W.make(6, 1, h_q, 1, [700, 64, 1, 129, 1000, 333], stride=640, seed=21, poison=True)
    w576 = W.Workload(**{**w640.__dict__, "kcache_alloc": w640.kcache_alloc[..., :576].contiguous(),
                         "stride": 576})
    o1, l1, _, _ = run_gpu(w640, parts=5)
    o2, l2, _, _ = run_gpu(w576, parts=5)
    assert torch.equal(o1, o2) and torch.equal(l1, l2)


@pytest.mark.parametrize("h_q", KERNEL_HEADS)
@pytest.mark.parametrize("causal,s_q", [(False, 1), (True, 2)])
def test_repeated_runs_bitwise_identical(causal, s_q, h_q):
    """Many short segments (1- and 2-page sequences, parts that cut sequences)
    stress every hand-off between the kernel's warp roles; any race shows up as
    a run that differs from the first one."""
    lens = [700, 64, 3000, 1, 129, 4096, 65, 128, 2, 900]
    heads = h_q if h_q == 128 else 16 // s_q
    w = W.make(len(lens), s_q, heads, 1, lens, causal=causal, stride=640, seed=23)
    first = run_gpu(w, parts=11)[:2]
    for _ in range(12):
        o, l = run_gpu(w, parts=11)[:2]
        assert torch.equal(o, first[0]) and torch.equal(l, first[1])


@pytest.mark.parametrize("h_q", KERNEL_HEADS)
def test_many_reruns_bitwise_identical(h_q):
    """A race between warp roles of the two CTAs of a cluster (an exchange slot
    returned to the peer before every load of it was ordered) showed up in
    about one run in 300 of this short-segment, poisoned-padding workload; 400
    back-to-back runs on the same inputs must all equal the first."""
    w = W.make(6, 1, h_q, 1, [700, 64, 1, 129, 1000, 333], stride=640, seed=21, poison=True)
    dev = to_device(w)
    status = ops.new_status()
    meta, nsplit = ops.get_mla_metadata(dev["cache_seqlens"], 5, status)
    args = (dev["q"], dev["kcache"], dev["block_table"], dev["cache_seqlens"], meta, nsplit,
            w.softmax_scale, w.causal)
    first = ops.mla_decode_with_kvcache(*args, status=status)
    differ = 0
    for _ in range(400):
        o, l = ops.mla_decode_with_kvcache(*args, status=status)
        differ += int(not (torch.equal(o, first[0]) and torch.equal(l, first[1])))
    torch.cuda.synchronize()
    ops.check_status(status)
    assert differ == 0


@pytest.mark.parametrize("h_q", [128, 8])
def test_page_permutation_identical(h_q):
    w = W.make(4, 2, h_q, 1, [300, 129, 64, 1000], causal=True, seed=22, permute=False)
    o1, l1, _, _ = run_gpu(w, parts=4)
    perm = torch.from_numpy(np.random.default_rng(5).permutation(w.num_blocks))
    kc2 = torch.empty_like(w.kcache_alloc)
    kc2[perm] = w.kcache_alloc
    bt = w.block_table.clone()
    bt[bt >= 0] = perm[bt[bt >= 0].long()].int()
    w2 = W.Workload(**{**w.__dict__, "kcache_alloc": kc2, "block_table": bt})
    o2, l2, _, _ = run_gpu(w2, parts=4)
    assert torch.equal(o1, o2) and torch.equal(l1, l2)


@pytest.mark.parametrize("h_q", KERNEL_HEADS)
@pytest.mark.parametrize("parts", [1, 2, 9, 150])
def test_split_count_invariance(parts, h_q):
    w = W.make(3, 1, h_q, 1, [2000, 513, 4096], stride=640, seed=23)
    out, lse, meta, nsplit = run_gpu(w, parts=parts)
    assert_matches(w, out, lse, all_rows(w))


@pytest.mark.parametrize("h_q", KERNEL_HEADS)
def test_bad_block_id_reported_not_faulted(h_q):
    w = W.make(2, 1, h_q, 1, [200, 100], seed=24)
    w.block_table[1, 0] = w.num_blocks + 5  # outside the cache
    dev = to_device(w)
    status = ops.new_status()
    meta, nsplit = ops.get_mla_metadata(dev["cache_seqlens"], 4, status)
    ops.mla_decode_with_kvcache(dev["q"], dev["kcache"], dev["block_table"], dev["cache_seqlens"],
                                meta, nsplit, w.softmax_scale, False, status=status)
    torch.cuda.synchronize()
    assert int(status.item()) == -5
    # the context is still usable
    w_ok = W.make(1, 1, 16, 1, [64], seed=25)
    out, lse, _, _ = run_gpu(w_ok)
    assert_matches(w_ok, out, lse, all_rows(w_ok))


def test_metadata_covers_every_page_once():
    from tests.test_scheduler import check_schedule
    sl = np.concatenate([[65536, 65536], np.random.default_rng(2).integers(64, 1024, 62)]).astype(np.int32)
    for parts in (1, 7, 76, 200):
        meta, nsplit = ops.get_mla_metadata(torch.from_numpy(sl).cuda(), parts)
        check_schedule(sl, parts, meta.cpu().numpy(), nsplit.cpu().numpy())


def test_num_parts_follows_the_kernel():
    """Tiles of at most 16 rows run one CTA per part and KV head (one per SM),
    larger tiles one 2-CTA cluster per part, row tile and KV head."""
    sms = torch.cuda.get_device_properties(0).multi_processor_count
    small = ops.num_parts(1, 16, 1)
    big = ops.num_parts(1, 128, 1)
    assert small == sms and big == sms // 2
    assert ops.num_parts(1, 16, 2) == sms // 2        # 8 heads per KV head, 2 KV heads
    assert ops.num_parts(2, 8, 1) == sms              # 2 positions x 8 heads = 16 rows
    assert ops.num_parts(2, 128, 1) == big // 2       # two 128-row tiles
    assert ops.num_parts(1, 32, 1) == big             # 32 rows: the cluster kernel


@pytest.mark.parametrize("h_q", KERNEL_HEADS)
def test_heads_identical_and_permuted(h_q):
    """Two identical query heads give bit-identical outputs, and permuting the
    heads permutes the outputs: bit for bit on the 16-row kernel (every row
    takes the same steps); to the tolerance on the cluster kernel, whose
    low-part pass is asked for by a warp of 16 rows for all of them, so a row
    moved to another warp may take it where it did not before."""
    w = W.make(3, 1, h_q, 1, [700, 77, 1500], stride=640, seed=41)
    w.q[:, :, 3] = w.q[:, :, 1]
    o, l, _, _ = run_gpu(w, parts=7)
    assert torch.equal(o[:, :, 3], o[:, :, 1]) and torch.equal(l[:, 3], l[:, 1])
    perm = torch.from_numpy(np.random.default_rng(6).permutation(h_q))
    w2 = W.Workload(**{**w.__dict__, "q": w.q[:, :, perm].contiguous()})
    o2, l2, _, _ = run_gpu(w2, parts=7)
    po, pl = o[:, :, perm.to(o.device)], l[:, perm.to(l.device)]
    if h_q <= 16:
        assert torch.equal(o2, po) and torch.equal(l2, pl)
    else:
        ref = po.float()
        assert torch.all((o2.float() - ref).abs() <= 1e-2 + 2e-2 * ref.abs())
        assert torch.all((l2 - pl).abs() <= 1e-3)


@pytest.mark.parametrize("h_q", [128, 8])
def test_causal_positions_equal_shorter_noncausal_runs(h_q):
    """With causal and s_q = 2, query 1 sees all L tokens and query 0 the
    first L - 1: each equals a non-causal s_q = 1 decode of that length (to
    the tolerance: the two runs take different schedules)."""
    L = [300, 65, 1000]
    w = W.make(3, 2, h_q, 1, L, stride=576, causal=True, seed=42)
    o, l, _, _ = run_gpu(w)
    for j in (0, 1):
        lens = torch.tensor([x - 1 + j for x in L], dtype=torch.int32)
        w1 = W.Workload(**{**w.__dict__, "q": w.q[:, j:j + 1].contiguous(), "s_q": 1, "causal": False,
                           "cache_seqlens": lens})
        o1, l1, _, _ = run_gpu(w1)
        ref = o1[:, 0].float()
        assert torch.all((o[:, j].float() - ref).abs() <= 1e-2 + 2e-2 * ref.abs())
        assert torch.all((l[:, :, j] - l1[:, :, 0]).abs() <= 1e-3)


@pytest.mark.parametrize("h_q", KERNEL_HEADS)
def test_thousands_of_short_sequences_sampled(h_q):
    """4096 sequences of 1-200 tokens: every part walks tens of segments (Q
    buffers, epilogues, split slots turn over many times); 3000 sampled rows
    plus the first and last sequence's rows against the oracle."""
    b = 4096
    sl = list(np.random.default_rng(4).integers(1, 200, size=b))
    w = W.make(b, 1, h_q, 1, sl, stride=640, seed=43, poison=True)
    out, lse, _, nsplit = run_gpu(w)
    assert int(nsplit[-1].item()) > b  # some sequences are cut
    extra = [(i, 0, h) for i in (0, b - 1) for h in range(h_q)]
    assert_matches(w, out, lse, sample_rows(w, 3000, seed=5, extra=extra))
