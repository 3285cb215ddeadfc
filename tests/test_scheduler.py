"""The split-KV schedule (mla_get_metadata).

No page states how the KV length must be cut -- Flash-Decoding only says that
it is cut and merged by log-sum-exp -- so any cut that covers every page of
every sequence exactly once, in order, is correct.  check_schedule() tests
exactly that, plus the balance the scheduler promises.  A host restatement of
the cut (host_schedule) lets the CPU suite exercise the properties on
many shapes and lets the GPU suite require the device output to equal it bit
for bit (integer work).
"""
import numpy as np
import pytest
import torch

SEGMENT_COST, MIN_PART_COST, PAGE = 6, 4, 64


def pages_of(L):
    return -(-int(L) // PAGE) if L > 0 else 0


def host_schedule(seqlens, parts):
    """The cut, restated on the host: returns (meta [parts, 8], num_splits [b+1]).

    Cost axis: sequence i with n_i > 0 pages occupies [C_i, C_i + n_i + F);
    part q takes [q*per, (q+1)*per) with per = max(ceil(total/parts), F + MIN);
    a cut at x lies in the last sequence with C_i <= x, at page max(0, x - C_i - F)."""
    F = SEGMENT_COST
    b = len(seqlens)
    width = [pages_of(L) + F if pages_of(L) > 0 else 0 for L in seqlens]
    C = np.concatenate([[0], np.cumsum(width)]).astype(np.int64)
    total = int(C[-1])
    per = max(-(-total // parts), MIN_PART_COST)

    def seq_at(x):
        return int(np.searchsorted(C[:b], x, side="right")) - 1

    def npages(i):
        return int(C[i + 1] - C[i] - F)

    meta = np.zeros((parts, 8), dtype=np.int32)
    for q in range(parts):
        x0, x1 = q * per, (q + 1) * per
        if x0 >= total:
            meta[q, :5] = [1, 0, 0, 0, 0]
            continue
        i0 = seq_at(x0)
        p0 = max(0, x0 - int(C[i0]) - F)
        if x1 >= total:
            i1 = seq_at(total - 1)
            pe1 = npages(i1)
        else:
            ie = seq_at(x1)
            oe = x1 - int(C[ie]) - F
            if oe > 0:
                i1, pe1 = ie, oe
            elif ie == i0 and p0 == 0:
                meta[q, :5] = [1, 0, 0, 0, 0]
                continue
            else:
                i1 = seq_at(int(C[ie]) - 1)
                pe1 = npages(i1)
        k0 = q - (int(C[i0]) + F) // per if p0 > 0 else 0
        meta[q, :5] = [i0, p0, i1, pe1, k0]
    segs = [1 + max(0, (int(C[i]) + w - 1) // per - (int(C[i]) + F) // per) if w > 0 else 0
            for i, w in enumerate(width)]
    return meta, np.concatenate([[0], np.cumsum(segs)]).astype(np.int32)


def check_schedule(seqlens, parts, meta, num_splits):
    """Every page of every sequence is covered exactly once, parts are in
    (sequence, page) order, split indices are 0..n-1 per sequence, num_splits
    is their prefix count, and no part is much over the even share."""
    pages = [pages_of(L) for L in seqlens]
    b = len(pages)
    assert meta.shape == (parts, 8) and num_splits.shape == (b + 1,)
    covered = [np.zeros(n, dtype=np.int32) for n in pages]
    seg_k = [[] for _ in range(b)]
    prev_end = (0, 0)
    costs = []
    for q in range(parts):
        i0, p0, i1, pe, k0 = (int(x) for x in meta[q, :5])
        cost = 0
        if i0 > i1:
            costs.append(0)
            continue
        assert (i0, p0) >= prev_end, f"part {q} starts before the previous part ended"
        for i in range(i0, i1 + 1):
            pb = p0 if i == i0 else 0
            pend = pe if i == i1 else pages[i]
            if pb >= pend:
                continue
            covered[i][pb:pend] += 1
            seg_k[i].append(k0 if i == i0 else 0)
            cost += SEGMENT_COST + pend - pb
        prev_end = (i1, pe)
        costs.append(cost)
    for i in range(b):
        assert np.all(covered[i] == 1), f"sequence {i}: pages covered {covered[i].tolist()}"
        assert seg_k[i] == list(range(len(seg_k[i]))), f"sequence {i}: split ids {seg_k[i]}"
        assert num_splits[i + 1] - num_splits[i] == len(seg_k[i])
    assert num_splits[0] == 0
    total = sum(n + SEGMENT_COST for n in pages if n > 0)
    per = max(-(-total // parts), MIN_PART_COST)
    # a part spans at most `per` units of the cost axis, plus the fixed cost of
    # a first segment whose start was paid for by the previous part
    assert max(costs, default=0) <= per + SEGMENT_COST, (max(costs), per)
    assert int(num_splits[-1]) <= b + parts


CASES = [
    ("bench", [4096] * 128),
    ("one", [256]),
    ("zeros", [0, 0, 5, 0, 4096, 0]),
    ("all_zero", [0, 0, 0]),
    ("skewed", [65536, 65536] + list(np.random.default_rng(0).integers(64, 1025, 62))),
    ("short", list(np.random.default_rng(1).integers(1, 200, 300))),
    ("mtp", list(np.clip(np.round(np.random.default_rng(2).normal(4096, 1024, 128)), 256, 8192).astype(int))),
    ("long_one", [1 << 20]),
    # more sequences than the single-warp path of the device scheduler takes
    ("many", list(np.random.default_rng(3).integers(0, 3000, 3000))),
]


@pytest.mark.parametrize("name,sl", CASES, ids=[c[0] for c in CASES])
@pytest.mark.parametrize("parts", [1, 2, 7, 38, 76, 500])
def test_host_schedule_is_valid(name, sl, parts):
    meta, ns = host_schedule(sl, parts)
    check_schedule(sl, parts, meta, ns)


def test_random_schedules_are_valid():
    rng = np.random.default_rng(7)
    for _ in range(300):
        b = int(rng.integers(1, 60))
        sl = rng.integers(0, 3000, b) * (rng.random(b) < 0.9)
        parts = int(rng.integers(1, 160))
        meta, ns = host_schedule(list(sl), parts)
        check_schedule(list(sl), parts, meta, ns)


def test_check_schedule_catches_a_gap():
    meta, ns = host_schedule([4096, 4096], 4)
    meta = meta.copy()
    meta[1, 1] += 1  # part 1 starts one page late
    with pytest.raises(AssertionError):
        check_schedule([4096, 4096], 4, meta, ns)


@pytest.mark.gpu
@pytest.mark.parametrize("name,sl", CASES, ids=[c[0] for c in CASES])
@pytest.mark.parametrize("parts", [1, 7, 76, 500])
def test_device_schedule_equals_host(name, sl, parts):
    from mla_decode_attention_03_gb300 import ops
    sl_t = torch.tensor(sl, dtype=torch.int32, device="cuda")
    status = ops.new_status()
    meta, ns = ops.get_mla_metadata(sl_t, parts, status)
    ops.check_status(status)
    hm, hn = host_schedule(sl, parts)
    assert np.array_equal(meta.cpu().numpy(), hm)
    assert np.array_equal(ns.cpu().numpy(), hn)
