"""Pins for the fp64 oracle (CPU only).

The oracle states the definition of MLA decode attention over a paged latent
cache (FlashMLA's flash_mla_with_kvcache as driven by the compare_a benchmark
of the PAI tutorial, section 4; 576/640-element entries per vLLM PR #12676).
Here it is tied to things other than itself: a dense NumPy/SciPy brute force
on tiny inputs, hand-derived closed forms (tests/golden), and invariants the
definition implies.  The last test plants known mistakes in the oracle and
checks that these pins catch every one of them.
"""
import math
import os

import numpy as np
import pytest
import torch
from scipy.special import logsumexp

import oracle
from mla_decode_attention_03_gb300 import workloads as W

GOLDEN = os.path.join(os.path.dirname(__file__), "golden", "closed_form_cases.txt")


# ----------------------------------------------------------------- helpers
def run(w, mutation=0, rows=None):
    qb, kb = w.numpy_bits()
    if rows is None:
        return oracle.decode(qb, kb, w.block_table.numpy(), w.cache_seqlens.numpy(), dv=w.dv,
                             softmax_scale=w.softmax_scale, causal=w.causal, mutation=mutation)
    return oracle.decode_rows(qb, kb, w.block_table.numpy(), w.cache_seqlens.numpy(), rows,
                              dv=w.dv, softmax_scale=w.softmax_scale, causal=w.causal,
                              mutation=mutation)


def brute(w):
    """Dense fp64 restatement: gather each sequence's keys into a matrix, take
    scores with a matmul, mask, SciPy's logsumexp, weights @ V."""
    q = w.q.double().numpy()
    kc = w.kcache.double().numpy()                     # [nb, 64, h_kv, 576]
    bt, sl = w.block_table.numpy(), w.cache_seqlens.numpy()
    b, s_q, h_q, _ = q.shape
    hpk = h_q // w.h_kv
    out = np.zeros((b, s_q, h_q, w.dv))
    lse = np.full((b, h_q, s_q), -np.inf)
    for i in range(b):
        L = int(sl[i])
        if L == 0:
            continue
        n = -(-L // 64)
        keys = kc[bt[i, :n]].reshape(n * 64, w.h_kv, 576)[:L]      # [L, h_kv, 576]
        t = np.arange(L)[None, :]
        j = np.arange(s_q)[:, None]
        allowed = (t <= L - s_q + j) if w.causal else np.ones((s_q, L), bool)
        for h in range(h_q):
            K = keys[:, h // hpk, :]
            S = w.softmax_scale * (q[i, :, h, :] @ K.T)             # [s_q, L]
            S = np.where(allowed, S, -np.inf)
            for jj in range(s_q):
                if not allowed[jj].any():
                    continue
                l = logsumexp(S[jj])
                lse[i, h, jj] = l
                out[i, jj, h] = np.exp(S[jj] - l) @ K[:, : w.dv]
    return out, lse


def close(a, b, tol=1e-12):
    a, b = np.asarray(a), np.asarray(b)
    fin = np.isfinite(b)
    if not np.array_equal(np.isfinite(a), fin):
        return False
    if not np.array_equal(a[~fin], b[~fin]):
        return False
    return bool(np.all(np.abs(a[fin] - b[fin]) <= tol * (1 + np.abs(b[fin]))))


def from_spec(shape, qs, ks, stride=576):
    b, s_q, h_q, h_kv, L = (shape[k] for k in ("b", "s_q", "h_q", "h_kv", "L"))
    n = max(1, -(-L // 64))
    q = torch.zeros((b, s_q, h_q, 576))
    for (i, j, h), ent in qs:
        for dim, v in ent:
            q[i, j, h, dim] = v
    kc = torch.zeros((n, 64, h_kv, stride))
    for t, ent in ks:
        for dim, v in ent:
            kc[t // 64, t % 64, 0, dim] = v
    return W.Workload(name="golden", q=q.to(torch.bfloat16), kcache_alloc=kc.to(torch.bfloat16),
                      block_table=torch.arange(n, dtype=torch.int32).view(1, n),
                      cache_seqlens=torch.tensor([L], dtype=torch.int32), s_q=s_q, h_q=h_q,
                      h_kv=h_kv, stride=stride, causal=bool(shape["causal"]),
                      softmax_scale=shape["scale"])


def parse_golden():
    def kv(tokens):
        return [(int(a), float(b)) for a, b in (x.split("=") for x in tokens)]
    cases, cur = [], None
    for raw in open(GOLDEN, encoding="utf-8"):
        line = raw.split("#", 1)[0].strip()
        if not line:
            continue
        f = line.split()
        if f[0] == "case":
            cur = dict(name=f[1], q=[], k=[], lse=[], out=[])
        elif f[0] == "shape":
            cur["shape"] = {a: (float(b) if a == "scale" else int(b))
                            for a, b in (x.split("=") for x in f[1:])}
        elif f[0] == "q":
            cur["q"].append(((int(f[1]), int(f[2]), int(f[3])), kv(f[5:])))
        elif f[0] == "k":
            cur["k"].append((int(f[1]), kv(f[3:])))
        elif f[0] == "expect_lse":
            cur["lse"].append(((int(f[1]), int(f[2]), int(f[3])), float(f[4])))
        elif f[0] == "expect_out":
            cur["out"].append(((int(f[1]), int(f[2]), int(f[3])), kv(f[5:])))
        elif f[0] == "end":
            cases.append(cur)
    return cases


# --------------------------------------------------------------- the pins
# Each check takes a mutation id and returns True when the oracle (so mutated)
# satisfies the pin.

BRUTE_CASES = [
    # b, s_q, h_q, h_kv, seqlens, stride, causal, permute
    (1, 1, 4, 1, [1], 576, False, False),
    (2, 1, 4, 1, [63, 130], 576, False, True),
    (2, 2, 4, 1, [64, 65], 640, True, True),
    (2, 1, 4, 2, [100, 7], 576, False, True),
    (3, 2, 2, 2, [2, 129, 0], 640, True, True),
    (1, 3, 2, 1, [70], 576, True, False),
]


def check_brute(mutation, case):
    b, s_q, h_q, h_kv, sl, stride, causal, permute = case
    w = W.make(b, s_q, h_q, h_kv, sl, stride=stride, causal=causal, permute=permute,
               seed=11 + len(sl))
    o, l = run(w, mutation)
    ob, lb = brute(w)
    return close(o, ob) and close(l, lb)


def check_golden(mutation, case):
    w = from_spec(case["shape"], case["q"], case["k"])
    o, l = run(w, mutation)
    ok = True
    for (i, h, j), v in case["lse"]:
        ok &= abs(l[i, h, j] - v) <= 1e-13 * (1 + abs(v))
    for (i, j, h), ent in case["out"]:
        want = np.zeros(w.dv)
        for dim, v in ent:
            want[dim] = v
        ok &= bool(np.all(np.abs(o[i, j, h] - want) <= 1e-13))
    return bool(ok)


def check_single_token(mutation):
    # L = 1: the softmax has one term, so out = V_0 exactly whatever q is.
    w = W.make(3, 1, 8, 1, [1, 1, 1], seed=5)
    o, _ = run(w, mutation)
    v = w.kcache.double().numpy()[w.block_table.numpy()[:, 0], 0, 0, : w.dv]
    return bool(np.all(o[:, 0] == v[:, None, :]))


def check_zero_query(mutation):
    # q = 0: every score is 0, so out = mean of the visible V_t and lse = ln(#visible).
    w = W.make(2, 1, 4, 1, [1, 97], seed=6)
    w.q.zero_()
    o, l = run(w, mutation)
    kc, bt = w.kcache.double().numpy(), w.block_table.numpy()
    ok = True
    for i, L in enumerate([1, 97]):
        V = np.concatenate([kc[bt[i, p], :, 0, : w.dv] for p in range(-(-L // 64))])[:L]
        ok &= close(o[i, 0], np.broadcast_to(V.mean(0), o[i, 0].shape), 1e-13)
        ok &= close(l[i], np.full_like(l[i], math.log(L)), 1e-13)
    return bool(ok)


def check_constant_key_tail(mutation):
    # q has only rope dims and every key's rope dims are the same constant:
    # all scores are equal, so out = mean of V over the visible tokens.
    w = W.make(1, 1, 2, 1, [150], seed=7)
    w.q[..., :512] = 0
    w.kcache_alloc[..., 512:576] = 0.5
    o, l = run(w, mutation)
    kc, bt = w.kcache.double().numpy(), w.block_table.numpy()
    V = np.concatenate([kc[bt[0, p], :, 0, : w.dv] for p in range(3)])[:150]
    s = w.softmax_scale * 0.5 * w.q[0, 0, :, 512:].double().sum(-1).numpy()
    return close(o[0, 0], np.broadcast_to(V.mean(0), (2, w.dv)), 1e-13) and \
        close(l[0, :, 0], s + math.log(150), 1e-13)


def check_dominant_key(mutation):
    # One key aligned with q scores ~43 above all others: out = that key's V to
    # within e^-40, lse = its score to within e^-40.
    w = W.make(1, 1, 1, 1, [200], seed=8)
    w.q.zero_()
    w.q[0, 0, 0, 0] = 16.0
    bt = w.block_table.numpy()
    w.kcache_alloc[..., 0] = 0.0
    star = 137
    w.kcache_alloc[bt[0, star // 64], star % 64, 0, 0] = 64.0
    o, l = run(w, mutation)
    v = w.kcache.double().numpy()[bt[0, star // 64], star % 64, 0, : w.dv]
    s_star = w.softmax_scale * 16.0 * 64.0
    return bool(np.all(np.abs(o[0, 0, 0] - v) <= 1e-15 * 200 * 64 + 200 * math.exp(-40)) and
                abs(l[0, 0, 0] - s_star) <= 200 * math.exp(-40))


def check_page_permutation(mutation):
    # Moving pages to other physical slots and updating block_table changes nothing.
    w = W.make(2, 1, 4, 1, [150, 64], seed=9, permute=False)
    o1, l1 = run(w, mutation)
    nb = w.num_blocks
    perm = np.random.default_rng(1).permutation(nb)
    kc2 = torch.empty_like(w.kcache_alloc)
    kc2[torch.from_numpy(perm)] = w.kcache_alloc
    bt = w.block_table.numpy()
    bt2 = np.where(bt >= 0, perm[np.maximum(bt, 0)], -1).astype(np.int32)
    w2 = W.Workload(**{**w.__dict__, "kcache_alloc": kc2, "block_table": torch.from_numpy(bt2)})
    o2, l2 = run(w2, mutation)
    return bool(np.array_equal(o1, o2) and np.array_equal(l1, l2))


def check_split_merge(mutation):
    # Attention over [0, L) equals the LSE-weighted merge of the attention over
    # [0, a) and [a, L) for a page boundary a (the Flash-Decoding combine).
    L, a = 200, 128
    w = W.make(1, 1, 4, 1, [L], seed=10)
    o, l = run(w, mutation)
    head = W.Workload(**{**w.__dict__, "cache_seqlens": torch.tensor([a], dtype=torch.int32)})
    bt = w.block_table.numpy()
    tail_bt = np.full_like(bt, -1)
    tail_bt[0, : bt.shape[1] - a // 64] = bt[0, a // 64:]
    tail = W.Workload(**{**w.__dict__, "block_table": torch.from_numpy(tail_bt),
                         "cache_seqlens": torch.tensor([L - a], dtype=torch.int32)})
    o1, l1 = run(head, mutation)
    o2, l2 = run(tail, mutation)
    lm = np.logaddexp(l1, l2)                                        # [1, h, 1]
    w1 = np.exp(l1 - lm).transpose(0, 2, 1)[..., None]
    w2 = np.exp(l2 - lm).transpose(0, 2, 1)[..., None]
    return close(lm, l, 1e-12) and close(w1 * o1 + w2 * o2, o, 1e-12)


def check_stride(mutation):
    # The same entries laid out at stride 576 and at stride 640 with a poisoned
    # pad give identical results: the pad is never part of an entry.
    w = W.make(2, 2, 4, 1, [90, 130], seed=12, stride=640, causal=True, poison=True)
    kc576 = w.kcache_alloc[..., :576].contiguous()
    w2 = W.Workload(**{**w.__dict__, "kcache_alloc": kc576, "stride": 576})
    o1, l1 = run(w, mutation)
    o2, l2 = run(w2, mutation)
    return bool(np.array_equal(o1, o2) and np.array_equal(l1, l2))


def check_unused_slots(mutation):
    # Cache slots past L in the last page do not matter: zeros and +-1e4 poison
    # give identical results.
    a = W.make(2, 1, 4, 1, [70, 33], seed=13)
    b = W.make(2, 1, 4, 1, [70, 33], seed=13, poison=True)
    oa, la = run(a, mutation)
    ob, lb = run(b, mutation)
    return bool(np.array_equal(oa, ob) and np.array_equal(la, lb))


def check_causal_equivalence(mutation):
    # Causal with s_q = 2: query 1 sees all L tokens (= non-causal s_q = 1 on L);
    # query 0 sees the first L-1 (= non-causal s_q = 1 on L-1).
    L = 130
    w = W.make(1, 2, 4, 1, [L], seed=14, causal=True)
    o, l = run(w, mutation)
    ok = True
    for j, Lj in ((0, L - 1), (1, L)):
        w1 = W.Workload(**{**w.__dict__, "q": w.q[:, j: j + 1].contiguous(), "s_q": 1,
                           "causal": False,
                           "cache_seqlens": torch.tensor([Lj], dtype=torch.int32)})
        o1, l1 = run(w1, mutation)
        ok &= np.array_equal(o[:, j], o1[:, 0]) and np.array_equal(l[:, :, j], l1[:, :, 0])
    return bool(ok)


def check_heads(mutation):
    # Identical query heads give identical rows; permuting heads permutes rows.
    w = W.make(1, 1, 6, 1, [77], seed=15)
    w.q[0, 0, 3] = w.q[0, 0, 1]
    o, l = run(w, mutation)
    perm = torch.tensor([5, 2, 0, 4, 1, 3])
    w2 = W.Workload(**{**w.__dict__, "q": w.q[:, :, perm].contiguous()})
    o2, l2 = run(w2, mutation)
    return bool(np.array_equal(o[0, 0, 3], o[0, 0, 1]) and
                np.array_equal(o2, o[:, :, perm.numpy()]) and
                np.array_equal(l2, l[:, perm.numpy()]))


def check_kv_groups(mutation):
    # With h_kv = 2, heads [0, h_q/2) read KV head 0 and the rest KV head 1:
    # each half equals an h_kv = 1 problem on that KV head's entries.
    w = W.make(1, 1, 4, 2, [100], seed=16)
    o, l = run(w, mutation)
    ok = True
    for g in range(2):
        kc = w.kcache_alloc[:, :, g: g + 1].contiguous()
        wg = W.Workload(**{**w.__dict__, "q": w.q[:, :, 2 * g: 2 * g + 2].contiguous(),
                           "kcache_alloc": kc, "h_q": 2, "h_kv": 1})
        og, lg = run(wg, mutation)
        ok &= np.array_equal(og, o[:, :, 2 * g: 2 * g + 2]) and \
            np.array_equal(lg, l[:, 2 * g: 2 * g + 2])
    return bool(ok)


GOLDEN_CASES = parse_golden()
PINS = (
    [(f"brute{n}", lambda m, c=c: check_brute(m, c)) for n, c in enumerate(BRUTE_CASES)]
    + [(f"golden_{c['name']}", lambda m, c=c: check_golden(m, c)) for c in GOLDEN_CASES]
    + [("single_token", check_single_token), ("zero_query", check_zero_query),
       ("constant_key_tail", check_constant_key_tail), ("dominant_key", check_dominant_key),
       ("page_permutation", check_page_permutation), ("split_merge", check_split_merge),
       ("stride", check_stride), ("unused_slots", check_unused_slots),
       ("causal_equivalence", check_causal_equivalence), ("heads", check_heads),
       ("kv_groups", check_kv_groups)]
)


@pytest.mark.parametrize("name,pin", PINS, ids=[n for n, _ in PINS])
def test_pin(name, pin):
    assert pin(0), name


def test_golden_file_has_cases():
    assert {c["name"] for c in GOLDEN_CASES} == {"two_token", "causal_three_token",
                                                 "rope_only_score"}


@pytest.mark.parametrize("mutation", sorted(oracle.MUTATIONS.items()),
                         ids=sorted(oracle.MUTATIONS))
def test_planted_mistake_is_caught(mutation):
    """Every planted mistake fails at least one pin other than the brute force,
    and the brute force catches it too where its cases reach it."""
    name, m = mutation

    def fails(pin):
        try:
            return not pin(m)
        except ValueError:  # the mutant read outside the cache: caught as well
            return True
    failed = [n for n, pin in PINS if fails(pin)]
    assert any(not n.startswith("brute") for n in failed), (name, failed)


def test_thread_count_does_not_change_results():
    w = W.make(3, 2, 8, 1, [300, 5, 64], seed=17, causal=True)
    qb, kb = w.numpy_bits()
    args = (qb, kb, w.block_table.numpy(), w.cache_seqlens.numpy())
    o1, l1 = oracle.decode(*args, softmax_scale=w.softmax_scale, causal=True, threads=1)
    o2, l2 = oracle.decode(*args, softmax_scale=w.softmax_scale, causal=True, threads=7)
    assert np.array_equal(o1, o2) and np.array_equal(l1, l2)


def test_rejects_bad_page_id():
    w = W.make(1, 1, 2, 1, [100], seed=18)
    w.block_table[0, 1] = w.num_blocks  # one past the end
    with pytest.raises(ValueError):
        run(w)


def test_empty_sequence_gives_zero_and_minus_inf():
    w = W.make(2, 1, 2, 1, [0, 10], seed=19)
    o, l = run(w)
    assert np.all(o[0] == 0) and np.all(np.isneginf(l[0])) and np.all(np.isfinite(l[1]))
