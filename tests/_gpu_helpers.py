"""Shared helpers for the GPU parity tests: run the CUDA path through the
C-ABI binding and compare with the fp64 oracle on the same seeded bytes."""
import numpy as np
import torch

import oracle
from mla_decode_attention_03_gb300 import ops

# Tolerance, element by element: |d out| <= ATOL + RTOL * |out_oracle| and
# |d lse| <= LSE_TOL, on every workload.
ATOL, RTOL, LSE_TOL = 1e-2, 2e-2, 1e-3


def to_device(w):
    kc_alloc = w.kcache_alloc.cuda()
    return dict(q=w.q.cuda(), kcache=kc_alloc[..., :576], kcache_alloc=kc_alloc,
                block_table=w.block_table.cuda(), cache_seqlens=w.cache_seqlens.cuda())


def run_gpu(w, parts=None, dev=None):
    dev = dev or to_device(w)
    parts = parts or ops.num_parts(w.s_q, w.h_q, w.h_kv)
    status = ops.new_status()
    meta, nsplit = ops.get_mla_metadata(dev["cache_seqlens"], parts, status)
    out, lse = ops.mla_decode_with_kvcache(dev["q"], dev["kcache"], dev["block_table"],
                                           dev["cache_seqlens"], meta, nsplit, w.softmax_scale,
                                           w.causal, status=status)
    torch.cuda.synchronize()
    ops.check_status(status)
    return out, lse, meta, nsplit


def oracle_rows(w, rows):
    qb, kb = w.numpy_bits()
    return oracle.decode_rows(qb, kb, w.block_table.numpy(), w.cache_seqlens.numpy(), rows,
                              dv=w.dv, softmax_scale=w.softmax_scale, causal=w.causal)


def compare_rows(w, out, lse, rows, chunk=8192):
    """out [b, s_q, h_q, 512] bf16 and lse [b, h_q, s_q] from the GPU vs the
    oracle at `rows` (n x 3 of i, j, h), in chunks of rows.  Returns
    (max elementwise excess over the tolerance, max |d lse|)."""
    rows = np.asarray(rows, dtype=np.int32).reshape(-1, 3)
    o = out.float().cpu().numpy()
    l = lse.float().cpu().numpy().astype(np.float64)
    ex_elem, lerr = -1.0, 0.0
    for c0 in range(0, len(rows), chunk):
        r = rows[c0:c0 + chunk]
        o_ref, l_ref = oracle_rows(w, r)
        i, j, h = r[:, 0], r[:, 1], r[:, 2]
        o_gpu = o[i, j, h].astype(np.float64)
        l_gpu = l[i, h, j]
        assert np.all(np.isfinite(o_gpu)), "non-finite output"
        err = np.abs(o_gpu - o_ref) - (ATOL + RTOL * np.abs(o_ref))
        ex_elem = max(ex_elem, float(err.max(initial=-1.0)))
        fin = np.isfinite(l_ref)
        assert np.array_equal(np.isfinite(l_gpu), fin), "lse -inf pattern differs"
        assert np.all(l_gpu[~fin] == l_ref[~fin])
        lerr = max(lerr, float(np.abs(l_gpu[fin] - l_ref[fin]).max(initial=0.0)))
    return ex_elem, lerr


def assert_matches(w, out, lse, rows):
    ex_elem, le = compare_rows(w, out, lse, rows)
    assert ex_elem <= 0.0, f"out outside |d| <= {ATOL} + {RTOL}|ref| by {ex_elem:.3e}"
    assert le <= LSE_TOL, f"lse error {le:.3e} > {LSE_TOL}"


def sample_rows(w, n, seed=0, extra=()):
    rng = np.random.default_rng(seed)
    rows = np.stack([rng.integers(0, w.b, n), rng.integers(0, w.s_q, n), rng.integers(0, w.h_q, n)], 1)
    if len(extra):
        rows = np.concatenate([rows, np.asarray(extra).reshape(-1, 3)])
    return rows.astype(np.int32)


def all_rows(w):
    return oracle.all_rows(w.b, w.s_q, w.h_q)
