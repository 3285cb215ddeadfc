"""Shared helpers for the GPU parity tests: run the CUDA path through the
C-ABI binding and compare with the fp64 oracle on the same seeded bytes."""
import numpy as np
import torch

import oracle
from mla_decode_attention_03_gb300 import ops

# Tolerance: |d out| <= ATOL + RTOL * scale and |d lse| <= LSE_TOL.  The
# relative term is read against the magnitude of the output row (one (i, j, h)
# vector, a single softmax-weighted average of V rows): scale = max |out_oracle|
# over that row.  The stricter elementwise form (scale = |out_oracle| of the
# element itself) is also asserted on every workload except those with
# deliberately peaky keys: there the weights are rounded to bf16 -- the operand
# type the tensor cores require next to a bf16 cache -- with a relative error
# up to 2^-8 each, and x4-scaled value rows that cancel can push single
# near-zero elements past 1e-2 absolute while the row stays within 0.2%.
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


def compare_rows(w, out, lse, rows):
    """out [b, s_q, h_q, 512] bf16 and lse [b, h_q, s_q] from the GPU vs the
    oracle at `rows` (n x 3 of i, j, h).  Returns (max_out_excess, max_lse_err)."""
    rows = np.asarray(rows, dtype=np.int32).reshape(-1, 3)
    o_ref, l_ref = oracle_rows(w, rows)
    o = out.float().cpu().numpy().astype(np.float64)
    l = lse.float().cpu().numpy().astype(np.float64)
    i, j, h = rows[:, 0], rows[:, 1], rows[:, 2]
    o_gpu = o[i, j, h]
    l_gpu = l[i, h, j]
    assert np.all(np.isfinite(o_gpu)), "non-finite output"
    err = np.abs(o_gpu - o_ref)
    row_scale = np.abs(o_ref).max(axis=1, keepdims=True)
    excess_row = err - (ATOL + RTOL * row_scale)
    excess_elem = err - (ATOL + RTOL * np.abs(o_ref))
    fin = np.isfinite(l_ref)
    assert np.array_equal(np.isfinite(l_gpu), fin), "lse -inf pattern differs"
    assert np.all(l_gpu[~fin] == l_ref[~fin])
    lerr = np.abs(l_gpu[fin] - l_ref[fin])
    return (float(excess_row.max(initial=-1.0)), float(excess_elem.max(initial=-1.0)),
            float(lerr.max(initial=0.0)))


def assert_matches(w, out, lse, rows):
    ex_row, ex_elem, le = compare_rows(w, out, lse, rows)
    assert ex_row <= 0.0, f"out outside |d| <= {ATOL} + {RTOL}*rowmax|ref| by {ex_row:.3e}"
    if "peaky_slots" not in w.extra:
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
