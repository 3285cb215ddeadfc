"""GPU: the host-buffer pipeline (mla_decode_host) against the device-buffer
call and the fp64 oracle.  With one run it makes the same schedule as the
device-buffer call and must match it bit for bit; with several runs each run
is its own split-KV schedule, so it is held to the oracle's tolerance, and two
calls with the same cut must agree bit for bit."""
import numpy as np
import pytest
import torch

from mla_decode_attention_03_gb300 import ops
from mla_decode_attention_03_gb300 import workloads as W
from tests._gpu_helpers import all_rows, assert_matches, run_gpu, to_device

pytestmark = pytest.mark.gpu


def host_inputs(w, pinned=True):
    f = (lambda t: t.contiguous().pin_memory()) if pinned else (lambda t: t.contiguous().clone())
    return f(w.q), f(w.block_table), f(w.cache_seqlens)


def run_host(w, hd, kc, chunks, pinned=True):
    q_h, bt_h, sl_h = host_inputs(w, pinned)
    out, lse = hd(q_h, kc, bt_h, sl_h, w.softmax_scale, w.causal, chunks=chunks)
    torch.cuda.synchronize()
    ops.check_status(hd.status)
    return out, lse


def test_one_run_equals_device_call():
    w = W.make(7, 1, 128, 1, [1, 63, 64, 65, 700, 0, 2000], stride=640, seed=31, poison=True)
    dev = to_device(w)
    parts = ops.num_parts(w.s_q, w.h_q, w.h_kv)
    o_dev, l_dev, _, _ = run_gpu(w, parts=parts, dev=dev)
    hd = ops.HostDecoder(w.b, w.s_q, w.h_q, w.block_table.shape[1], w.h_kv, parts=parts)
    o_h, l_h = run_host(w, hd, dev["kcache"], chunks=1)
    hd.close()
    assert torch.equal(o_h, o_dev.cpu()) and torch.equal(l_h, l_dev.cpu())


@pytest.mark.parametrize("h_q", [128, 8])
@pytest.mark.parametrize("chunks", [2, 3, 8])
def test_several_runs_all_rows(chunks, h_q):
    w = W.make(9, 2, h_q, 1, [0, 5, 64, 129, 700, 1, 3000, 0, 333], stride=640, causal=True, seed=32,
               poison=True)
    dev = to_device(w)
    hd = ops.HostDecoder(w.b, w.s_q, w.h_q, w.block_table.shape[1], w.h_kv, parts=5)
    out, lse = run_host(w, hd, dev["kcache"], chunks=chunks)
    hd.close()
    assert_matches(w, out, lse, all_rows(w))


def test_back_to_back_calls_and_pageable_memory():
    """Calls enqueued without a synchronisation between them, on one stream
    and across two (each call's copies in must wait for the previous call's
    decode and copies out), give what each gives alone; pageable host tensors
    give the pinned result."""
    w1 = W.make(6, 1, 64, 1, [900, 64, 1, 129, 1000, 333], stride=576, seed=33)
    w2 = W.make(6, 1, 64, 1, [900, 64, 1, 129, 1000, 333], stride=576, seed=34)
    w2 = W.Workload(**{**w2.__dict__, "kcache_alloc": w1.kcache_alloc, "block_table": w1.block_table})
    dev = to_device(w1)
    hd = ops.HostDecoder(w1.b, w1.s_q, w1.h_q, w1.block_table.shape[1], w1.h_kv, parts=4)
    a1 = run_host(w1, hd, dev["kcache"], chunks=3)
    a2 = run_host(w2, hd, dev["kcache"], chunks=3)
    a1_one = run_host(w1, hd, dev["kcache"], chunks=1)
    x1, x2 = host_inputs(w1), host_inputs(w2)
    b1 = hd(*x1[:1], dev["kcache"], *x1[1:], w1.softmax_scale, w1.causal, chunks=3)
    b2 = hd(*x2[:1], dev["kcache"], *x2[1:], w2.softmax_scale, w2.causal, chunks=3)
    # a one-run call on another stream must still wait for the call before it
    side = torch.cuda.Stream()
    with torch.cuda.stream(side):
        b3 = hd(*x1[:1], dev["kcache"], *x1[1:], w1.softmax_scale, w1.causal, chunks=1)
    b4 = hd(*x2[:1], dev["kcache"], *x2[1:], w2.softmax_scale, w2.causal, chunks=3)
    torch.cuda.synchronize()
    ops.check_status(hd.status)
    c2 = run_host(w2, hd, dev["kcache"], chunks=3, pinned=False)
    hd.close()
    for (o, l), (o_ref, l_ref) in ((b1, a1), (b2, a2), (b3, a1_one), (b4, a2), (c2, a2)):
        assert torch.equal(o, o_ref) and torch.equal(l, l_ref)
    assert_matches(w2, *a2, all_rows(w2))


def test_bench_workload_all_rows():
    """The benchmark's workload through the host-buffer entry point with the
    automatic cut (the configuration its end-to-end figure times), every row."""
    w = W.named("bench")
    dev = to_device(w)
    assert len(ops.host_chunks(w.cache_seqlens)) - 1 == 3
    hd = ops.HostDecoder(w.b, w.s_q, w.h_q, w.block_table.shape[1], w.h_kv)
    out, lse = run_host(w, hd, dev["kcache"], chunks=0)
    hd.close()
    assert_matches(w, out, lse, all_rows(w))
    assert torch.isfinite(out.float()).all() and torch.isfinite(lse).all()
