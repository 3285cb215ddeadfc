"""The allocation-free decode entry point, mla_decode_with_kvcache_static.

Some callers cannot allocate device memory at the point where they run the
decode: a plug-in inside a host program that owns all device memory through
its own pool and hands its plug-ins no allocator, or a serving loop that must
not call cudaMalloc because it can synchronise the whole device.
This entry point takes its split-KV scratch from a buffer the library keeps in
device memory itself.  The test calls it through the C ABI twice in a row, on
two different inputs, and checks each result against mla_decode_with_kvcache
(the caller-provided-workspace entry point) on the same inputs: both run the
same schedule and kernels, so the results must be bit for bit identical.

The file is named so that pytest collects it last.
"""
import ctypes

import pytest
import torch

from mla_decode_attention_03_gb300 import ops
from mla_decode_attention_03_gb300 import workloads as W

pytestmark = pytest.mark.gpu


def _static_entry():
    lib = ops.load_library()
    f = lib.mla_decode_with_kvcache_static
    P, I, I64, F = ctypes.c_void_p, ctypes.c_int, ctypes.c_int64, ctypes.c_float
    f.restype = ctypes.c_int32
    f.argtypes = [P, I, I, I, I, P, I64, I, I, I, P, I, P, I, P, I, P, F, I, P, P, P, P]
    return f


def _inputs(w, parts):
    kc = w.kcache_alloc.cuda()[..., :576]
    d = dict(q=w.q.cuda(), kc=kc, bt=w.block_table.cuda(), sl=w.cache_seqlens.cuda())
    d["status"] = ops.new_status()
    d["meta"], d["nsplit"] = ops.get_mla_metadata(d["sl"], parts, d["status"])
    return d


def _call_static(f, w, d, parts):
    out = torch.full((w.b, w.s_q, w.h_q, 512), float("nan"), dtype=torch.bfloat16, device="cuda")
    lse = torch.full((w.b, w.h_q, w.s_q), float("nan"), dtype=torch.float32, device="cuda")
    rc = f(d["q"].data_ptr(), w.b, w.s_q, w.h_q, 576, d["kc"].data_ptr(), w.num_blocks, 64, w.h_kv,
           ops.entry_stride(d["kc"]), d["bt"].data_ptr(), d["bt"].shape[1], d["sl"].data_ptr(), 512,
           d["meta"].data_ptr(), parts, d["nsplit"].data_ptr(), w.softmax_scale, int(w.causal),
           out.data_ptr(), lse.data_ptr(), d["status"].data_ptr(), torch.cuda.current_stream().cuda_stream)
    assert rc == 0, ops.status_string(rc)
    return out, lse


def test_static_scratch_matches_caller_workspace_on_two_calls():
    f = _static_entry()
    cases = [
        # several long sequences cut into many pieces, 640-element entries
        (W.make(6, 1, 128, 1, [300, 4096, 1, 64, 2000, 700], stride=640, seed=31), 9),
        # causal s_q = 2 (two row tiles), a different split pattern
        (W.make(5, 2, 128, 1, [129, 2, 3000, 64, 900], stride=576, causal=True, seed=32), 7),
        # 16 heads: the 16-row kernel
        (W.make(6, 1, 16, 1, [300, 4096, 1, 64, 2000, 700], stride=640, seed=33), 9),
    ]
    for w, parts in cases:
        d = _inputs(w, parts)
        ref_out, ref_lse = ops.mla_decode_with_kvcache(d["q"], d["kc"], d["bt"], d["sl"], d["meta"],
                                                       d["nsplit"], w.softmax_scale, w.causal,
                                                       status=d["status"])
        out, lse = _call_static(f, w, d, parts)
        torch.cuda.synchronize()
        ops.check_status(d["status"])
        assert int(d["nsplit"][-1].item()) > w.b  # the scratch was really used
        # same schedule, same kernels: only the scratch differs, so the results
        # must be identical
        assert torch.equal(out, ref_out) and torch.equal(lse, ref_lse)


def test_static_scratch_rejects_shapes_beyond_its_size():
    f = _static_entry()
    big = ops.workspace_bytes(4096, 2, 128, 76)
    assert big > (64 << 20)
    fake = 1 << 20  # never dereferenced: the size check comes first
    rc = f(fake, 4096, 2, 128, 576, fake, 1000, 64, 1, 576, fake, 64, fake, 512, fake, 76, fake,
           0.04, 0, fake, fake, fake, None)
    assert rc == -8 and ops.status_string(rc).startswith("MLA_ERR_SCRATCH_TOO_SMALL")
