"""Failure detection of the decode kernels on the GPU, without a GPU fault.

Every wait in the decode kernels is bounded (about 2 s).  The diagnostic entry
point mla_selftest_wait_timeout runs the decode with one wait on a barrier
that nothing ever completes, placed before any copy is issued: the wait gives
up, every other warp role leaves its own wait through the CTA's abort flag
(both CTAs of each cluster in the 128-row kernel), and the status word reports
MLA_ERR_TIMEOUT (-6).  The context must stay usable: a normal decode right
after it matches the oracle.  Both kernels are covered: 128 heads per KV head
run on the 128-row kernel, 16 on the 16-row one.
"""
import pytest
import torch

from mla_decode_attention_03_gb300 import ops
from mla_decode_attention_03_gb300 import workloads as W
from tests._gpu_helpers import all_rows, assert_matches, run_gpu, to_device

pytestmark = pytest.mark.gpu


@pytest.mark.parametrize("h_q", [128, 16])
def test_wait_that_never_ends_reports_timeout_and_context_survives(h_q):
    w = W.make(2, 1, h_q, 1, [100, 300], stride=640, seed=28)
    dev = to_device(w)
    status = ops.new_status()
    parts = 4
    meta, nsplit = ops.get_mla_metadata(dev["cache_seqlens"], parts, status)
    out = torch.empty((w.b, 1, h_q, 512), dtype=torch.bfloat16, device="cuda")
    lse = torch.empty((w.b, h_q, 1), dtype=torch.float32, device="cuda")
    ws = torch.empty((ops.workspace_bytes(w.b, 1, h_q, parts),), dtype=torch.uint8, device="cuda")
    kc = dev["kcache"]
    bt, sl = dev["block_table"], dev["cache_seqlens"]
    rc = ops.load_library().mla_selftest_wait_timeout(
        dev["q"].data_ptr(), w.b, 1, h_q, 576, kc.data_ptr(), w.num_blocks, 64, 1, ops.entry_stride(kc),
        bt.data_ptr(), bt.shape[1], sl.data_ptr(), 512, meta.data_ptr(), parts, nsplit.data_ptr(),
        w.softmax_scale, 0, out.data_ptr(), lse.data_ptr(), ws.data_ptr(), ws.numel(), status.data_ptr(),
        torch.cuda.current_stream().cuda_stream)
    assert rc == 0
    torch.cuda.synchronize()
    assert int(status.item()) == -6
    # the context is still usable
    o2, l2, _, _ = run_gpu(w, dev=dev)
    assert_matches(w, o2, l2, all_rows(w))


@pytest.mark.parametrize("name", ["v2lite", "tiny"])
def test_small_head_tiles_repeated_back_to_back(name):
    """16-head tiles on the 16-row kernel, many back-to-back decodes: a waiter
    on one of its two-slot barriers (stages, Q buffers, maxima, P buffers)
    that could fall two phases behind would show up only after several of
    them (a timeout, not a fault): 40 decodes, the status word checked every
    eighth, the last output compared with the oracle on every row."""
    w = W.named(name)
    dev = to_device(w)
    parts = ops.num_parts(w.s_q, w.h_q, w.h_kv)
    dec = ops.MLADecoder(w.b, w.s_q, w.h_q, w.h_kv, parts=parts)
    meta, nsplit = ops.get_mla_metadata(dev["cache_seqlens"], parts, dec.status)
    flush = torch.empty(256 << 20, dtype=torch.uint8, device="cuda")
    for k in range(40):
        flush.fill_(k)
        out, lse = ops.mla_decode_with_kvcache(dev["q"], dev["kcache"], dev["block_table"], dev["cache_seqlens"],
                                               meta, nsplit, w.softmax_scale, w.causal, workspace=dec.workspace,
                                               status=dec.status)
        if k % 8 == 7:
            torch.cuda.synchronize()
            assert int(dec.status.item()) == 0, f"decode {k}: status {int(dec.status.item())}"
    torch.cuda.synchronize()
    assert int(dec.status.item()) == 0
    assert_matches(w, out, lse, all_rows(w))
