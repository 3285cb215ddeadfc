"""A whole decode step captured in a CUDA graph.

FlashMLA's metadata is computed once per decode step and shared by every layer
(vLLM's FlashMLAMetadataBuilder calls get_mla_metadata, FlashMLAImpl calls
flash_mla_with_kvcache per layer; PAI tutorial, section 2), and the tutorial's
vLLM runs note enforce_eager, i.e. the graph-captured path is the serving
default.  The C ABI allocates nothing and never synchronises, so the step
(metadata + three layers of decode and combine) can be captured once and
replayed; replays must equal the eager calls, also after the inputs change in
place, and the first replay is checked against the fp64 oracle on every row.
"""
import pytest
import torch

from tests._gpu_helpers import all_rows, assert_matches

from mla_decode_attention_03_gb300 import ops
from mla_decode_attention_03_gb300 import workloads as W

pytestmark = pytest.mark.gpu

LAYERS = 3


def _layer_inputs(seed, stride=640, h_q=128):
    # same lengths and block table for every layer (one step: pages in order,
    # so every layer's table is the same), different q and cache
    return W.make(6, 1, h_q, 1, [700, 64, 3000, 1, 129, 4096], stride=stride, seed=seed, permute=False)


@pytest.mark.parametrize("h_q", [128, 16])
def test_captured_step_equals_eager_and_tracks_new_inputs(h_q):
    ws = [_layer_inputs(40 + k, h_q=h_q) for k in range(LAYERS)]
    assert all(torch.equal(w.block_table, ws[0].block_table) for w in ws)
    sl = ws[0].cache_seqlens.cuda()
    bt = ws[0].block_table.cuda()
    qs = [w.q.cuda() for w in ws]
    kcs = [w.kcache_alloc.cuda()[..., :576] for w in ws]
    dec = ops.MLADecoder(6, 1, h_q, 1, parts=11)
    outs = [torch.empty((6, 1, h_q, 512), dtype=torch.bfloat16, device="cuda") for _ in range(LAYERS)]
    lses = [torch.empty((6, h_q, 1), dtype=torch.float32, device="cuda") for _ in range(LAYERS)]
    scale = ws[0].softmax_scale

    def step():
        dec.plan(sl)
        for k in range(LAYERS):
            dec(qs[k], kcs[k], bt, sl, scale, out=outs[k], lse=lses[k])

    # eager reference (also loads the library's kernels and sets their attributes
    # before capture)
    step()
    torch.cuda.synchronize()
    ref = [(o.clone(), l.clone()) for o, l in zip(outs, lses)]

    stream = torch.cuda.Stream()
    stream.wait_stream(torch.cuda.current_stream())
    graph = torch.cuda.CUDAGraph()
    with torch.cuda.stream(stream):
        with torch.cuda.graph(graph, stream=stream):
            step()
    torch.cuda.current_stream().wait_stream(stream)
    for o in outs:
        o.zero_()
    graph.replay()
    torch.cuda.synchronize()
    ops.check_status(dec.status)
    for (o, l), (ro, rl) in zip(zip(outs, lses), ref):
        assert torch.equal(o, ro) and torch.equal(l, rl)
    for w, o, l in zip(ws, outs, lses):
        assert_matches(w, o, l, all_rows(w))

    # new q values in place: the replay must follow them
    for k in range(LAYERS):
        qs[k].copy_(W.make(6, 1, h_q, 1, [1] * 6, seed=90 + k).q.cuda())
    graph.replay()
    torch.cuda.synchronize()
    got = [(o.clone(), l.clone()) for o, l in zip(outs, lses)]
    step()
    torch.cuda.synchronize()
    for (o, l), (eo, el) in zip(got, zip(outs, lses)):
        assert torch.equal(o, eo) and torch.equal(l, el)
    assert not torch.equal(got[0][0], ref[0][0])
