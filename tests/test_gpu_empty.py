"""An empty batch (T = 0) through every layer entry point.

A serving or expert-parallel step can hand a layer no tokens at all.  The
layer's outputs are then defined by their sums: no expert receives a row
(counts, offsets and padded offsets all 0, [kucoin] §01's layout of zero
tokens), the forward and combine produce no rows, and every weight gradient
is an empty sum over token rows, so exactly zero ([kucoin] §01: the backward's
weight gradients accumulate over the tokens an expert saw).  Each call returns
MOK_OK, and the workspace's status word reads OK afterwards.
"""
import pytest
import torch

from combine_top_routing_gb300 import inputs as I
from combine_top_routing_gb300 import mok
from combine_top_routing_gb300.layer import scale_words
from mokhelp import Routed, make_layer

pytestmark = pytest.mark.gpu

CASES = {
    "bf16": I.Workload("empty_bf16", T=0, d=256, E=8, k=2, F=384, dtype="bf16",
                       router="softmax", seed=91),
    "mxfp8": I.Workload("empty_mx", T=0, d=512, E=16, k=4, F=256, dtype="mxfp8",
                        router="sigmoid", seed=92),
}


def _poisoned(*shape, dtype):
    t = torch.empty(shape, dtype=dtype, device="cuda")
    t.view(torch.uint8).fill_(0x5A)
    return t


@pytest.mark.parametrize("name", list(CASES))
def test_empty_batch_forward_backward(name):
    w = CASES[name]
    layer, inp = make_layer(w, training=True)
    layer.prepare_backward()
    # the saved routing is written even for no tokens: no expert has a row
    layer.ctx.fill_(0x5A)
    out = layer.forward()
    torch.cuda.synchronize()
    assert layer.status() == 0
    assert out.shape == (0, w.d)
    for field in ("counts", "offsets", "pad_offsets"):
        n = w.E if field == "counts" else w.E + 1
        assert torch.equal(layer.ctx_view(field, torch.int32, (n,)),
                           torch.zeros(n, dtype=torch.int32, device="cuda")), field
    # every weight gradient is an empty sum: zero, whatever the buffers held
    for g in layer.grads.values():
        g.view(torch.uint8).fill_(0x5A)
    layer.dW_r.fill_(3.0)
    layer.bws.fill_(0x5A)
    dX = layer.backward(inp["dY"])
    torch.cuda.synchronize()
    assert mok.get_device_status(layer.bws) == 0
    assert dX.shape == (0, w.d)
    for name_g, g in layer.grads.items():
        assert not g.view(torch.int16).any(), name_g
    assert not layer.dW_r.any()


@pytest.mark.parametrize("name", list(CASES))
def test_empty_batch_step_entry_points(name):
    w = CASES[name]
    layer, _ = make_layer(w)
    R = Routed(layer)
    torch.cuda.synchronize()
    assert not R.counts.any() and not R.offsets.any() and not R.pad_offsets.any()
    # the same call into buffers that held other bytes
    counts = _poisoned(w.E, dtype=torch.int32)
    offsets = _poisoned(w.E + 1, dtype=torch.int32)
    pad = _poisoned(w.E + 1, dtype=torch.int32)
    mok.route_layout(layer.cfg, layer.x_src, layer.W_r, layer.bias, R.ids, R.gates, R.sel, R.logits,
                     counts, offsets, pad, R.slot_pos, R.row_tok, R.row_j, layer.ws)
    torch.cuda.synchronize()
    assert not counts.any() and not offsets.any() and not pad.any()
    # the workspace-free layout too
    counts = _poisoned(w.E, dtype=torch.int32)
    offsets = _poisoned(w.E + 1, dtype=torch.int32)
    pad = _poisoned(w.E + 1, dtype=torch.int32)
    mok.layout_static(layer.cfg, R.ids, counts, offsets, pad, R.slot_pos, R.row_tok, R.row_j)
    torch.cuda.synchronize()
    assert not counts.any() and not offsets.any() and not pad.any()
    # dispatch, expert FFN, combine and the fused call have nothing to do
    rows = layer.rows_pad
    mx = w.dtype == "mxfp8"
    xe = torch.empty((rows, w.d), dtype=torch.uint8 if mx else torch.bfloat16, device="cuda")
    xs = torch.empty(scale_words(rows, w.d), dtype=torch.int32, device="cuda") if mx else None
    ystage = torch.empty((0, w.k, w.d), dtype=torch.bfloat16, device="cuda")
    out = torch.empty((0, w.d), dtype=torch.bfloat16, device="cuda")
    mok.dispatch(layer.cfg, layer.x_src, R.ids, R.offsets, R.pad_offsets, R.row_tok, R.row_j, xe, xs)
    mok.dispatch_by_token(layer.cfg, layer.x_src, R.ids, R.slot_pos, R.offsets, R.pad_offsets, xe, xs)
    mok.expert_ffn(layer.cfg, xe, xs, layer.wstruct, R.offsets, R.pad_offsets, R.row_tok, R.row_j,
                   ystage, None, None, None, layer.ws)
    mok.combine(layer.cfg, ystage, R.gates, out)
    layer.ws[:256].fill_(0x5A)  # the status word sits at the front of the workspace
    mok.moe_fused(layer.cfg, layer.x_src, layer.wstruct, R.ids, R.gates, R.counts, R.offsets,
                  R.pad_offsets, R.slot_pos, R.row_tok, R.row_j, ystage, out, layer.ws)
    torch.cuda.synchronize()
    assert layer.status() == 0


def test_empty_batch_chain():
    w = CASES["bf16"]
    layer, _ = make_layer(w)
    wss = [layer.ws, torch.empty_like(layer.ws)]
    for ws in wss:
        ws[:256].fill_(0x5A)
    outs = [torch.empty((0, w.d), dtype=torch.bfloat16, device="cuda") for _ in range(3)]
    mok.moe_forward_chain(layer.cfg, [layer.x_src] * 3, layer.W_r, layer.bias, layer.wstruct, outs,
                          [wss[i % 2] for i in range(3)])
    torch.cuda.synchronize()
    for ws in wss:
        assert mok.get_device_status(ws) == 0
