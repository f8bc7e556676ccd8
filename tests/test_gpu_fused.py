"""The fused persistent forward (A7): one cooperative kernel with a gather
role and a GEMM role handing minibatches over through on-GPU counters and a
fixed-size token ring.

  * bit-identical to the separate-kernel path (route_layout, dispatch,
    expert_ffn, combine) -- every tile is the same instruction sequence;
  * bit-identical across gather SM fractions {1/8, 1/4, 1/3}, minibatch
    {64, 128, 256} and ring sizes down to 256 rows (many wraps) -- the
    pages' determinism claim;
  * a ring smaller than one minibatch is refused on the host;
  * a device wait that runs out reports MOK_ERR_TIMEOUT through the status
    word, and the context stays usable for the next call.
"""
import itertools

import numpy as np
import pytest
import torch

from combine_top_routing_gb300 import inputs as I
from combine_top_routing_gb300 import mok
from combine_top_routing_gb300.layer import MoELayer, scale_words
from mokhelp import Routed, make_layer, sha

pytestmark = pytest.mark.gpu

CASES = {
    "mx_skew_sources": I.Workload("mx_skew_sources", T=2048, d=512, E=32, k=8, F=384,
                                  dtype="mxfp8", router="sigmoid", seed=61, zipf_alpha=0.46,
                                  n_sources=8),
    "bf16": I.Workload("bf16", T=1000, d=256, E=8, k=2, F=512, dtype="bf16",
                       router="softmax", seed=62),
    # d not a multiple of 256: the GEMM role runs one CTA per tile
    "mx_d384": I.Workload("mx_d384", T=640, d=384, E=16, k=4, F=256, dtype="mxfp8",
                          router="sigmoid", seed=63),
}


def _stepwise(layer):
    """The same layer through the four step entry points."""
    w = layer.w
    R = Routed(layer)
    rows = layer.rows_pad
    if w.dtype == "mxfp8":
        xe = torch.empty((rows, w.d), dtype=torch.uint8, device="cuda")
        xs = torch.empty(scale_words(rows, w.d), dtype=torch.int32, device="cuda")
    else:
        xe = torch.empty((rows, w.d), dtype=torch.bfloat16, device="cuda")
        xs = None
    mok.dispatch(layer.cfg, layer.x_src, R.ids, R.offsets, R.pad_offsets, R.row_tok, R.row_j, xe, xs)
    ystage = torch.empty((w.T, w.k, w.d), dtype=torch.bfloat16, device="cuda")
    mok.expert_ffn(layer.cfg, xe, xs, layer.wstruct, R.offsets, R.pad_offsets, R.row_tok, R.row_j,
                   ystage, None, None, None, layer.ws)
    out = torch.empty((w.T, w.d), dtype=torch.bfloat16, device="cuda")
    mok.combine(layer.cfg, ystage, R.gates, out)
    torch.cuda.synchronize()
    return out


@pytest.mark.parametrize("name", list(CASES))
def test_fused_equals_stepwise_bit_exact(name):
    w = CASES[name]
    layer, _ = make_layer(w)
    fused = layer.forward().clone()
    torch.cuda.synchronize()
    assert layer.status() == 0
    assert torch.equal(fused, _stepwise(layer))


@pytest.mark.parametrize("name", ["mx_skew_sources", "bf16"])
def test_fused_cta_pairs_equal_single_cta_bit_exact(name):
    """d a multiple of 256: the GEMM role on CTA pairs (256-row tiles, ghost
    odd halves for experts with an odd number of row tiles) gives the same
    bits as one CTA per 128-row tile."""
    w = CASES[name]
    layer, _ = make_layer(w)
    layer.cfg.c.fused_cta_pairs = mok.MOK_PAIRS_ON
    paired = layer.forward().clone()
    torch.cuda.synchronize()
    assert layer.status() == 0
    plan = mok.fused_plan(layer.cfg)
    assert plan["cta_pairs"] == 1 and plan["gather_ctas"] % 2 == 0
    layer.cfg.c.fused_cta_pairs = mok.MOK_PAIRS_OFF
    assert mok.fused_plan(layer.cfg)["cta_pairs"] == 0
    single = layer.forward().clone()
    torch.cuda.synchronize()
    assert layer.status() == 0
    assert torch.equal(paired, single)


def test_fused_bit_identical_across_splits_minibatches_rings():
    w = CASES["mx_skew_sources"]
    inp = I.make_inputs(w, device="cuda")
    row_bytes = w.d + w.d // 32
    hashes = {}
    for frac, mb, ring_rows in itertools.product((0.125, 0.25, 1 / 3), (64, 128, 256), (0, 256, 1024)):
        layer = MoELayer(w, inp, gather_sm_fraction=frac, minibatch_rows=mb,
                         ring_bytes=ring_rows * row_bytes)
        out = layer.forward()
        torch.cuda.synchronize()
        assert layer.status() == 0, (frac, mb, ring_rows)
        hashes[(frac, mb, ring_rows)] = sha(out)
    assert len(set(hashes.values())) == 1, hashes


def test_full_size_skewed_layer_bit_identical_across_repeats_splits_minibatches():
    """[miku]: results are bit-identical whatever the schedule.  The
    DeepSeek-V3-shaped layer with Zipf-skewed routing (hottest expert about
    20x the mean), 64 source buffers and a 256 MB token ring that wraps:
    three repeats at the shape-chosen knobs, then every gather share in
    {1/8, 1/4, 1/3} x minibatch in {64, 128, 256}, all with the same output
    bytes."""
    w = I.WORKLOADS["dsv3_skew_ep"]
    layer, _ = make_layer(w)
    plan = mok.fused_plan(layer.cfg)
    assert plan["ring_rows"] < layer.rows_pad   # the ring wraps
    hashes = {}
    for rep in range(3):
        hashes[("auto", rep)] = sha(layer.forward())
    for frac, mb in itertools.product((0.125, 0.25, 1 / 3), (64, 128, 256)):
        layer.cfg.c.gather_sm_fraction = frac
        layer.cfg.c.minibatch_rows = mb
        hashes[(frac, mb)] = sha(layer.forward())
    torch.cuda.synchronize()
    assert layer.status() == 0
    assert len(set(hashes.values())) == 1, hashes


@pytest.mark.parametrize("name", ["mx_skew_sources", "bf16"])
def test_gather_first_equals_split_gather_bit_exact(name):
    """A gather share of 1: the dispatch kernel pulls whole tokens first (one
    read per token), then every CTA of the fused kernel runs the GEMM role --
    the same bits as the split gather, on one CTA per tile and on CTA pairs."""
    w = CASES[name]
    layer, _ = make_layer(w)
    ref = layer.forward().clone()
    for pairs in (mok.MOK_PAIRS_OFF, mok.MOK_PAIRS_ON):
        layer.cfg.c.fused_cta_pairs = pairs
        layer.cfg.c.gather_sm_fraction = 1.0
        plan = mok.fused_plan(layer.cfg)
        assert plan["gather_ctas"] == plan["ctas"]
        out = layer.forward().clone()
        torch.cuda.synchronize()
        assert layer.status() == 0
        assert torch.equal(out, ref), pairs


def test_gather_first_needs_an_uncapped_ring():
    w = CASES["bf16"]
    layer, _ = make_layer(w, gather_sm_fraction=1.0)
    layer.cfg.c.ring_bytes = 512 * w.d * 2
    with pytest.raises(mok.MokError) as ei:
        layer.forward()
    assert ei.value.code == mok.MOK_ERR_INVALID_ARG


def test_ring_smaller_than_a_minibatch_is_refused():
    w = CASES["bf16"]
    layer, _ = make_layer(w)
    layer.cfg.c.ring_bytes = 100 * w.d * 2   # 100 rows < 256
    with pytest.raises(mok.MokError) as ei:
        layer.forward()
    assert ei.value.code == mok.MOK_ERR_INVALID_ARG


def test_device_timeout_is_reported_and_context_stays_usable():
    # one CTA per tile and a split gather: the GEMM role waits for its first
    # minibatch of rows, a wait that a 1 ns limit cannot survive
    w = CASES["mx_skew_sources"]
    layer, _ = make_layer(w, fused_cta_pairs=mok.MOK_PAIRS_OFF, gather_sm_fraction=0.25)
    good = layer.forward().clone()
    torch.cuda.synchronize()
    assert layer.status() == 0
    # a 1 ns limit: the GEMM role cannot find its first minibatch gathered in time
    layer.cfg.c.wait_limit_ns = 1
    layer.forward()
    torch.cuda.synchronize()
    assert layer.status() == mok.MOK_ERR_TIMEOUT
    layer.cfg.c.wait_limit_ns = 0
    again = layer.forward()
    torch.cuda.synchronize()
    assert layer.status() == 0
    assert torch.equal(again, good)


def test_moe_fused_entry_equals_forward():
    w = CASES["mx_skew_sources"]
    layer, _ = make_layer(w)
    ref = layer.forward().clone()
    R = Routed(layer)
    ystage = torch.empty((w.T, w.k, w.d), dtype=torch.bfloat16, device="cuda")
    out = torch.empty((w.T, w.d), dtype=torch.bfloat16, device="cuda")
    for _ in range(2):
        mok.moe_fused(layer.cfg, layer.x_src, layer.wstruct, R.ids, R.gates, R.counts, R.offsets,
                      R.pad_offsets, R.slot_pos, R.row_tok, R.row_j, ystage, out, layer.ws)
        torch.cuda.synchronize()
        assert layer.status() == 0
        assert torch.equal(out, ref)


@pytest.mark.parametrize("name,pairs", [("bf16", mok.MOK_PAIRS_AUTO), ("bf16", mok.MOK_PAIRS_OFF),
                                        ("mx_skew_sources", mok.MOK_PAIRS_AUTO),
                                        ("mx_d384", mok.MOK_PAIRS_AUTO)])
def test_forward_chain_equals_separate_calls_bit_exact(name, pairs):
    """Macrobatch pipelining ([kucoin] §02): three back-to-back calls, each
    call's combine run inside the next call's fused kernel, with two
    workspaces alternating -- the same bits as three separate forwards."""
    w = CASES[name]
    layer, _ = make_layer(w, fused_cta_pairs=pairs)
    xs = [I.make_inputs(I.scaled(w, seed=w.seed + 100 * i), device="cuda", with_weights=False)["x"]
          for i in range(3)]
    srcs = [I.split_sources(x, w.n_sources) if w.n_sources > 1 else [x] for x in xs]
    wss = [layer.ws, torch.empty_like(layer.ws)]
    want = []
    for src in srcs:
        mok.moe_forward(layer.cfg, src, layer.W_r, layer.bias, layer.wstruct, layer.out, None, layer.ws)
        want.append(layer.out.clone())
    outs = [torch.full_like(layer.out, 7) for _ in range(3)]
    mok.moe_forward_chain(layer.cfg, srcs, layer.W_r, layer.bias, layer.wstruct, outs,
                          [wss[i % 2] for i in range(3)])
    torch.cuda.synchronize()
    for ws in wss:
        assert mok.get_device_status(ws) == 0
    for i in range(3):
        assert torch.equal(outs[i], want[i]), i


def test_forward_chain_refuses_a_shared_workspace():
    w = CASES["bf16"]
    layer, inp = make_layer(w)
    outs = [torch.empty_like(layer.out) for _ in range(2)]
    with pytest.raises(mok.MokError) as ei:
        mok.moe_forward_chain(layer.cfg, [layer.x_src, layer.x_src], layer.W_r, layer.bias, layer.wstruct,
                              outs, [layer.ws, layer.ws])
    assert ei.value.code == mok.MOK_ERR_INVALID_ARG
