"""GPU parity of A4/A5 (tcgen05 grouped SwiGLU FFN, BF16 and MXFP8) and of
the whole forward layer against the oracle, plus bit-reproducibility.

The oracle is fed the GPU's routing (ids, gates) so that fp near-ties in the
router cannot flip an expert choice; everything after routing is the
oracle's own arithmetic from the BF16 inputs (its own dispatch, its own MXFP8
quantisation of x, the weights and h).  Tolerance: relative L2 <= 5e-3 and
max-abs <= 2e-2 on the BF16 outputs."""
import numpy as np
import pytest
import torch

from combine_top_routing_gb300 import inputs as I
from oracle import oracle as O
from mokhelp import (Routed, bf16_np, check_close, expert_weights_np, f32_np, make_layer, sha)

pytestmark = pytest.mark.gpu

SMALL = {
    "tiny": I.WORKLOADS["tiny"],
    "bf16_ragged": I.Workload("bf16_ragged", T=300, d=256, E=8, k=2, F=384, dtype="bf16",
                              router="softmax", seed=31),
    "mx_ragged": I.Workload("mx_ragged", T=520, d=384, E=16, k=4, F=256, dtype="mxfp8",
                            router="sigmoid", seed=32, zipf_alpha=0.46),
    "mx_sources": I.Workload("mx_sources", T=512, d=512, E=32, k=8, F=384, dtype="mxfp8",
                             router="sigmoid", seed=33, n_sources=4),
    "bf16_many_empty": I.Workload("bf16_many_empty", T=16, d=256, E=64, k=2, F=256,
                                  dtype="bf16", router="sigmoid", seed=34),
    "mx_one_token": I.Workload("mx_one_token", T=1, d=128, E=4, k=4, F=128, dtype="mxfp8",
                               router="softmax", seed=35),
    # degenerate routing: one expert takes every token (gate 1, three row tiles,
    # so the CTA-pair tiles end in a ghost half) and top-1 over four experts
    "bf16_single_expert": I.Workload("bf16_single_expert", T=300, d=256, E=1, k=1, F=256,
                                     dtype="bf16", router="softmax", seed=36),
    "mx_top1": I.Workload("mx_top1", T=257, d=256, E=4, k=1, F=128, dtype="mxfp8",
                          router="sigmoid", seed=37),
    # the largest expert count and top-k the library takes (1024, 8): about
    # three rows per expert, so nearly every row tile is a ragged tail, and the
    # kernels' per-expert tables are full (BF16 on CTA pairs, MXFP8 on single CTAs)
    "bf16_max_experts": I.Workload("bf16_max_experts", T=384, d=256, E=1024, k=8, F=256,
                                   dtype="bf16", router="softmax", seed=38),
    "mx_max_experts": I.Workload("mx_max_experts", T=384, d=256, E=1024, k=8, F=256,
                                 dtype="mxfp8", router="sigmoid", seed=39),
}


def _oracle_out(w, inp, R, tokens):
    x = bf16_np(inp["x"])
    ids = R.ids.cpu().numpy()[tokens]
    gates = f32_np(R.gates)[tokens]
    ge = lambda e: expert_weights_np(inp, e)
    ref = O.forward(x, f32_np(inp["Wr"]), None if inp["bias"] is None else f32_np(inp["bias"]),
                    ge, E=w.E, k=w.k, kind=O.SOFTMAX if w.router == "softmax" else O.SIGMOID,
                    mode=w.dtype, tokens=tokens, ids=ids, gates=gates)
    return ref


@pytest.mark.parametrize("name", list(SMALL))
def test_forward_small_full_parity(name):
    w = SMALL[name]
    layer, inp = make_layer(w, training=True)
    out = layer.forward()
    torch.cuda.synchronize()
    assert layer.status() == 0
    R = Routed(layer)  # same routing as the forward (bit-reproducible)
    torch.cuda.synchronize()
    tokens = np.arange(w.T)
    ref = _oracle_out(w, inp, R, tokens)
    # the forward's saved routing equals a fresh route_layout call
    ids_ctx = layer.ctx_view("ids", torch.int32, (w.T, w.k))
    assert torch.equal(ids_ctx, R.ids)
    # ystage rows (push to staging) and the combined output
    ystage = layer.ctx_view("ystage", torch.bfloat16, (w.T, w.k, w.d))
    check_close(bf16_np(ystage), ref["ystage"], what="ystage")
    check_close(bf16_np(out), ref["out"], what="out")
    # combine is bit-exact given the GPU's own ystage and gates
    assert np.array_equal(bf16_np(out), O.combine(bf16_np(ystage), f32_np(R.gates)))


@pytest.mark.parametrize("name", ["mixtral_bf16", "dsv3_mxfp8", "dsv3_skew_ep"])
def test_forward_full_size_sampled(name):
    w = I.WORKLOADS[name]
    layer, inp = make_layer(w, training=True)
    out = layer.forward()
    torch.cuda.synchronize()
    assert layer.status() == 0
    R = Routed(layer)
    torch.cuda.synchronize()
    # 64 tokens: one routed to the hottest expert, one to the coldest expert
    # that has rows, the rest drawn at random
    ids = R.ids.cpu().numpy()
    counts = np.bincount(ids.reshape(-1), minlength=w.E)
    hot = int(np.argmax(counts))
    cold = int(np.argmin(np.where(counts > 0, counts, 1 << 30)))
    rng = np.random.default_rng(w.seed + 100)
    picked = {int(np.nonzero((ids == hot).any(1))[0][0]), int(np.nonzero((ids == cold).any(1))[0][0])}
    rest = rng.permutation(w.T)
    tokens = np.sort(np.array(list(picked) + [int(t) for t in rest if t not in picked][:64 - len(picked)]))
    assert len(tokens) == 64 and (ids[tokens] == hot).any() and (ids[tokens] == cold).any()
    ref = _oracle_out(w, inp, R, tokens)
    check_close(bf16_np(out[torch.from_numpy(tokens).cuda()]), ref["out"], what="out")
    ystage = layer.ctx_view("ystage", torch.bfloat16, (w.T, w.k, w.d))
    ys = bf16_np(ystage[torch.from_numpy(tokens).cuda()])
    check_close(ys, ref["ystage"], what="ystage")
    # combine bit-exact on the sampled tokens given the GPU's ystage and gates
    g = f32_np(R.gates)[tokens]
    assert np.array_equal(bf16_np(out[torch.from_numpy(tokens).cuda()]), O.combine(ys, g))


def test_forward_bit_reproducible():
    w = SMALL["mx_sources"]
    layer, _ = make_layer(w)
    hashes = set()
    for _ in range(3):
        hashes.add(sha(layer.forward()))
    torch.cuda.synchronize()
    assert len(hashes) == 1
    w2 = SMALL["bf16_ragged"]
    layer2, _ = make_layer(w2)
    assert sha(layer2.forward()) == sha(layer2.forward())
