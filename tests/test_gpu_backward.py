"""GPU parity of the backward layer (B1-B6) against the oracle, and bit
reproducibility.

Small layers are compared in full: the oracle runs its own forward and
backward from the BF16 inputs with the GPU's routing injected.  The
DeepSeek-V3-shaped MXFP8 forward+backward is checked on sampled tokens (dX,
dgates, dlogits) and on sampled experts for the weight gradients, where the
oracle's wgrad step is fed the GPU's step-boundary operands (dy rows, saved
h, da, db and the gathered x rows) and quantises them itself.  Tolerance:
relative L2 <= 5e-3 and max-abs <= 2e-2 (BF16 / fp32-accumulated), the
max-abs error of a reduction's element (dgates, dlogits, dW_r, dW) measured
against the root-sum-square of its terms where that exceeds max(1, |ref|)
(see mokhelp); MXFP8 weight gradients end to end: max-abs <= 2^-4 in the same
units (mokhelp.MAX_ABS_MX_CHAIN)."""
import numpy as np
import pytest
import torch

from combine_top_routing_gb300 import inputs as I
from combine_top_routing_gb300 import mok
from oracle import oracle as O
from mokhelp import (MAX_ABS_MX_CHAIN, bf16_np, check_close, expert_weights_np, f32_np,
                     make_layer, sha)

pytestmark = pytest.mark.gpu

SMALL = {
    "tiny": I.WORKLOADS["tiny"],
    "bf16_ragged": I.Workload("bf16_ragged", T=300, d=256, E=8, k=2, F=384, dtype="bf16",
                              router="softmax", seed=41),
    "mx_ragged": I.Workload("mx_ragged", T=520, d=384, E=16, k=4, F=256, dtype="mxfp8",
                            router="sigmoid", seed=42, zipf_alpha=0.46),
    "mx_sources": I.Workload("mx_sources", T=512, d=512, E=32, k=8, F=384, dtype="mxfp8",
                             router="sigmoid", seed=43, n_sources=4),
    "bf16_many_empty": I.Workload("bf16_many_empty", T=16, d=256, E=64, k=2, F=256,
                                  dtype="bf16", router="sigmoid", seed=44),
    # d and F multiples of 256: every weight-gradient GEMM runs on CTA pairs
    "mx_pairs": I.Workload("mx_pairs", T=600, d=512, E=16, k=4, F=512, dtype="mxfp8",
                           router="sigmoid", seed=45),
    # ~1000 token rows per expert: the weight-gradient K (an expert's rows) spans
    # more stages than the operand ring holds, so the ring wraps inside a tile
    "bf16_bigk": I.Workload("bf16_bigk", T=2048, d=256, E=4, k=2, F=256, dtype="bf16",
                            router="softmax", seed=46),
    "mx_bigk": I.Workload("mx_bigk", T=2048, d=256, E=4, k=2, F=256, dtype="mxfp8",
                          router="sigmoid", seed=47),
    # degenerate routing: one slot per token, and a single expert taking every token
    "bf16_top1": I.Workload("bf16_top1", T=300, d=256, E=8, k=1, F=256, dtype="bf16",
                            router="softmax", seed=48),
    "mx_one_expert": I.Workload("mx_one_expert", T=384, d=256, E=1, k=1, F=256, dtype="mxfp8",
                                router="sigmoid", seed=49),
    # the largest expert count and top-k (1024, 8): most experts have a few
    # rows or none, every weight gradient of an expert without rows is zero
    "mx_max_experts": I.Workload("mx_max_experts", T=384, d=256, E=1024, k=8, F=256,
                                 dtype="mxfp8", router="sigmoid", seed=40),
}


def _kind(w):
    return O.SOFTMAX if w.router == "softmax" else O.SIGMOID


def _run(w):
    layer, inp = make_layer(w, training=True)
    layer.prepare_backward()
    layer.forward()
    layer.backward(inp["dY"])
    torch.cuda.synchronize()
    assert layer.status() == 0
    return layer, inp


def _routing(layer, w):
    ids = layer.ctx_view("ids", torch.int32, (w.T, w.k)).cpu().numpy()
    gates = f32_np(layer.ctx_view("gates", torch.float32, (w.T, w.k)))
    return ids, gates


@pytest.mark.parametrize("name", list(SMALL))
def test_backward_small_full_parity(name):
    w = SMALL[name]
    layer, inp = _run(w)
    ids, gates = _routing(layer, w)
    x = bf16_np(inp["x"])
    Wr = f32_np(inp["Wr"])
    bias = None if inp["bias"] is None else f32_np(inp["bias"])
    ge = lambda e: expert_weights_np(inp, e)
    f = O.forward(x, Wr, bias, ge, E=w.E, k=w.k, kind=_kind(w), mode=w.dtype, ids=ids, gates=gates)
    g = O.backward(f, bf16_np(inp["dY"]), x, Wr, ge, E=w.E, k=w.k, kind=_kind(w), mode=w.dtype,
                   rss=True)
    check_close(f32_np(layer.dgates), g["dgates"], what="dgates", scale=g["dgates_rss"])
    # B1 at its step boundary: the GPU's own ystage and gates into the
    # oracle's reverse-combine -- dy rows bit-exact, dgates to fp32 accuracy
    ystage = bf16_np(layer.ctx_view("ystage", torch.bfloat16, (w.T, w.k, w.d)))
    dy_ref, dg_ref = O.rev_combine(bf16_np(inp["dY"]), gates, ystage)
    slot_pos = layer.ctx_view("slot_pos", torch.int32, (w.T, w.k)).cpu().numpy()
    off = layer.ctx_view("offsets", torch.int32, (w.E + 1,)).cpu().numpy()
    pad = layer.ctx_view("pad_offsets", torch.int32, (w.E + 1,)).cpu().numpy()
    q = pad[ids] + slot_pos - off[ids]
    R = layer.rows_pad
    dy_rows = bf16_np(_bwd_view(layer, "dy", torch.bfloat16, (R, w.d)))
    assert np.array_equal(dy_rows[q.reshape(-1)], dy_ref.reshape(-1, w.d))
    # B5 at its step boundary: the GPU's dx rows and chosen-logit gradients
    # through the oracle's reverse dispatch (contract: fp32, slot rows then
    # router terms in ascending j, fused multiply-adds) -- dX bit for bit
    dx_rows = bf16_np(_bwd_view(layer, "dx", torch.bfloat16, (R, w.d)))
    dl_sel = f32_np(_bwd_view(layer, "dl_sel", torch.float32, (w.T, w.k)))
    dX_step = O.rev_dispatch(dx_rows, q.astype(np.int32), ids, dl_sel, Wr)
    assert np.array_equal(bf16_np(layer.dX), dX_step)
    dg = f32_np(layer.dgates)
    assert np.all(np.abs(dg - dg_ref) <= 1e-5 * (1 + np.abs(dg_ref)) + 1e-6 * w.d)
    check_close(f32_np(layer.dlogits), g["dlogits"], what="dlogits", scale=g["dlogits_rss"])
    check_close(bf16_np(layer.dX), g["dX"], what="dX")
    check_close(f32_np(layer.dW_r), g["dWr"], what="dW_r", scale=g["dWr_rss"])
    st = {key: np.stack([g["experts"][e][key] for e in range(w.E)])
          for key in ("dWg", "dWu", "dWd", "dWg_rss", "dWu_rss", "dWd_rss")}
    if w.dtype == "mxfp8":
        # End to end the MXFP8 chain gets its own element bound (MAX_ABS_MX_CHAIN:
        # re-quantised operands can differ by one E4M3 step); the contract's
        # 2e-2 holds at the step boundary, the GPU's own saved operands through
        # the oracle's weight-gradient step
        for name, key in (("d_gate", "dWg"), ("d_up", "dWu"), ("d_down", "dWd")):
            check_close(bf16_np(layer.grads[name]), st[key], mabs=MAX_ABS_MX_CHAIN,
                        what=f"{key} (chain)", scale=st[key + "_rss"])
        _check_wgrad_step(layer, inp, w, ids, range(w.E))
    else:
        for name, key in (("d_gate", "dWg"), ("d_up", "dWu"), ("d_down", "dWd")):
            check_close(bf16_np(layer.grads[name]), st[key], what=key, scale=st[key + "_rss"])
    counts = np.bincount(ids.reshape(-1), minlength=w.E)
    for e in np.where(counts == 0)[0]:
        assert not layer.grads["d_gate"][e].any() and not layer.grads["d_down"][e].any()


@pytest.mark.parametrize("name,ntok", [("dsv3_fwdbwd", 16), ("mixtral_bf16", 16)])
def test_backward_full_size_sampled(name, ntok):
    """Full-size layers: the DeepSeek-V3-shaped MXFP8 forward+backward and the
    Mixtral-shaped BF16 one (its dgrad GEMM has K = 2F = 28672).  dX, dgates
    and dlogits on sampled tokens end to end; the weight gradients of the
    hottest and the coldest expert at their step boundary (all their rows)."""
    w = I.WORKLOADS[name]
    layer, inp = _run(w)
    ids, gates = _routing(layer, w)
    rng = np.random.default_rng(7)
    tokens = np.sort(rng.choice(w.T, ntok, replace=False))
    x = bf16_np(inp["x"])
    Wr = f32_np(inp["Wr"])
    bias = None if inp["bias"] is None else f32_np(inp["bias"])
    ge = lambda e: expert_weights_np(inp, e)
    f = O.forward(x, Wr, bias, ge, E=w.E, k=w.k, kind=_kind(w), mode=w.dtype, tokens=tokens,
                  ids=ids[tokens], gates=gates[tokens])
    dY = bf16_np(inp["dY"][torch.from_numpy(tokens).cuda()])
    g = O.backward(f, dY, x, Wr, ge, E=w.E, k=w.k, kind=_kind(w), mode=w.dtype, rss=True)
    tk = torch.from_numpy(tokens).cuda()
    check_close(bf16_np(layer.dX[tk]), g["dX"], what="dX")
    check_close(f32_np(layer.dgates[tk]), g["dgates"], what="dgates", scale=g["dgates_rss"])
    check_close(f32_np(layer.dlogits[tk]), g["dlogits"], what="dlogits", scale=g["dlogits_rss"])

    # weight gradients of sampled experts from the GPU's step-boundary operands
    counts = layer.ctx_view("counts", torch.int32, (w.E,)).cpu().numpy()
    sampled = (int(np.argmax(counts)), int(np.argmin(np.where(counts > 0, counts, 1 << 30))))
    _check_wgrad_step(layer, inp, w, ids, sampled)
    for e in sampled:
        # router weight gradient of e: only tokens routed to e carry dlogits[:, e]
        sel = np.where((ids == e).any(1))[0]
        sc = f32_np(layer.ctx_view("sel_scores", torch.float32, (w.T, w.k)))
        scores = np.zeros((len(sel), w.E))
        np.put_along_axis(scores, ids[sel].astype(np.int64), sc[sel], 1)
        rb = O.router_bwd(x[sel], Wr, scores, ids[sel], gates[sel], f32_np(layer.dgates)[sel], _kind(w))
        check_close(f32_np(layer.dW_r[e]), rb["dWr"][e], what=f"dW_r[{e}]")


def _check_wgrad_step(layer, inp, w, ids, experts):
    """B4 at its step boundary: the GPU's saved h and its dy, da, db rows and
    the tokens' x rows through the oracle's weight-gradient step, for the
    given experts, against the GPU's dW."""
    R = layer.rows_pad
    x = bf16_np(inp["x"])
    counts = layer.ctx_view("counts", torch.int32, (w.E,)).cpu().numpy()
    pad = layer.ctx_view("pad_offsets", torch.int32, (w.E + 1,)).cpu().numpy()
    off = layer.ctx_view("offsets", torch.int32, (w.E + 1,)).cpu().numpy()
    row_tok = layer.ctx_view("row_tok", torch.int32, (w.S,)).cpu().numpy()
    h = layer.ctx_view("h", torch.bfloat16, (R, w.F))
    dy_rows = _bwd_view(layer, "dy", torch.bfloat16, (R, w.d))
    da = _bwd_view(layer, "da", torch.bfloat16, (R, w.F))
    db = _bwd_view(layer, "db", torch.bfloat16, (R, w.F))
    for e in experts:
        if counts[e] == 0:
            continue
        rows = slice(int(pad[e]), int(pad[e]) + int(counts[e]))
        toks = row_tok[off[e]:off[e] + counts[e]]
        ref = O.expert_wgrad(bf16_np(dy_rows[rows]), bf16_np(h[rows]), bf16_np(da[rows]),
                             bf16_np(db[rows]), x[toks], w.dtype, rss=True)
        for name, key in (("d_down", "dWd"), ("d_gate", "dWg"), ("d_up", "dWu")):
            check_close(bf16_np(layer.grads[name][e]), ref[key], what=f"{key}[{e}]",
                        scale=ref[key + "_rss"])


def _bwd_view(layer, field, dtype, shape):
    """A view of one intermediate of the backward workspace (mok_bwd_ws_layout)."""
    off = getattr(mok.bwd_ws_layout(layer.cfg), field)
    n = int(np.prod(shape)) * torch.tensor([], dtype=dtype).element_size()
    return layer.bws[off:off + n].view(dtype).view(shape)


def test_backward_bit_reproducible():
    w = SMALL["mx_sources"]
    layer, inp = make_layer(w, training=True)
    layer.prepare_backward()
    hashes = set()
    for _ in range(3):
        layer.forward()
        layer.backward(inp["dY"])
        hashes.add((sha(layer.dX), sha(layer.grads["d_gate"]), sha(layer.grads["d_down"]),
                    sha(layer.dW_r), sha(layer.dgates)))
    torch.cuda.synchronize()
    assert len(hashes) == 1


@pytest.mark.parametrize("name", ["mx_pairs", "bf16_many_empty", "mx_sources", "mx_bigk"])
def test_wgrad_cta_pairs_equal_single_cta(name):
    """The weight-gradient GEMMs on CTA pairs (256 dW rows per pair tile)
    give the same bits as one CTA per 128-row tile, experts without rows
    included (their dW blocks are zero)."""
    w = SMALL[name]
    layer, inp = make_layer(w, training=True)
    layer.prepare_backward()
    layer.forward()
    grads = {}
    for pair in ("0", "1"):
        layer.cfg.c.gemm_cta_pairs = mok.MOK_PAIRS_ON if pair == "1" else mok.MOK_PAIRS_OFF
        layer.backward(inp["dY"])
        torch.cuda.synchronize()
        grads[pair] = {k: v.clone() for k, v in layer.grads.items()}
        grads[pair]["dX"] = layer.dX.clone()
    for k in grads["0"]:
        assert torch.equal(grads["0"][k], grads["1"][k]), k
