"""GPU parity of the HBM-bound steps: A3 dispatch (BF16 copy and fused MXFP8
quantisation), the MXFP8 weight quantiser (both blockings) and A6 combine --
all bit-exact against the oracle given the same inputs."""
import numpy as np
import pytest
import torch

from combine_top_routing_gb300 import inputs as I
from combine_top_routing_gb300 import mok
from combine_top_routing_gb300.layer import scale_words
from oracle import oracle as O
from mokhelp import Routed, bf16_np, f32_np, make_layer, scales_to_canonical

pytestmark = pytest.mark.gpu

CASES = {
    "bf16_ragged": I.Workload("bf16_ragged", T=300, d=256, E=8, k=2, F=384, dtype="bf16",
                              router="softmax", seed=21),
    "mx_ragged": I.Workload("mx_ragged", T=520, d=384, E=16, k=4, F=256, dtype="mxfp8",
                            router="sigmoid", seed=22, zipf_alpha=0.46),
    "mx_sources": I.Workload("mx_sources", T=512, d=512, E=32, k=8, F=256, dtype="mxfp8",
                             router="sigmoid", seed=23, n_sources=4),
}


def _dispatch(layer, R):
    w = layer.w
    rows = layer.rows_pad
    if w.dtype == "mxfp8":
        xe = torch.empty((rows, w.d), dtype=torch.uint8, device="cuda")
        sc = torch.zeros(scale_words(rows, w.d), dtype=torch.int32, device="cuda")
    else:
        xe = torch.empty((rows, w.d), dtype=torch.bfloat16, device="cuda")
        sc = None
    mok.dispatch(layer.cfg, layer.x_src, R.ids, R.offsets, R.pad_offsets, R.row_tok, R.row_j, xe, sc)
    torch.cuda.synchronize()
    return xe, sc


@pytest.mark.parametrize("name", list(CASES))
def test_dispatch_bit_exact(name):
    w = CASES[name]
    layer, inp = make_layer(w)
    R = Routed(layer)
    xe, sc = _dispatch(layer, R)
    ids = R.ids.cpu().numpy()
    off = R.offsets.cpu().numpy()
    pad = R.pad_offsets.cpu().numpy()
    row_tok = R.row_tok.cpu().numpy()
    x = bf16_np(inp["x"])
    # dense row p of expert e -> padded row pad[e] + p - off[e]
    e_of_p = np.repeat(np.arange(w.E), np.diff(off))
    q = pad[e_of_p] + np.arange(w.S) - off[e_of_p]
    ref = O.dispatch(x, row_tok, w.dtype)
    if w.dtype == "mxfp8":
        codes = xe.cpu().numpy()[q]
        assert np.array_equal(codes, ref["codes"])
        scales = scales_to_canonical(sc, layer.rows_pad, w.d)[q]
        assert np.array_equal(scales, ref["scales"])
    else:
        assert np.array_equal(bf16_np(xe)[q], ref["xe"])
    assert np.all(ids.reshape(-1)[np.argsort(R.slot_pos.cpu().numpy().reshape(-1))] == e_of_p)


@pytest.mark.parametrize("name", list(CASES))
def test_dispatch_by_token_equals_pull_dispatch(name):
    """One read per token, written into its k slots: the same bytes (codes,
    scales, padding rows untouched) as the per-slot pull."""
    w = CASES[name]
    layer, _ = make_layer(w)
    R = Routed(layer)
    rows = layer.rows_pad
    outs = []
    for by_token in (False, True):
        if w.dtype == "mxfp8":
            xe = torch.zeros((rows, w.d), dtype=torch.uint8, device="cuda")
            sc = torch.zeros(scale_words(rows, w.d), dtype=torch.int32, device="cuda")
        else:
            xe = torch.zeros((rows, w.d), dtype=torch.bfloat16, device="cuda")
            sc = None
        if by_token:
            mok.dispatch_by_token(layer.cfg, layer.x_src, R.ids, R.slot_pos, R.offsets, R.pad_offsets, xe, sc)
        else:
            mok.dispatch(layer.cfg, layer.x_src, R.ids, R.offsets, R.pad_offsets, R.row_tok, R.row_j, xe, sc)
        torch.cuda.synchronize()
        outs.append((xe, sc))
    assert torch.equal(outs[0][0], outs[1][0])
    if w.dtype == "mxfp8":
        assert torch.equal(outs[0][1], outs[1][1])


@pytest.mark.parametrize("E,rows,K", [(2, 256, 384), (3, 384, 256), (1, 128, 128)])
def test_weight_quantiser_bit_exact_both_blockings(E, rows, K):
    g = torch.Generator(device="cuda")
    g.manual_seed(E * 1000 + rows + K)
    src = (torch.randn((E, rows, K), device="cuda", generator=g) *
           torch.exp(torch.randn((E, rows, 1), device="cuda", generator=g) * 3)).to(torch.bfloat16)
    src[0, 0, :64] = 0  # an all-zero block
    codes = torch.empty((E, rows, K), dtype=torch.uint8, device="cuda")
    sc = torch.empty(scale_words(E * rows, K), dtype=torch.int32, device="cuda")
    mok.quantize_mx(src, E, rows, K, 0, codes, sc)
    codes_t = torch.empty((E, K, rows), dtype=torch.uint8, device="cuda")
    sc_t = torch.empty(scale_words(E * K, rows), dtype=torch.int32, device="cuda")
    mok.quantize_mx(src, E, rows, K, 1, codes_t, sc_t)
    torch.cuda.synchronize()
    a = bf16_np(src).reshape(E * rows, K)
    rc, rs = O.mx_quantize(a)
    assert np.array_equal(codes.cpu().numpy().reshape(E * rows, K), rc)
    assert np.array_equal(scales_to_canonical(sc, E * rows, K), rs)
    at = bf16_np(src).transpose(0, 2, 1).reshape(E * K, rows)
    rct, rst = O.mx_quantize(at)
    assert np.array_equal(codes_t.cpu().numpy().reshape(E * K, rows), rct)
    assert np.array_equal(scales_to_canonical(sc_t, E * K, rows), rst)


def test_weight_quantiser_full_size_sampled_rows():
    w = I.WORKLOADS["dsv3_mxfp8"]
    wsmall = I.scaled(w, E=8)
    inp = I.make_inputs(wsmall, device="cuda")
    E, F, d = wsmall.E, wsmall.F, wsmall.d
    codes = torch.empty((E, F, d), dtype=torch.uint8, device="cuda")
    sc = torch.empty(scale_words(E * F, d), dtype=torch.int32, device="cuda")
    mok.quantize_mx(inp["Wg"], E, F, d, 0, codes, sc)
    torch.cuda.synchronize()
    rows = np.random.default_rng(0).choice(E * F, 64, replace=False)
    a = bf16_np(inp["Wg"].reshape(E * F, d)[torch.from_numpy(rows).cuda()])
    rc, rs = O.mx_quantize(a)
    assert np.array_equal(codes.reshape(E * F, d).cpu().numpy()[rows], rc)
    assert np.array_equal(scales_to_canonical(sc, E * F, d)[rows], rs)


@pytest.mark.parametrize("T,k,d", [(300, 2, 256), (64, 8, 7168), (1, 1, 128)])
def test_combine_bit_exact(T, k, d):
    g = torch.Generator(device="cuda")
    g.manual_seed(T + k + d)
    y = torch.randn((T, k, d), device="cuda", generator=g).to(torch.bfloat16)
    gates = torch.rand((T, k), device="cuda", generator=g)
    gates = gates / gates.sum(1, keepdim=True)
    cfg = mok.Config(T, d, max(k, 2), k, 128, 0, 0)
    out = torch.empty((T, d), dtype=torch.bfloat16, device="cuda")
    mok.combine(cfg, y, gates, out)
    torch.cuda.synchronize()
    ref = O.combine(bf16_np(y), f32_np(gates))
    assert np.array_equal(bf16_np(out), ref)


def test_swiglu_h_quantisation_bit_exact_given_the_same_fp32_input():
    """MXFP8 quantisation of h ([kucoin] §02: fused into SwiGLU), checked the
    way the contract states it: given the GPU's own fp32 SwiGLU output, its
    E4M3 codes and E8M0 scales (blocks of 32 along F) equal the oracle's
    quantisation of those fp32 values bit for bit.  mok_swiglu_quantize_mx
    runs the FFN1 epilogue's own SwiGLU and block quantiser on fp32 a, b
    from memory.  Rows cover the edge cases: an all-zero block (scale byte 0),
    rows scaled by 2^-20 .. 2^6 (h from about 2^-80 to 2^12; elements far
    below their block maximum get subnormal codes), a block whose maximum has
    mantissa 1.111b (saturates at 448), and random N(0,1) accumulators."""
    rows, F = 256, 512
    g = torch.Generator(device="cpu").manual_seed(61)
    a = torch.randn((rows, F), generator=g, dtype=torch.float64)
    b = torch.randn((rows, F), generator=g, dtype=torch.float64)
    row_scale = 2.0 ** torch.randint(-20, 7, (rows, 1), generator=g).double()
    a, b = a * row_scale, b * row_scale
    a[3, 32:64] = 0.0                                  # h = 0 over one block: scale byte 0
    b[5] *= 2.0 ** -20                                 # tiny h: scale exponents near -60
    a[7, :32], b[7, :32] = 20.0, 192.0                 # silu(20) = 20 in fp32: h = 3840 = 1.111b x 2^11,
    #                                                    which the OCP scale rule saturates to 448 x 2^3
    a, b = a.float().cuda(), b.float().cuda()
    h = torch.empty((rows, F), dtype=torch.float32, device="cuda")
    codes = torch.empty((rows, F), dtype=torch.uint8, device="cuda")
    scales = torch.zeros(scale_words(rows, F), dtype=torch.int32, device="cuda")
    mok.swiglu_quantize_mx(a, b, rows, F, h, codes, scales)
    torch.cuda.synchronize()
    hv = h.double().cpu().numpy()
    ref_codes, ref_scales = O.mx_quantize(hv)
    assert np.array_equal(codes.cpu().numpy(), ref_codes)
    assert np.array_equal(scales_to_canonical(scales, rows, F), ref_scales)
    # h = silu(0) b = +-0: scale byte 0, codes +0 (0x00) or -0 (0x80)
    assert ref_scales[3, 1] == 0 and ((ref_codes[3, 32:64] & 0x7F) == 0).all()
    assert ref_scales[7, 0] == 127 + 3 and ref_codes[7, 0] == 0x7E
    # the fp32 SwiGLU itself: within a few fp32 ulps of the fp64 formula
    ref_h = O.swiglu(a.double().cpu().numpy(), b.double().cpu().numpy())
    assert np.all(np.abs(hv - ref_h) <= 1e-5 * np.abs(ref_h) + 1e-30)
