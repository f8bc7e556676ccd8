"""Pins of the oracle's forward (A3-A6) and backward (B1-B6) (CPU only).

  * forward (rounding off) equals a dense-masked reformulation: every expert
    on every token, weighted by a [T,E] gate matrix that is zero off the
    top-k -- textbook, with no layout, dispatch or combine in it;
  * zero down-projection gives zero output in every mode;
  * combine: identity experts return the input within one BF16 ulp,
    one-hot gates return that expert's row exactly;
  * MXFP8 mode equals the exact GEMMs when the operands are exactly
    representable under blocking along K (and not under another blocking);
  * token-subset runs reproduce the rows of the full run bit for bit;
  * backward equals central finite differences of L = <dY, out> for every
    input, in fp64, and the softmax-renormalised logit gradient sums to 0.
"""
import numpy as np
import pytest

from oracle import oracle as O


def _tiny(seed, T=6, d=32, E=4, k=2, F=32, bias=False):
    rng = np.random.default_rng(seed)
    x = rng.standard_normal((T, d))
    Wr = rng.standard_normal((E, d)) * 0.4
    b = rng.standard_normal(E) * 0.5 if bias else None
    Wg = rng.standard_normal((E, F, d)) / np.sqrt(d)
    Wu = rng.standard_normal((E, F, d)) / np.sqrt(d)
    Wd = rng.standard_normal((E, d, F)) / np.sqrt(F)
    return x, Wr, b, Wg, Wu, Wd


def _dense_masked(x, Wr, b, Wg, Wu, Wd, k, kind):
    """Textbook MoE: out = sum_e G[:, e] * FFN_e(x) with G zero off the top-k."""
    l = x @ Wr.T + (0 if b is None else b)
    s = np.exp(l - l.max(1, keepdims=True))
    s = s / s.sum(1, keepdims=True) if kind == O.SOFTMAX else 1 / (1 + np.exp(-l))
    T, E = s.shape
    G = np.zeros((T, E))
    for t in range(T):
        top = sorted(range(E), key=lambda e: (-s[t, e], e))[:k]
        G[t, top] = s[t, top] / s[t, top].sum()
    out = np.zeros_like(x)
    for e in range(E):
        a = x @ Wg[e].T
        bb = x @ Wu[e].T
        h = a / (1 + np.exp(-a)) * bb
        out += G[:, e:e + 1] * (h @ Wd[e].T)
    return out


@pytest.mark.parametrize("kind,bias", [(O.SOFTMAX, False), (O.SIGMOID, True)])
def test_forward_equals_dense_masked_reformulation(kind, bias):
    x, Wr, b, Wg, Wu, Wd = _tiny(0, T=16, E=5, k=2, bias=bias)
    f = O.forward(x, Wr, b, lambda e: (Wg[e], Wu[e], Wd[e]), E=5, k=2, kind=kind,
                  mode="exact")
    ref = _dense_masked(x, Wr, b, Wg, Wu, Wd, 2, kind)
    assert np.allclose(f["out"], ref, rtol=1e-12, atol=1e-12)


def test_forward_rounded_modes_close_to_exact():
    x, Wr, b, Wg, Wu, Wd = _tiny(1, T=16, d=64, F=64)
    x = O.bf16_round(x)
    ge = lambda e: (O.bf16_round(Wg[e]), O.bf16_round(Wu[e]), O.bf16_round(Wd[e]))
    ex = O.forward(x, Wr, b, ge, E=4, k=2, kind=O.SOFTMAX, mode="exact")["out"]
    bf = O.forward(x, Wr, b, ge, E=4, k=2, kind=O.SOFTMAX, mode="bf16")["out"]
    mx = O.forward(x, Wr, b, ge, E=4, k=2, kind=O.SOFTMAX, mode="mxfp8")["out"]
    rel = lambda a: np.linalg.norm(a - ex) / np.linalg.norm(ex)
    assert rel(bf) < 8e-3
    assert rel(mx) < 1.5e-1   # four chained E4M3 operands (3 mantissa bits each)
    assert np.array_equal(bf, O.bf16_round(bf))


@pytest.mark.parametrize("mode", ["exact", "bf16", "mxfp8"])
def test_zero_down_projection_gives_zero(mode):
    x, Wr, b, Wg, Wu, Wd = _tiny(2)
    f = O.forward(x, Wr, b, lambda e: (Wg[e], Wu[e], 0 * Wd[e]), E=4, k=2,
                  kind=O.SIGMOID, mode=mode)
    assert np.all(f["out"] == 0)


def test_combine_identity_experts_returns_input():
    rng = np.random.default_rng(4)
    T, k, d = 64, 8, 96
    x = O.bf16_round(rng.standard_normal((T, d)))
    g = rng.uniform(0.01, 1, (T, k))
    g = O.fp32(g / g.sum(1, keepdims=True))
    ystage = np.repeat(x[:, None, :], k, axis=1)
    out = O.combine(ystage, g)
    ulp = 2.0 ** (np.floor(np.log2(np.abs(x) + 1e-300)) - 7)
    assert np.all(np.abs(out - x) <= ulp)
    assert np.allclose(O.combine(ystage, g, exact=True), x, rtol=1e-6)


def test_combine_one_hot_gates_exact():
    rng = np.random.default_rng(6)
    T, k, d = 16, 4, 64
    y = O.bf16_round(rng.standard_normal((T, k, d)))
    g = np.zeros((T, k))
    pick = rng.integers(0, k, T)
    g[np.arange(T), pick] = 1.0
    out = O.combine(y, g)
    assert np.array_equal(out, y[np.arange(T), pick])


def test_combine_contract_is_fp32_fma_chain():
    # With k = 1 the contract reduces to bf16(fp32(g * y)) -- a single
    # correctly rounded product, which fp64 computes exactly.
    rng = np.random.default_rng(8)
    y = O.bf16_round(rng.standard_normal((32, 1, 64)))
    g = O.fp32(rng.uniform(0, 1, (32, 1)))
    out = O.combine(y, g)
    assert np.array_equal(out, O.bf16_round(O.fp32(g[:, :, None] * y)[:, 0]))


def test_mxfp8_mode_equals_exact_on_representable_operands():
    rng = np.random.default_rng(12)
    T, d, E, k, F = 32, 64, 2, 1, 64
    # Each 32-wide block along d is small integers times one power of two, so
    # it is exact in MXFP8 when blocked along d; scales differ from block to
    # block and from row to row (2^0 vs 2^-16), so blocking along the rows
    # would flush the small rows to zero.
    blk_scale = 2.0 ** np.arange(-2, 2 * (d // 32) - 2, 2)
    def rep(shape):
        # |v| <= 14: the OCP scale rule maps a block maximum with mantissa
        # 1.111b (e.g. 15) above 448, where it saturates.
        v = rng.integers(-14, 15, shape).astype(float)
        row_scale = 2.0 ** (-16.0 * (np.arange(shape[0]) % 2))[:, None]
        return v * np.repeat(blk_scale, 32)[None, :shape[-1]] * row_scale / 16
    x = rep((T, d))
    Wg = np.stack([rep((F, d)) for _ in range(E)]) / 8
    Wu = np.stack([rep((F, d)) for _ in range(E)]) / 8
    Wd = rng.standard_normal((E, d, F)) / 8
    Wr = rng.standard_normal((E, d))
    assert np.array_equal(O.mx_qdq(x), x)
    assert not np.array_equal(O.mx_qdq(x.T.copy()).T, x)
    ge = lambda e: (Wg[e], Wu[e], Wd[e])
    ex = O.forward(x, Wr, None, ge, E=E, k=k, kind=O.SOFTMAX, mode="exact")
    mx = O.forward(x, Wr, None, ge, E=E, k=k, kind=O.SOFTMAX, mode="mxfp8")
    for e in ex["experts"]:
        assert np.array_equal(ex["experts"][e]["a"], mx["experts"][e]["a"])
        assert np.array_equal(ex["experts"][e]["b"], mx["experts"][e]["b"])


@pytest.mark.parametrize("mode", ["bf16", "mxfp8"])
def test_token_subset_matches_full_run(mode):
    x, Wr, b, Wg, Wu, Wd = _tiny(3, T=40, d=64, E=6, k=3, F=64, bias=True)
    ge = lambda e: (Wg[e], Wu[e], Wd[e])
    full = O.forward(x, Wr, b, ge, E=6, k=3, kind=O.SIGMOID, mode=mode)
    tok = np.array([3, 17, 0, 39, 22])
    sub = O.forward(x, Wr, b, ge, E=6, k=3, kind=O.SIGMOID, mode=mode, tokens=tok)
    assert np.array_equal(sub["out"], full["out"][tok])


def _loss_and_grads(x, Wr, b, Wg, Wu, Wd, dY, k, kind):
    E = Wr.shape[0]
    ge = lambda e: (Wg[e], Wu[e], Wd[e])
    f = O.forward(x, Wr, b, ge, E=E, k=k, kind=kind, mode="exact")
    g = O.backward(f, dY, x, Wr, ge, E=E, k=k, kind=kind, mode="exact")
    return float((dY * f["out"]).sum()), f, g


@pytest.mark.parametrize("kind", [O.SOFTMAX, O.SIGMOID])
def test_backward_matches_finite_differences(kind):
    T, d, E, k, F = 4, 8, 4, 2, 8
    x, Wr, b, Wg, Wu, Wd = _tiny(21 + kind, T=T, d=d, E=E, k=k, F=F)
    Wr = Wr * 3  # well-separated routing: no top-k flips under the probe
    dY = np.random.default_rng(99).standard_normal((T, d))
    L0, f0, g = _loss_and_grads(x, Wr, b, Wg, Wu, Wd, dY, k, kind)
    ids0 = f0["router"]["ids"].copy()
    h = 1e-6

    def fd(arr, idx):
        old = arr[idx]
        arr[idx] = old + h
        Lp, fp, _ = _loss_and_grads(x, Wr, b, Wg, Wu, Wd, dY, k, kind)
        arr[idx] = old - h
        Lm, fm, _ = _loss_and_grads(x, Wr, b, Wg, Wu, Wd, dY, k, kind)
        arr[idx] = old
        assert np.array_equal(fp["router"]["ids"], ids0)
        assert np.array_equal(fm["router"]["ids"], ids0)
        return (Lp - Lm) / (2 * h)

    def close(num, ana):
        assert abs(num - ana) <= 1e-6 * max(1.0, abs(ana)), (num, ana)

    for idx in np.ndindex(x.shape):
        close(fd(x, idx), g["dX"][idx])
    for idx in np.ndindex(Wr.shape):
        close(fd(Wr, idx), g["dWr"][idx])
    for e in range(E):
        gr = g["experts"][e]
        for idx in list(np.ndindex(Wg[e].shape))[::5]:
            close(fd(Wg, (e,) + idx), gr["dWg"][idx])
            close(fd(Wu, (e,) + idx), gr["dWu"][idx])
        for idx in list(np.ndindex(Wd[e].shape))[::5]:
            close(fd(Wd, (e,) + idx), gr["dWd"][idx])


@pytest.mark.parametrize("mode", ["exact", "bf16", "mxfp8"])
def test_empty_batch_gives_empty_outputs_and_zero_weight_gradients(mode):
    """No tokens: the layout is empty, there is no output row, and every
    gradient that sums over tokens (dW of each expert, dW_r) is the zero
    matrix of its weight's shape -- an empty sum, whatever the weights."""
    _, Wr, b, Wg, Wu, Wd = _tiny(41, T=1, d=32, E=4, k=2, F=64)
    x = np.zeros((0, 32))
    ge = lambda e: (Wg[e], Wu[e], Wd[e])
    f = O.forward(x, Wr, b, ge, E=4, k=2, kind=O.SIGMOID, mode=mode)
    assert f["out"].shape == (0, 32)
    assert np.array_equal(f["layout"]["counts"], np.zeros(4)) and np.array_equal(f["layout"]["offsets"], np.zeros(5))
    g = O.backward(f, np.zeros((0, 32)), x, Wr, ge, E=4, k=2, kind=O.SIGMOID, mode=mode, rss=True)
    assert g["dX"].shape == (0, 32) and g["dgates"].shape == (0, 2)
    assert g["dWr"].shape == (4, 32) and not g["dWr"].any()
    for e in range(4):
        assert g["experts"][e]["dWg"].shape == (64, 32) and not g["experts"][e]["dWg"].any()
        assert g["experts"][e]["dWu"].shape == (64, 32) and not g["experts"][e]["dWu"].any()
        assert g["experts"][e]["dWd"].shape == (32, 64) and not g["experts"][e]["dWd"].any()


def test_softmax_logit_grad_sums_to_zero_and_gate_grad_closed_form():
    x, Wr, b, Wg, Wu, Wd = _tiny(30, T=12)
    dY = np.random.default_rng(1).standard_normal(x.shape)
    _, f, g = _loss_and_grads(x, Wr, b, Wg, Wu, Wd, dY, 2, O.SOFTMAX)
    assert np.allclose(g["dlogits"].sum(1), 0, atol=1e-14)
    nz = (g["dlogits"] != 0).sum(1)
    assert np.all(nz <= 2)
    # dgates_tj = <dY_t, y_tj>: checked against a perturbation of the gate
    ys = f["ystage"]
    for t in range(x.shape[0]):
        for j in range(2):
            gp = f["router"]["gates"].copy()
            gp[t, j] += 1e-6
            gm = f["router"]["gates"].copy()
            gm[t, j] -= 1e-6
            num = ((dY * O.combine(ys, gp, exact=True)).sum()
                   - (dY * O.combine(ys, gm, exact=True)).sum()) / 2e-6
            assert abs(num - g["dgates"][t, j]) < 1e-7 * max(1, abs(num))


def test_mxfp8_backward_close_to_exact():
    x, Wr, b, Wg, Wu, Wd = _tiny(40, T=32, d=64, E=4, k=2, F=64)
    x = O.bf16_round(x)
    dY = O.bf16_round(np.random.default_rng(2).standard_normal(x.shape))
    ge = lambda e: (O.bf16_round(Wg[e]), O.bf16_round(Wu[e]), O.bf16_round(Wd[e]))
    res = {}
    for mode in ("exact", "bf16", "mxfp8"):
        f = O.forward(x, Wr, None, ge, E=4, k=2, kind=O.SIGMOID, mode=mode)
        res[mode] = O.backward(f, dY, x, Wr, ge, E=4, k=2, kind=O.SIGMOID, mode=mode)
    rel = lambda a, b_: np.linalg.norm(a - b_) / np.linalg.norm(b_)
    assert rel(res["bf16"]["dX"], res["exact"]["dX"]) < 1e-2
    assert rel(res["mxfp8"]["dX"], res["exact"]["dX"]) < 1e-1
    for e in range(4):
        for key in ("dWd", "dWg", "dWu"):
            assert rel(res["bf16"]["experts"][e][key], res["exact"]["experts"][e][key]) < 1e-2
            assert rel(res["mxfp8"]["experts"][e][key], res["exact"]["experts"][e][key]) < 1.5e-1


# ---------------------------------------------------------------------------
# Error scales of the reductions (used as comparison units by the GPU tests)
# ---------------------------------------------------------------------------

def test_terms_rss_brute_force():
    rng = np.random.default_rng(50)
    A, B = rng.standard_normal((7, 3)), rng.standard_normal((7, 4))
    got = O.terms_rss(A, B)
    for i in range(3):
        for j in range(4):
            assert np.isclose(got[i, j], np.sqrt(sum((A[r, i] * B[r, j]) ** 2 for r in range(7))))
    # one term: the scale is the magnitude of the sum itself
    assert np.allclose(O.terms_rss(A[:1], B[:1]), np.abs(A[:1].T @ B[:1]))


def test_gate_grad_rss_brute_force():
    rng = np.random.default_rng(51)
    dY, y = rng.standard_normal((3, 5)), rng.standard_normal((3, 2, 5))
    got = O.gate_grad_rss(dY, y)
    for t in range(3):
        for j in range(2):
            assert np.isclose(got[t, j], np.sqrt(np.sum((dY[t] * y[t, j]) ** 2)))


@pytest.mark.parametrize("kind", [O.SOFTMAX, O.SIGMOID])
def test_router_bwd_rss_uses_the_jacobian_of_the_router_backward(kind):
    """router_bwd is linear in dgates: its Jacobian, taken column by column
    from router_bwd itself, propagates per-gate scales in quadrature."""
    rng = np.random.default_rng(52 + kind)
    T, d, E, k = 5, 8, 6, 3
    x, Wr = rng.standard_normal((T, d)), rng.standard_normal((E, d))
    r = O.router(x, Wr, None, k, kind)
    dg_rss = rng.uniform(0.5, 2.0, (T, k))
    got = O.router_bwd_rss(r["scores"], r["ids"], r["gates"], dg_rss, kind)
    base = O.router_bwd(x, Wr, r["scores"], r["ids"], r["gates"], np.zeros((T, k)), kind)["dlogits"]
    want = np.zeros((T, E))
    for jp in range(k):
        unit = np.zeros((T, k))
        unit[:, jp] = 1.0
        col = O.router_bwd(x, Wr, r["scores"], r["ids"], r["gates"], unit, kind)["dlogits"] - base
        want += (col * dg_rss[:, jp:jp + 1]) ** 2
    assert np.allclose(got, np.sqrt(want), rtol=1e-12, atol=1e-15)
