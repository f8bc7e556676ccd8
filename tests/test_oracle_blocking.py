"""Pins of the oracle's MXFP8 blocking axes and of the backward's contract
rounding (CPU only).

MXFP8 ("Cursor's MoK achieves 2.37x performance boost on NVIDIA GB300
NVL72", kucoin.com, §02: quantisation fused into dispatch, the grouped GEMM
and SwiGLU) shares one scale between 32 consecutive elements along a GEMM's
K.  Each test below builds operands that are exactly representable when
blocked along the axis the contract names and are NOT representable under
the plausible wrong blocking (the other axis, a longer block, a different
pad).  With exact operands every MXFP8-mode result must equal the same step
without quantisation (BF16 mode) bit for bit; with the wrong blocking some
operand would lose bits and the equality would fail.

Scales are made to differ by 2^20 along the wrong axis: a block then spans
more than the 2^17 that E4M3 covers below its maximum (8 binades of normals,
9 bits of subnormals), so its small elements flush to zero.

The contract rounding of reverse-combine and reverse-dispatch is pinned by the
hand-worked cases in tests/golden/contract_rounding.txt.
"""
import os

import numpy as np
import pytest

from oracle import oracle as O

GOLDEN = os.path.join(os.path.dirname(__file__), "golden", "contract_rounding.txt")
BIG = 2.0 ** 20


def _ints(rng, shape, lo=-14, hi=14):
    # |v| <= 14 keeps a block maximum below the 15 * 2^e values that the OCP
    # scale rule saturates (see the golden MXFP8 blocks)
    return rng.integers(lo, hi + 1, shape).astype(float)


def _alternating(n):
    """1, 2^-20, 1, 2^-20, ... -- per-index scales 2^20 apart."""
    return np.where(np.arange(n) % 2 == 0, 1.0, 1.0 / BIG)


def _exact_along_last(a):
    return np.array_equal(O.mx_qdq(a), a)


# ---------------------------------------------------------------------------
# Forward, FFN2: h blocked along F, W_d blocked along F
# ---------------------------------------------------------------------------

def test_mxfp8_ffn2_blocks_h_and_w_down_along_F():
    rng = np.random.default_rng(101)
    T, d, F = 64, 64, 64
    # token rows scaled 1 / 2^10 alternately; x has one non-zero element per row
    c = np.where(np.arange(T) % 2 == 0, 1.0, 2.0 ** 10)
    x = np.zeros((T, d))
    x[:, 0] = c
    # a = 64 c >= 64: silu(a) = a exactly in fp64 (exp(-64) < 2^-53), so
    # h = a * b = 64 c^2 v_f with v_f small integers times a per-32-block scale
    Wg = np.zeros((1, F, d))
    Wg[0, :, 0] = 64.0
    v = _ints(rng, F) * np.repeat(2.0 ** np.array([0.0, -3.0]), 32)
    Wu = np.zeros((1, F, d))
    Wu[0, :, 0] = v
    # W_d [d, F]: each row has one scale (1 or 2^-20, alternating by row)
    Wd = (_ints(rng, (d, F)) * _alternating(d)[:, None])[None]
    Wr = np.zeros((1, d))
    ge = lambda e: (Wg[e], Wu[e], Wd[e])
    ex = O.forward(x, Wr, None, ge, E=1, k=1, kind=O.SOFTMAX, mode="exact")["experts"][0]
    mx = O.forward(x, Wr, None, ge, E=1, k=1, kind=O.SOFTMAX, mode="mxfp8")["experts"][0]
    h = ex["h"]
    # the construction separates the axes: h and W_d are exact along F only
    assert np.array_equal(h, 64.0 * (c * c)[:, None] * v[None, :])
    assert _exact_along_last(h) and not _exact_along_last(h.T.copy())
    assert _exact_along_last(Wd[0]) and not _exact_along_last(Wd[0].T.copy())
    # MXFP8 mode: h' = h, and y = BF16 of the exact product
    assert np.array_equal(mx["h_op"], h)
    assert np.array_equal(mx["y"], O.bf16_round(ex["y"]))


# ---------------------------------------------------------------------------
# Backward, dgrad: dy and W_d^T along d (DGRAD2's K); da, db, W_g^T and
# W_u^T along F (DGRAD1's K)
# ---------------------------------------------------------------------------

def _dgrad_operands(seed):
    rng = np.random.default_rng(seed)
    R, d, F = 64, 64, 64
    c = _alternating(R)                      # per-row scale of dy (and so of da, db)
    dy = np.zeros((R, d))
    dy[:, 0] = c * 2.0 ** rng.integers(0, 3, R)   # powers of two: da, db keep <= 4 bits
    sig = _alternating(F)                    # per-column scale of W_d: W_d^T rows
    Wd = _ints(rng, (d, F)) * sig[None, :]   # (along d) exact, W_d rows (along F) not
    # a = 64 / sigma_f >= 64: sigmoid(a) = 1 and silu(a) = a exactly in fp64, so
    # da = dh * b and db = dh * a; with b = 1 / sigma_f both are row-scaled integers
    a_s = np.broadcast_to(64.0 / sig, (R, F)).copy()
    b_s = np.broadcast_to(1.0 / sig, (R, F)).copy()
    tau = _alternating(d)                    # per-column scale of W_g, W_u
    Wg = _ints(rng, (F, d)) * tau[None, :]
    Wu = _ints(rng, (F, d)) * tau[None, :]
    return dy, a_s, b_s, Wg, Wu, Wd


def test_mxfp8_dgrad_blocks_each_gemm_along_its_K():
    dy, a_s, b_s, Wg, Wu, Wd = _dgrad_operands(102)
    bf = O.expert_dgrad(dy, a_s, b_s, Wg, Wu, Wd, "bf16")
    mx = O.expert_dgrad(dy, a_s, b_s, Wg, Wu, Wd, "mxfp8")
    # the construction separates the axes
    assert _exact_along_last(dy) and not _exact_along_last(dy.T.copy())
    assert _exact_along_last(Wd.T.copy()) and not _exact_along_last(Wd)
    assert _exact_along_last(bf["da"]) and not _exact_along_last(bf["da"].T.copy())
    assert _exact_along_last(bf["db"]) and not _exact_along_last(bf["db"].T.copy())
    assert _exact_along_last(Wg.T.copy()) and not _exact_along_last(Wg)
    assert _exact_along_last(Wu.T.copy()) and not _exact_along_last(Wu)
    assert np.any(bf["da"] != 0) and np.any(bf["db"] != 0)
    for key in ("dh", "da", "db", "dx"):
        assert np.array_equal(mx[key], bf[key]), key


def test_mxfp8_dgrad_reusing_forward_weight_blocking_would_differ():
    """The same operands with W_d and W_g quantised along their forward K (the
    wrong axis for dgrad) lose bits: the pin above can tell the two apart."""
    dy, a_s, b_s, Wg, Wu, Wd = _dgrad_operands(102)
    bf = O.expert_dgrad(dy, a_s, b_s, Wg, Wu, Wd, "bf16")
    wrong = O.expert_dgrad(dy, a_s, b_s, O.mx_qdq(Wg), O.mx_qdq(Wu), O.mx_qdq(Wd), "bf16")
    assert not np.array_equal(wrong["dh"], bf["dh"])
    assert not np.array_equal(wrong["dx"], bf["dx"])


# ---------------------------------------------------------------------------
# Backward, wgrad: every operand along the expert's token rows, blocks of 32
# from the expert's first row, the last block zero-padded
# ---------------------------------------------------------------------------

def _wgrad_operand(rng, R, X):
    # column scales 2^20 apart (so blocking along the columns fails) and row
    # scales 1 for rows 0..31, 2^-20 for rows 32.. (so a block that mixes the
    # two -- 64 rows, or 32 rows from another start -- fails)
    row = np.where(np.arange(R) < 32, 1.0, 1.0 / BIG)
    return _ints(rng, (R, X)) * row[:, None] * _alternating(X)[None, :]


def test_mxfp8_wgrad_blocks_along_rows_zero_padded():
    rng = np.random.default_rng(103)
    R, d, F = 45, 64, 96          # 45 rows: the second block holds 13 rows + 19 pad
    dy, h, da, db, xe = (_wgrad_operand(rng, R, n) for n in (d, F, F, F, d))
    for op in (dy, h, da, db, xe):
        assert np.array_equal(O.mx_qdq_rows_padded(op), op)
        assert not _exact_along_last(op[:32].copy())              # along columns
        padded_ones = np.vstack([op, np.ones((64 - R, op.shape[1]))])
        assert not np.array_equal(O.mx_qdq(padded_ones.T.copy()).T[:R], op)  # pad != 0
        block64 = np.vstack([op, np.zeros((64 - R, op.shape[1]))])
        assert not np.array_equal(_qdq_rows_block(block64, 64)[:R], op)       # 64-row blocks
    bf = O.expert_wgrad(dy, h, da, db, xe, "bf16")
    mx = O.expert_wgrad(dy, h, da, db, xe, "mxfp8")
    for key in ("dWd", "dWg", "dWu"):
        assert np.array_equal(mx[key], bf[key]), key
        assert np.any(bf[key] != 0)


def _qdq_rows_block(a, block):
    """Quantise along rows with one scale per `block` rows (block a multiple
    of 32: the same amax over a longer run), to show the pin rejects it."""
    out = np.empty_like(a)
    for r0 in range(0, a.shape[0], block):
        chunk = a[r0:r0 + block]
        amax = np.abs(chunk).max(axis=0)
        for c in range(a.shape[1]):
            x = O.mx_scale_exponent(float(amax[c]))
            out[r0:r0 + block, c] = [O.e4m3_decode(O.e4m3_encode(v * 2.0 ** -x)) * 2.0 ** x
                                     for v in chunk[:, c]]
    return out


# ---------------------------------------------------------------------------
# Contract rounding of reverse-combine and reverse-dispatch (hand-worked)
# ---------------------------------------------------------------------------

def _golden(kind):
    out = []
    with open(GOLDEN) as f:
        for line in f:
            line = line.strip()
            if not line or line.startswith("#"):
                continue
            parts = [p.strip() for p in line.split("|")]
            if parts[0] == kind:
                out.append(parts[1:])
    assert out
    return out


@pytest.mark.parametrize("case", _golden("rev_combine"))
def test_rev_combine_contract_rounds_the_fp32_product(case):
    g, dY, want_contract, want_exact = (float(v) for v in case)
    assert O.fp32(g) == g
    dy, dg = O.rev_combine(np.array([[dY]]), np.array([[g]]), np.zeros((1, 1, 1)))
    assert dy[0, 0, 0] == want_contract
    # the same product rounded once from fp64 gives the other value
    assert O.bf16_round(np.array([g * dY]))[0] == want_exact != want_contract


@pytest.mark.parametrize("case", _golden("rev_dispatch"), ids=["sum_order", "fused_router_term"])
def test_rev_dispatch_contract_fp32_order_and_fma(case):
    rows = np.array([float(v) for v in case[0].split()])
    k = len(rows)
    dx_rows = rows[:, None]                     # d = 1, slot j of the token at row j
    slot_pos = np.arange(k, dtype=np.int32)[None, :]
    if case[1] == "-":
        got = O.rev_dispatch(dx_rows, slot_pos)
        got_exact = O.rev_dispatch(dx_rows, slot_pos, exact=True)
    else:
        dl = np.array([[float(case[1])]])
        Wr = np.array([[float(case[2])]])
        ids = np.zeros((1, k), dtype=np.int32)
        assert O.fp32(dl[0, 0]) == dl[0, 0] and O.fp32(Wr[0, 0]) == Wr[0, 0]
        got = O.rev_dispatch(dx_rows, slot_pos, ids, dl, Wr)
        got_exact = O.rev_dispatch(dx_rows, slot_pos, ids, dl, Wr, exact=True)
    want_contract, want_exact = float(case[-2]), float(case[-1])
    assert got[0, 0] == want_contract
    assert O.bf16_round(got_exact)[0, 0] == want_exact


def test_rev_dispatch_router_term_equals_dense_router_product():
    """sum_j dl_j W_r[ids_j] (the chosen logits only) equals dlogits W_r over
    every expert (the router backward's dense product), in fp64."""
    rng = np.random.default_rng(104)
    T, d, E, k = 12, 16, 6, 3
    x = rng.standard_normal((T, d))
    Wr = rng.standard_normal((E, d))
    r = O.router(x, Wr, None, k, O.SIGMOID)
    dg = rng.standard_normal((T, k))
    rb = O.router_bwd(x, Wr, r["scores"], r["ids"], r["gates"], dg, O.SIGMOID)
    dl_sel = O.chosen_logit_grads(rb["dlogits"], r["ids"])
    zeros = np.zeros((T * k, d))
    slot_pos = np.arange(T * k, dtype=np.int32).reshape(T, k)
    got = O.rev_dispatch(zeros, slot_pos, r["ids"], dl_sel, Wr, exact=True)
    assert np.allclose(got, rb["dxr"], rtol=1e-13, atol=1e-13)
    # and the logits off the chosen set carry nothing
    mask = np.zeros((T, E), dtype=bool)
    np.put_along_axis(mask, r["ids"].astype(np.int64), True, 1)
    assert np.all(rb["dlogits"][~mask] == 0)
