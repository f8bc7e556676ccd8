"""Plain CPU oracle for one Mixture-of-Experts layer, forward and backward.

TEST INFRASTRUCTURE ONLY: the tests, the smoke check and the benchmark's
CPU-baseline leg import this module; the product path never does.  It shares
no code with the CUDA library.  Scalar rounding (BF16, E4M3/E8M0, the fp32
fused multiply-add order of the combine) lives in ``mok_oracle.c``; dense
products are numpy fp64 matrix products (a library primitive used as a
step, with no blocking or reordering of our own).

Pages followed (the pages give prose only, no formulas):
  [kucoin] "Cursor's MoK achieves 2.37x performance boost on NVIDIA GB300
           NVL72" (kucoin.com flash, Arabic): §01 the communication tax
           (router, dispatch, layout, combine), §02 push vs pull, the
           megakernel, MXFP8 fused into dispatch / grouped GEMM / SwiGLU,
           §03 the measured layer (routing, expert FFN, combine, final
           weighted combine).

Modes: ``"bf16"`` and ``"mxfp8"`` mirror the contract rounding points of
the GPU path; ``"exact"`` turns every rounding point off (pure fp64), which
is what the textbook pins (dense reformulation, finite differences) compare.

Every function here is pinned by ``tests/test_oracle_*.py`` against values
the format definitions, the mathematics or brute force fix.
"""
from __future__ import annotations

import ctypes
import os
import subprocess
import threading

import numpy as np

_HERE = os.path.dirname(os.path.abspath(__file__))
_SRC = os.path.join(_HERE, "mok_oracle.c")
_LIB = os.path.join(_HERE, "libmok_oracle.so")
_lock = threading.Lock()
_lib = None

SOFTMAX, SIGMOID = 0, 1

_d = ctypes.POINTER(ctypes.c_double)
_i32 = ctypes.POINTER(ctypes.c_int32)
_u8 = ctypes.POINTER(ctypes.c_uint8)
_u16 = ctypes.POINTER(ctypes.c_uint16)
_i64 = ctypes.c_int64
_int = ctypes.c_int


def build(force: bool = False) -> str:
    """Compile ``mok_oracle.c`` with gcc into ``libmok_oracle.so``."""
    if (not force and os.path.exists(_LIB)
            and os.path.getmtime(_LIB) >= os.path.getmtime(_SRC)):
        return _LIB
    tmp = _LIB + f".tmp{os.getpid()}"
    cmd = ["gcc", "-O2", "-std=c11", "-ffp-contract=off", "-fopenmp", "-shared",
           "-fPIC", "-o", tmp, _SRC, "-lm"]
    subprocess.run(cmd, check=True)
    os.replace(tmp, _LIB)
    return _LIB


def lib():
    global _lib
    with _lock:
        if _lib is None:
            L = ctypes.CDLL(build())
            sig = {
                "mko_bf16_round": (ctypes.c_double, [ctypes.c_double]),
                "mko_bf16_round_array": (None, [_d, _d, _i64]),
                "mko_bf16_bits_array": (None, [_d, _u16, _i64]),
                "mko_bf16_values_array": (None, [_u16, _d, _i64]),
                "mko_e4m3_decode": (ctypes.c_double, [ctypes.c_uint8]),
                "mko_e4m3_encode": (ctypes.c_uint8, [ctypes.c_double]),
                "mko_mx_scale_exponent": (_int, [ctypes.c_double]),
                "mko_mx_quantize": (None, [_d, _i64, _i64, _u8, _u8]),
                "mko_mx_dequantize": (None, [_u8, _u8, _i64, _i64, _d]),
                "mko_router": (None, [_int, _int, _int, _int, _int, _d, _d, _d,
                                      _d, _d, _i32, _d]),
                "mko_layout": (None, [_int, _int, _int, _i32, _i32, _i32, _i32,
                                      _i32, _u8]),
                "mko_swiglu": (None, [_i64, _d, _d, _d]),
                "mko_combine": (None, [_int, _int, _int, _int, _d, _d, _d]),
                "mko_rev_combine": (None, [_int, _int, _int, _int, _d, _d, _d,
                                           _d, _d]),
                "mko_swiglu_bwd": (None, [_i64, _d, _d, _d, _d, _d]),
                "mko_router_bwd": (None, [_int, _int, _int, _int, _int, _d, _d,
                                          _d, _i32, _d, _d, _d, _d, _d]),
                "mko_rev_dispatch": (None, [_int, _int, _int, _int, _d, _i32,
                                            _i32, _d, _d, _d]),
            }
            for name, (res, args) in sig.items():
                f = getattr(L, name)
                f.restype = res
                f.argtypes = args
            _lib = L
    return _lib


def _p(a, ty):
    return a.ctypes.data_as(ty)


def _f64(a):
    return np.ascontiguousarray(a, dtype=np.float64)


# ---------------------------------------------------------------------------
# Rounding points
# ---------------------------------------------------------------------------

def bf16_round(a):
    """Round fp64 values to the nearest BF16 value (ties to even)."""
    a = _f64(a)
    out = np.empty_like(a)
    lib().mko_bf16_round_array(_p(a, _d), _p(out, _d), a.size)
    return out


def bf16_bits(a):
    a = _f64(a)
    out = np.empty(a.shape, dtype=np.uint16)
    lib().mko_bf16_bits_array(_p(a, _d), _p(out, _u16), a.size)
    return out


def bf16_values(bits):
    bits = np.ascontiguousarray(bits, dtype=np.uint16)
    out = np.empty(bits.shape, dtype=np.float64)
    lib().mko_bf16_values_array(_p(bits, _u16), _p(out, _d), bits.size)
    return out


def fp32(a):
    """Round fp64 values to the nearest fp32 (IEEE conversion)."""
    return _f64(a).astype(np.float32).astype(np.float64)


def e4m3_encode(v: float) -> int:
    return int(lib().mko_e4m3_encode(float(v)))


def e4m3_decode(c: int) -> float:
    return float(lib().mko_e4m3_decode(int(c)))


def mx_scale_exponent(amax: float) -> int:
    return int(lib().mko_mx_scale_exponent(float(amax)))


def mx_quantize(a):
    """MXFP8 quantise a 2-D array in blocks of 32 along its last axis.

    Returns (codes uint8 [rows, cols], scales uint8 [rows, cols/32])."""
    a = _f64(a)
    rows, cols = a.shape
    assert cols % 32 == 0
    codes = np.empty((rows, cols), dtype=np.uint8)
    scales = np.empty((rows, cols // 32), dtype=np.uint8)
    lib().mko_mx_quantize(_p(a, _d), rows, cols, _p(codes, _u8), _p(scales, _u8))
    return codes, scales


def mx_dequantize(codes, scales):
    codes = np.ascontiguousarray(codes, dtype=np.uint8)
    scales = np.ascontiguousarray(scales, dtype=np.uint8)
    rows, cols = codes.shape
    out = np.empty((rows, cols), dtype=np.float64)
    lib().mko_mx_dequantize(_p(codes, _u8), _p(scales, _u8), rows, cols, _p(out, _d))
    return out


def mx_qdq(a):
    """Quantise along the last axis and return the values the tensor core sees."""
    return mx_dequantize(*mx_quantize(a))


def mx_qdq_rows_padded(a):
    """Quantise a [rows, cols] operand along its ROWS (the K of a weight-gradient
    GEMM), zero-padding rows to a multiple of 32; returns [rows, cols] values."""
    a = _f64(a)
    rows, cols = a.shape
    pad = (-rows) % 32
    at = np.zeros((cols, rows + pad))
    at[:, :rows] = a.T
    return mx_qdq(at)[:, :rows].T.copy()


# ---------------------------------------------------------------------------
# A1 router, A2 layout
# ---------------------------------------------------------------------------

def router(x, Wr, bias, k, kind):
    """[kucoin] §01 router: logits, scores, top-k ids (ties to lower id), gates."""
    x = _f64(x)
    Wr = _f64(Wr)
    T, d = x.shape
    E = Wr.shape[0]
    b = None if bias is None else _f64(bias)
    logits = np.empty((T, E))
    scores = np.empty((T, E))
    ids = np.empty((T, k), dtype=np.int32)
    gates = np.empty((T, k))
    lib().mko_router(T, d, E, k, kind, _p(x, _d), _p(Wr, _d),
                     None if b is None else _p(b, _d),
                     _p(logits, _d), _p(scores, _d), _p(ids, _i32), _p(gates, _d))
    return dict(logits=logits, scores=scores, ids=ids, gates=gates)


def layout(ids, E):
    """[kucoin] §01 layout: stable counting sort of slots t*k+j by expert."""
    ids = np.ascontiguousarray(ids, dtype=np.int32)
    T, k = ids.shape
    S = T * k
    counts = np.empty(E, dtype=np.int32)
    offsets = np.empty(E + 1, dtype=np.int32)
    slot_pos = np.empty((T, k), dtype=np.int32)
    row_tok = np.empty(S, dtype=np.int32)
    row_j = np.empty(S, dtype=np.uint8)
    lib().mko_layout(T, k, E, _p(ids, _i32), _p(counts, _i32), _p(offsets, _i32),
                     _p(slot_pos, _i32), _p(row_tok, _i32), _p(row_j, _u8))
    return dict(counts=counts, offsets=offsets, slot_pos=slot_pos,
                row_tok=row_tok, row_j=row_j)


# ---------------------------------------------------------------------------
# A3 dispatch, A4/A5 expert FFN, A6 combine
# ---------------------------------------------------------------------------

def dispatch(x, row_tok, mode):
    """[kucoin] §02 pull dispatch: row p of the expert-ordered buffer is token
    row_tok[p]; in MXFP8 mode the rows are quantised along d on the way."""
    xe = _f64(x)[np.asarray(row_tok)]
    if mode == "mxfp8":
        codes, scales = mx_quantize(xe)
        return dict(xe=xe, codes=codes, scales=scales, op=mx_dequantize(codes, scales))
    return dict(xe=xe, op=xe)


def swiglu(a, b):
    a = _f64(a)
    b = _f64(b)
    h = np.empty_like(a)
    lib().mko_swiglu(a.size, _p(a, _d), _p(b, _d), _p(h, _d))
    return h


def weight_operands(Wg, Wu, Wd, mode):
    """Operand values of one expert's weights as the tensor cores see them:
    BF16 values as given, or MXFP8 along each forward GEMM's K
    (W_g, W_u [F,d] along d; W_d [d,F] along F)."""
    if mode == "mxfp8":
        return mx_qdq(Wg), mx_qdq(Wu), mx_qdq(Wd)
    return _f64(Wg), _f64(Wu), _f64(Wd)


def expert_ffn(xe_op, Wg_op, Wu_op, Wd_op, mode):
    """One expert's SwiGLU FFN over its rows ([kucoin] §01/§02 grouped GEMM).

    a = xe W_g^T, b = xe W_u^T, h = silu(a) b, y = h' W_d^T where h' is h
    rounded to BF16 (bf16 mode), MXFP8-quantised along F (mxfp8 mode) or left
    alone (exact); y is stored as BF16 unless exact."""
    a = _f64(xe_op) @ _f64(Wg_op).T
    b = _f64(xe_op) @ _f64(Wu_op).T
    h = swiglu(a, b)
    if mode == "bf16":
        h_op = bf16_round(h)
    elif mode == "mxfp8":
        h_op = mx_qdq(h)
    else:
        h_op = h
    y = h_op @ _f64(Wd_op).T
    if mode != "exact":
        y = bf16_round(y)
    return dict(a=a, b=b, h=h, h_op=h_op, y=y)


def combine(ystage, gates, exact=False):
    """A6 final weighted combine: out[t] = sum_j g_tj y_tj.

    Contract mode folds fp32 fmaf over j = 0..k-1 from 0 and rounds to BF16;
    gates are taken as fp32 values."""
    ystage = _f64(ystage)
    T, k, d = ystage.shape
    g = _f64(gates) if exact else fp32(gates)
    out = np.empty((T, d))
    lib().mko_combine(T, k, d, int(bool(exact)), _p(ystage, _d), _p(g, _d), _p(out, _d))
    return out


def forward(x, Wr, bias, get_expert, *, E, k, kind, mode, tokens=None,
            ids=None, gates=None):
    """The whole layer for a set of tokens (all by default).

    x [T,d] values; get_expert(e) -> (W_g [F,d], W_u [F,d], W_d [d,F]) values.
    Per-token results do not depend on the other tokens once routing is
    fixed, so a token subset gives the same rows as the full run.  ``ids`` /
    ``gates`` (for the chosen tokens) override the router, for unit parity
    with routing injected at the step boundary."""
    x = _f64(x)
    tok = np.arange(x.shape[0]) if tokens is None else np.asarray(tokens)
    xs = x[tok]
    r = router(xs, Wr, bias, k, kind)
    if ids is not None:
        r["ids"] = np.ascontiguousarray(ids, dtype=np.int32)
    if gates is not None:
        r["gates"] = _f64(gates)
    lay = layout(r["ids"], E)
    dsp = dispatch(xs, lay["row_tok"], mode)
    S, d = dsp["xe"].shape
    y_rows = np.zeros((S, d))
    saved = {}
    off = lay["offsets"]
    for e in range(E):
        lo, hi = int(off[e]), int(off[e + 1])
        if hi == lo:
            continue
        Wg, Wu, Wd = weight_operands(*get_expert(e), mode)
        f = expert_ffn(dsp["op"][lo:hi], Wg, Wu, Wd, mode)
        y_rows[lo:hi] = f["y"]
        saved[e] = f
    T = xs.shape[0]
    ystage = y_rows[lay["slot_pos"].reshape(-1)].reshape(T, k, d)
    out = combine(ystage, r["gates"], exact=(mode == "exact"))
    return dict(out=out, ystage=ystage, router=r, layout=lay, dispatch=dsp,
                experts=saved, tokens=tok)


# ---------------------------------------------------------------------------
# Error scales of the reductions
# ---------------------------------------------------------------------------
# A sum of K terms whose factors each carry an independent relative rounding
# error of size u (BF16 storage, an MXFP8 code) is off by about u times the
# root-sum-square of its terms -- whatever the sum itself is, since the terms
# can cancel to near zero.  These give that scale for every reduction of the
# backward, propagated through the linear maps that follow it, so a
# comparison can measure an element's error against it.

def terms_rss(A, B):
    """sqrt(sum_r (A[r, i] B[r, j])^2) for every element (i, j) of A^T B."""
    A, B = _f64(A), _f64(B)
    return np.sqrt((A * A).T @ (B * B))


def gate_grad_rss(dY, ystage):
    """Terms' root-sum-square of dgates[t, j] = <dY[t], y_tj>: [T, k]."""
    dY, ystage = _f64(dY), _f64(ystage)
    return np.sqrt(np.einsum("tc,tjc->tj", dY * dY, ystage * ystage))


def router_bwd_rss(scores, ids, gates, dg_rss, kind):
    """Error scale of dlogits [T, E] from the dgates scale: the router backward
    is linear in dgates, dl_j = sum_j' J_jj' dg_j' with
    J = diag(g) (I - 1 g^T) (softmax) or diag(s (1 - s) / sum_sel s) (I - 1 g^T)
    (sigmoid), so independent errors of scale dg_rss map to
    sqrt(sum_j' J_jj'^2 dg_rss_j'^2).  Zero off the chosen experts."""
    scores, gates, dg_rss = _f64(scores), _f64(gates), _f64(dg_rss)
    ids = np.asarray(ids, dtype=np.int64)
    T, k = ids.shape
    sel = np.take_along_axis(scores, ids, axis=1)
    M = np.eye(k)[None, :, :] - gates[:, None, :]            # I - 1 g^T, [T, k, k]
    if kind == SOFTMAX:
        row = gates
    else:
        row = sel * (1.0 - sel) / sel.sum(axis=1, keepdims=True)
    J = row[:, :, None] * M
    rss_sel = np.sqrt(np.einsum("tjl,tl->tj", J * J, dg_rss * dg_rss))
    out = np.zeros((T, scores.shape[1]))
    np.put_along_axis(out, ids, rss_sel, axis=1)
    return out


# ---------------------------------------------------------------------------
# Backward
# ---------------------------------------------------------------------------

def rev_combine(dY, gates, ystage, exact=False):
    """B1 pull reverse-combine: dy_slot = g dY[t] (BF16 of the fp32 product),
    dgates = <dY[t], y_tj>."""
    dY = _f64(dY)
    ystage = _f64(ystage)
    T, k, d = ystage.shape
    g = _f64(gates) if exact else fp32(gates)
    dy = np.empty((T, k, d))
    dg = np.empty((T, k))
    lib().mko_rev_combine(T, k, d, int(bool(exact)), _p(dY, _d), _p(g, _d),
                          _p(ystage, _d), _p(dy, _d), _p(dg, _d))
    return dy, dg


def swiglu_bwd(dh, a, b):
    dh, a, b = _f64(dh), _f64(a), _f64(b)
    da = np.empty_like(dh)
    db = np.empty_like(dh)
    lib().mko_swiglu_bwd(dh.size, _p(dh, _d), _p(a, _d), _p(b, _d), _p(da, _d), _p(db, _d))
    return da, db


def expert_dgrad(dy, a_saved, b_saved, Wg, Wu, Wd, mode):
    """B2 + B3 for one expert's rows.

    dh = dy W_d (K = d), SwiGLU backward with the saved a, b, then
    dx = da W_g + db W_u (K = F).  In mxfp8 mode each GEMM's operands are
    quantised along that GEMM's K (dy along d, W_d^T along d; da, db along F,
    W_g^T / W_u^T along F); da and db are first stored as BF16."""
    dy = _f64(dy)
    if mode == "mxfp8":
        dh = mx_qdq(dy) @ mx_qdq(_f64(Wd).T).T
    else:
        dh = dy @ _f64(Wd)
    da, db = swiglu_bwd(dh, a_saved, b_saved)
    if mode != "exact":
        da, db = bf16_round(da), bf16_round(db)
    if mode == "mxfp8":
        dx = mx_qdq(da) @ mx_qdq(_f64(Wg).T).T + mx_qdq(db) @ mx_qdq(_f64(Wu).T).T
    else:
        dx = da @ _f64(Wg) + db @ _f64(Wu)
    if mode != "exact":
        dx = bf16_round(dx)
    return dict(dh=dh, da=da, db=db, dx=dx)


def expert_wgrad(dy, h_saved, da, db, xe, mode, rss=False):
    """B4 for one expert: dW_d = dy^T h, dW_g = da^T xe, dW_u = db^T xe,
    K = the expert's rows.  mxfp8: every operand quantised along the rows
    (zero-padded to a multiple of 32).  Stored as BF16 unless exact.
    rss: also the root-sum-square of each element's terms (terms_rss)."""
    ops = [_f64(v) for v in (dy, h_saved, da, db, xe)]
    if mode == "mxfp8":
        ops = [mx_qdq_rows_padded(v) for v in ops]
    dy_, h_, da_, db_, xe_ = ops
    dWd = dy_.T @ h_
    dWg = da_.T @ xe_
    dWu = db_.T @ xe_
    if mode != "exact":
        dWd, dWg, dWu = bf16_round(dWd), bf16_round(dWg), bf16_round(dWu)
    out = dict(dWd=dWd, dWg=dWg, dWu=dWu)
    if rss:
        out.update(dWd_rss=terms_rss(dy_, h_), dWg_rss=terms_rss(da_, xe_),
                   dWu_rss=terms_rss(db_, xe_))
    return out


def router_bwd(x, Wr, scores, ids, gates, dgates, kind):
    """B6: gradients through the renormalised top-k gates to the logits,
    dW_r = dlogits^T x and the router's share of dX, dlogits W_r."""
    x, Wr, scores, gates, dgates = map(_f64, (x, Wr, scores, gates, dgates))
    ids = np.ascontiguousarray(ids, dtype=np.int32)
    T, d = x.shape
    E = Wr.shape[0]
    k = ids.shape[1]
    dl = np.empty((T, E))
    dWr = np.empty((E, d))
    dxr = np.empty((T, d))
    lib().mko_router_bwd(T, d, E, k, kind, _p(x, _d), _p(Wr, _d), _p(scores, _d),
                         _p(ids, _i32), _p(gates, _d), _p(dgates, _d),
                         _p(dl, _d), _p(dWr, _d), _p(dxr, _d))
    return dict(dlogits=dl, dWr=dWr, dxr=dxr)


def rev_dispatch(dx_rows, slot_pos, ids=None, dl_sel=None, Wr=None, exact=False):
    """B5 push reverse-dispatch with the router's share of dX:
    dX[t] = sum_j dx_rows[slot_pos[t,j]] + sum_j dl_sel[t,j] W_r[ids[t,j]].

    Contract mode: one fp32 accumulator from 0, the slot rows added in
    ascending j, then the router terms folded in ascending j with fmaf, then
    BF16; dl_sel and W_r are taken as fp32 values, dx rows as BF16 values.
    ``dl_sel=None`` leaves the router term out."""
    dx_rows = _f64(dx_rows)
    slot_pos = np.ascontiguousarray(slot_pos, dtype=np.int32)
    T, k = slot_pos.shape
    d = dx_rows.shape[1]
    if dl_sel is None:
        ids_, dl_, wr_ = None, None, None
    else:
        ids_ = np.ascontiguousarray(ids, dtype=np.int32)
        dl_ = _f64(dl_sel) if exact else fp32(dl_sel)
        wr_ = _f64(Wr) if exact else fp32(Wr)
    dX = np.empty((T, d))
    lib().mko_rev_dispatch(T, k, d, int(bool(exact)), _p(dx_rows, _d), _p(slot_pos, _i32),
                           None if ids_ is None else _p(ids_, _i32),
                           None if dl_ is None else _p(dl_, _d),
                           None if wr_ is None else _p(wr_, _d), _p(dX, _d))
    return dX


def chosen_logit_grads(dlogits, ids):
    """The logit gradients of the chosen experts, [T, k] in slot order (the
    other logits get none)."""
    return np.take_along_axis(_f64(dlogits), np.asarray(ids, dtype=np.int64), axis=1)


def backward(fwd, dY, x, Wr, get_expert, *, E, k, kind, mode, rss=False):
    """Full backward of ``forward`` (all tokens of that call).

    Quantisers are straight-through (treated as identity); routing is
    piecewise constant so only the chosen logits get gradient.  rss: also
    the error scales of the reductions (dgates_rss, dlogits_rss, dWr_rss,
    and dW*_rss per expert; see terms_rss)."""
    r, lay = fwd["router"], fwd["layout"]
    exact = mode == "exact"
    dY = _f64(dY)
    T = dY.shape[0]
    dy_slot, dgates = rev_combine(dY, r["gates"], fwd["ystage"], exact=exact)
    S = T * k
    d = dY.shape[1]
    dy_rows = np.empty((S, d))
    dy_rows[lay["slot_pos"].reshape(-1)] = dy_slot.reshape(S, d)
    dx_rows = np.zeros((S, d))
    off = lay["offsets"]
    grads = {}
    # d_ff from an expert that has rows, else from the weights themselves (a
    # call in which no expert has a row still owes every expert a zero dW)
    F = (next(iter(fwd["experts"].values()))["a"].shape[1] if fwd["experts"]
         else get_expert(0)[0].shape[0])
    for e in range(E):
        lo, hi = int(off[e]), int(off[e + 1])
        if hi == lo:
            grads[e] = dict(dWd=np.zeros((d, F)), dWg=np.zeros((F, d)), dWu=np.zeros((F, d)))
            if rss:
                grads[e].update(dWd_rss=np.zeros((d, F)), dWg_rss=np.zeros((F, d)),
                                dWu_rss=np.zeros((F, d)))
            continue
        Wg, Wu, Wd = get_expert(e)
        f = fwd["experts"][e]
        a_s, b_s = (f["a"], f["b"]) if exact else (bf16_round(f["a"]), bf16_round(f["b"]))
        h_s = f["h"] if exact else bf16_round(f["h"])
        g = expert_dgrad(dy_rows[lo:hi], a_s, b_s, Wg, Wu, Wd, mode)
        dx_rows[lo:hi] = g["dx"]
        xe_rows = fwd["dispatch"]["xe"][lo:hi]
        grads[e] = expert_wgrad(dy_rows[lo:hi], h_s, g["da"], g["db"], xe_rows, mode, rss=rss)
    xs = _f64(x)[fwd["tokens"]]
    rb = router_bwd(xs, Wr, r["scores"], r["ids"], r["gates"], dgates, kind)
    dl_sel = chosen_logit_grads(rb["dlogits"], r["ids"])
    dX = rev_dispatch(dx_rows, lay["slot_pos"], r["ids"], dl_sel, Wr, exact=exact)
    out = dict(dX=dX, dgates=dgates, dlogits=rb["dlogits"], dWr=rb["dWr"],
               dxr=rb["dxr"], dy_rows=dy_rows, dx_rows=dx_rows, experts=grads)
    if rss:
        dg_rss = gate_grad_rss(dY, fwd["ystage"])
        dl_rss = router_bwd_rss(r["scores"], r["ids"], r["gates"], dg_rss, kind)
        out.update(dgates_rss=dg_rss, dlogits_rss=dl_rss, dWr_rss=terms_rss(dl_rss, xs))
    return out
