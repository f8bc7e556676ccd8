"""ctypes binding of libmok.so (include/mok.h).

Argument marshalling only: every step of the layer runs in the library's CUDA
kernels.  Tensors are torch tensors used as device memory; the functions
below take them, check dtype/shape/device, and pass raw pointers and the
current CUDA stream.  There is no fallback: if the library cannot be loaded
the import of the functions raises.
"""
from __future__ import annotations

import ctypes
import os

import torch

from . import build as _build

_HERE = os.path.dirname(os.path.abspath(__file__))

MOK_OK, MOK_ERR_INVALID_ARG, MOK_ERR_UNSUPPORTED, MOK_ERR_CUDA, MOK_ERR_TIMEOUT = range(5)
MOK_ROUTER_SOFTMAX, MOK_ROUTER_SIGMOID = 0, 1
MOK_BF16, MOK_MXFP8 = 0, 1
MOK_PAIRS_AUTO, MOK_PAIRS_ON, MOK_PAIRS_OFF = 0, 1, 2
MOK_ROW_ALIGN = 128
MOK_MAX_SOURCES = 64

EXPORTS = [
    "mok_max_padded_rows", "mok_workspace_size", "mok_saved_ctx_layout", "mok_route_layout",
    "mok_dispatch", "mok_expert_ffn", "mok_combine", "mok_moe_fused", "mok_moe_forward",
    "mok_moe_backward",
    "mok_quantize_mx", "mok_transpose_bf16", "mok_reset_device_status", "mok_get_device_status",
    "mok_status_string", "mok_layout_static", "mok_fused_plan", "mok_dispatch_by_token",
    "mok_bwd_ws_layout", "mok_swiglu_quantize_mx", "mok_moe_forward_chain",
]


class MokConfig(ctypes.Structure):
    _fields_ = [
        ("T", ctypes.c_int), ("d_model", ctypes.c_int), ("n_experts", ctypes.c_int),
        ("top_k", ctypes.c_int), ("d_ff", ctypes.c_int), ("router", ctypes.c_int),
        ("dtype", ctypes.c_int), ("n_sources", ctypes.c_int),
        ("source_rows", ctypes.POINTER(ctypes.c_int)), ("minibatch_rows", ctypes.c_int),
        ("gather_sm_fraction", ctypes.c_float), ("ring_bytes", ctypes.c_size_t),
        ("wait_limit_ns", ctypes.c_ulonglong), ("fused_cta_pairs", ctypes.c_int),
        ("gemm_cta_pairs", ctypes.c_int),
    ]


class MokWeights(ctypes.Structure):
    _fields_ = [(n, ctypes.c_void_p) for n in (
        "w_gate", "w_up", "w_down", "q_gate", "q_up", "q_down", "s_gate", "s_up", "s_down",
        "qt_gate", "qt_up", "qt_down", "st_gate", "st_up", "st_down", "wt_gate", "wt_up",
        "wt_down")]


class MokWeightGrads(ctypes.Structure):
    _fields_ = [(n, ctypes.c_void_p) for n in ("d_gate", "d_up", "d_down")]


class MokBwdLayout(ctypes.Structure):
    _fields_ = [(n, ctypes.c_size_t) for n in ("status", "dy", "da", "db", "dx", "dl_sel", "total")]


class MokCtxLayout(ctypes.Structure):
    _fields_ = [(n, ctypes.c_size_t) for n in (
        "ids", "gates", "sel_scores", "counts", "offsets", "pad_offsets", "slot_pos", "row_tok",
        "row_j", "logits", "a", "b", "h", "ystage", "total")]


_lib = None


def lib(build_if_missing: bool = True) -> ctypes.CDLL:
    """Load libmok.so (building it in-tree first if it is missing or stale)."""
    global _lib
    if _lib is None:
        path = _build.LIB
        if build_if_missing and not _build.up_to_date():
            _build.build()
        if not os.path.exists(path):
            raise RuntimeError(f"libmok.so not built ({path}); run __graft_entry__.build()")
        L = ctypes.CDLL(path)
        vp, i64, sz = ctypes.c_void_p, ctypes.c_int64, ctypes.c_size_t
        cfgp = ctypes.POINTER(MokConfig)
        L.mok_max_padded_rows.argtypes = [cfgp]
        L.mok_max_padded_rows.restype = i64
        L.mok_workspace_size.argtypes = [cfgp, ctypes.POINTER(sz), ctypes.POINTER(sz), ctypes.POINTER(sz)]
        L.mok_saved_ctx_layout.argtypes = [cfgp, ctypes.POINTER(MokCtxLayout)]
        L.mok_route_layout.argtypes = [cfgp, vp] + [vp] * 13
        L.mok_dispatch.argtypes = [cfgp, vp] + [vp] * 8
        L.mok_dispatch_by_token.argtypes = [cfgp, vp] + [vp] * 7
        L.mok_expert_ffn.argtypes = [cfgp, vp, vp, ctypes.POINTER(MokWeights)] + [vp] * 10
        L.mok_combine.argtypes = [cfgp, vp, vp, vp, vp]
        L.mok_moe_fused.argtypes = [cfgp, vp, ctypes.POINTER(MokWeights)] + [vp] * 12
        L.mok_moe_forward.argtypes = [cfgp, vp, vp, vp, ctypes.POINTER(MokWeights), vp, vp, vp, vp]
        L.mok_moe_forward_chain.argtypes = [cfgp, ctypes.c_int, vp, vp, vp, ctypes.POINTER(MokWeights), vp, vp, vp]
        L.mok_moe_backward.argtypes = [cfgp, vp, vp, vp, vp, ctypes.POINTER(MokWeights), vp,
                                       ctypes.POINTER(MokWeightGrads), vp, vp, vp, vp, vp]
        L.mok_quantize_mx.argtypes = [vp, i64, i64, i64, ctypes.c_int, vp, vp, vp]
        L.mok_transpose_bf16.argtypes = [vp, i64, i64, i64, vp, vp]
        L.mok_layout_static.argtypes = [cfgp] + [vp] * 8
        L.mok_bwd_ws_layout.argtypes = [cfgp, ctypes.POINTER(MokBwdLayout)]
        L.mok_swiglu_quantize_mx.argtypes = [vp, vp, i64, i64, vp, vp, vp, vp]
        L.mok_fused_plan.argtypes = [cfgp] + [ctypes.POINTER(ctypes.c_int)] * 4 + [ctypes.POINTER(i64)]
        L.mok_reset_device_status.argtypes = [vp, vp]
        L.mok_get_device_status.argtypes = [vp, vp]
        L.mok_status_string.argtypes = [ctypes.c_int]
        L.mok_status_string.restype = ctypes.c_char_p
        _lib = L
    return _lib


class MokError(RuntimeError):
    def __init__(self, fn: str, code: int):
        super().__init__(f"{fn} returned {lib().mok_status_string(code).decode()} ({code})")
        self.code = code


def _check(fn: str, code: int) -> None:
    if code != MOK_OK:
        raise MokError(fn, code)


def _ptr(t) -> int | None:
    if t is None:
        return None
    assert isinstance(t, torch.Tensor) and t.is_cuda and t.is_contiguous(), "need a contiguous CUDA tensor"
    return t.data_ptr()


def _stream(stream=None):
    s = stream if stream is not None else torch.cuda.current_stream()
    return ctypes.c_void_p(s.cuda_stream)


class Config:
    """Owns a MokConfig (and the host source_rows array it points to)."""

    def __init__(self, T, d_model, n_experts, top_k, d_ff, router, dtype, n_sources=1,
                 source_rows=None, minibatch_rows=0, gather_sm_fraction=0.0, ring_bytes=0,
                 wait_limit_ns=0, fused_cta_pairs=MOK_PAIRS_AUTO, gemm_cta_pairs=MOK_PAIRS_AUTO):
        self._rows = None
        if n_sources > 1:
            rows = source_rows or [T // n_sources] * n_sources
            self._rows = (ctypes.c_int * n_sources)(*rows)
        self.c = MokConfig(T, d_model, n_experts, top_k, d_ff, router, dtype, n_sources,
                           self._rows if self._rows is not None else None, minibatch_rows,
                           gather_sm_fraction, ring_bytes, wait_limit_ns, fused_cta_pairs,
                           gemm_cta_pairs)

    @classmethod
    def from_workload(cls, w, **kw):
        opts = dict(n_sources=w.n_sources,
                    source_rows=w.source_rows if w.n_sources > 1 else None,
                    ring_bytes=w.ring_bytes)
        opts.update(kw)
        return cls(w.T, w.d, w.E, w.k, w.F,
                   MOK_ROUTER_SOFTMAX if w.router == "softmax" else MOK_ROUTER_SIGMOID,
                   MOK_MXFP8 if w.dtype == "mxfp8" else MOK_BF16, **opts)

    @property
    def ref(self):
        return ctypes.byref(self.c)


def max_padded_rows(cfg: Config) -> int:
    return int(lib().mok_max_padded_rows(cfg.ref))


def workspace_size(cfg: Config) -> tuple[int, int, int]:
    a, b, c = ctypes.c_size_t(), ctypes.c_size_t(), ctypes.c_size_t()
    _check("mok_workspace_size", lib().mok_workspace_size(cfg.ref, ctypes.byref(a), ctypes.byref(b), ctypes.byref(c)))
    return a.value, b.value, c.value


def saved_ctx_layout(cfg: Config) -> MokCtxLayout:
    out = MokCtxLayout()
    _check("mok_saved_ctx_layout", lib().mok_saved_ctx_layout(cfg.ref, ctypes.byref(out)))
    return out


def bwd_ws_layout(cfg: Config) -> MokBwdLayout:
    out = MokBwdLayout()
    _check("mok_bwd_ws_layout", lib().mok_bwd_ws_layout(cfg.ref, ctypes.byref(out)))
    return out


def _src_array(x_src):
    arr = (ctypes.c_void_p * len(x_src))(*[_ptr(x) for x in x_src])
    return arr


def route_layout(cfg, x_src, W_r, bias, ids, gates, sel_scores, logits, counts, offsets,
                 pad_offsets, slot_pos, row_tok, row_j, ws, stream=None):
    arr = _src_array(x_src)
    _check("mok_route_layout", lib().mok_route_layout(
        cfg.ref, arr, _ptr(W_r), _ptr(bias), _ptr(ids), _ptr(gates), _ptr(sel_scores), _ptr(logits),
        _ptr(counts), _ptr(offsets), _ptr(pad_offsets), _ptr(slot_pos), _ptr(row_tok), _ptr(row_j),
        _ptr(ws), _stream(stream)))


def dispatch(cfg, x_src, ids, offsets, pad_offsets, row_tok, row_j, xe, xe_scales, stream=None):
    arr = _src_array(x_src)
    _check("mok_dispatch", lib().mok_dispatch(
        cfg.ref, arr, _ptr(ids), _ptr(offsets), _ptr(pad_offsets), _ptr(row_tok), _ptr(row_j),
        _ptr(xe), _ptr(xe_scales), _stream(stream)))


def dispatch_by_token(cfg, x_src, ids, slot_pos, offsets, pad_offsets, xe, xe_scales, stream=None):
    arr = _src_array(x_src)
    _check("mok_dispatch_by_token", lib().mok_dispatch_by_token(
        cfg.ref, arr, _ptr(ids), _ptr(slot_pos), _ptr(offsets), _ptr(pad_offsets), _ptr(xe),
        _ptr(xe_scales), _stream(stream)))


def weights_struct(w: dict) -> MokWeights:
    s = MokWeights()
    for name, _ in MokWeights._fields_:
        t = w.get(name)
        setattr(s, name, _ptr(t) if t is not None else None)
    return s


def expert_ffn(cfg, xe, xe_scales, weights: MokWeights, offsets, pad_offsets, row_tok, row_j,
               ystage, saved_a, saved_b, saved_h, ws, stream=None):
    _check("mok_expert_ffn", lib().mok_expert_ffn(
        cfg.ref, _ptr(xe), _ptr(xe_scales), ctypes.byref(weights), _ptr(offsets), _ptr(pad_offsets),
        _ptr(row_tok), _ptr(row_j), _ptr(ystage), _ptr(saved_a), _ptr(saved_b), _ptr(saved_h),
        _ptr(ws), _stream(stream)))


def combine(cfg, ystage, gates, out, stream=None):
    _check("mok_combine", lib().mok_combine(cfg.ref, _ptr(ystage), _ptr(gates), _ptr(out), _stream(stream)))


def moe_fused(cfg, x_src, weights: MokWeights, ids, gates, counts, offsets, pad_offsets, slot_pos,
              row_tok, row_j, ystage, out, ws, stream=None):
    arr = _src_array(x_src)
    _check("mok_moe_fused", lib().mok_moe_fused(
        cfg.ref, arr, ctypes.byref(weights), _ptr(ids), _ptr(gates), _ptr(counts), _ptr(offsets),
        _ptr(pad_offsets), _ptr(slot_pos), _ptr(row_tok), _ptr(row_j), _ptr(ystage), _ptr(out),
        _ptr(ws), _stream(stream)))


def moe_forward(cfg, x_src, W_r, bias, weights: MokWeights, out, saved_ctx, ws, stream=None):
    arr = _src_array(x_src)
    _check("mok_moe_forward", lib().mok_moe_forward(
        cfg.ref, arr, _ptr(W_r), _ptr(bias), ctypes.byref(weights), _ptr(out), _ptr(saved_ctx),
        _ptr(ws), _stream(stream)))


def moe_forward_chain(cfg, x_srcs, W_r, bias, weights: MokWeights, outs, wss, stream=None):
    """n back-to-back inference calls; call i's combine runs inside call i+1's kernel."""
    n = len(x_srcs)
    assert len(outs) == n and len(wss) == n
    keep = [_src_array(x) for x in x_srcs]
    srcs = (ctypes.c_void_p * n)(*[ctypes.cast(a, ctypes.c_void_p).value for a in keep])
    o = (ctypes.c_void_p * n)(*[_ptr(t) for t in outs])
    ws = (ctypes.c_void_p * n)(*[_ptr(t) for t in wss])
    _check("mok_moe_forward_chain", lib().mok_moe_forward_chain(
        cfg.ref, n, srcs, _ptr(W_r), _ptr(bias), ctypes.byref(weights), o, ws, _stream(stream)))


def moe_backward(cfg, x_src, W_r, saved_ctx, dY, weights: MokWeights, dX, grads: MokWeightGrads,
                 dgates, dlogits, dW_r, ws, stream=None):
    arr = _src_array(x_src)
    _check("mok_moe_backward", lib().mok_moe_backward(
        cfg.ref, arr, _ptr(W_r), _ptr(saved_ctx), _ptr(dY), ctypes.byref(weights), _ptr(dX),
        ctypes.byref(grads), _ptr(dgates), _ptr(dlogits), _ptr(dW_r), _ptr(ws), _stream(stream)))


def quantize_mx(src, batch, rows, K, transpose, codes, scales, stream=None):
    _check("mok_quantize_mx", lib().mok_quantize_mx(
        _ptr(src), batch, rows, K, int(transpose), _ptr(codes), _ptr(scales), _stream(stream)))


def swiglu_quantize_mx(a, b, rows, F, h, codes, scales, stream=None):
    """The expert GEMM epilogue's SwiGLU + MXFP8 quantisation of h on fp32 a, b."""
    _check("mok_swiglu_quantize_mx", lib().mok_swiglu_quantize_mx(
        _ptr(a), _ptr(b), rows, F, _ptr(h), _ptr(codes), _ptr(scales), _stream(stream)))


def transpose_bf16(src, batch, rows, K, dst, stream=None):
    _check("mok_transpose_bf16", lib().mok_transpose_bf16(_ptr(src), batch, rows, K, _ptr(dst),
                                                          _stream(stream)))


def weight_grads_struct(g: dict) -> MokWeightGrads:
    s = MokWeightGrads()
    for name, _ in MokWeightGrads._fields_:
        setattr(s, name, _ptr(g[name]))
    return s


def layout_static(cfg, ids, counts, offsets, pad_offsets, slot_pos, row_tok, row_j,
                  stream=None):
    """The layout step with the library's own fixed scratch: no workspace."""
    _check("mok_layout_static", lib().mok_layout_static(
        cfg.ref, _ptr(ids), _ptr(counts), _ptr(offsets), _ptr(pad_offsets), _ptr(slot_pos),
        _ptr(row_tok), _ptr(row_j), _stream(stream)))


def fused_plan(cfg) -> dict:
    """CTAs, CTA pairs (0/1), gather CTAs, minibatch rows and ring rows the fused forward will use."""
    c, p, g, m, r = ctypes.c_int(), ctypes.c_int(), ctypes.c_int(), ctypes.c_int(), ctypes.c_int64()
    _check("mok_fused_plan", lib().mok_fused_plan(cfg.ref, ctypes.byref(c), ctypes.byref(p), ctypes.byref(g),
                                                  ctypes.byref(m), ctypes.byref(r)))
    return {"ctas": c.value, "cta_pairs": p.value, "gather_ctas": g.value, "minibatch_rows": m.value,
            "ring_rows": r.value}


def reset_device_status(ws, stream=None):
    _check("mok_reset_device_status", lib().mok_reset_device_status(_ptr(ws), _stream(stream)))


def get_device_status(ws, stream=None) -> int:
    return int(lib().mok_get_device_status(_ptr(ws), _stream(stream)))


def status_string(code: int) -> str:
    return lib().mok_status_string(code).decode()
