"""A convenience owner of the device buffers one MoE layer call needs.

The library never allocates; this class allocates the caller-side buffers
(workspace, saved context, outputs, MXFP8 weight copies) with torch and
calls the C ABI through ``mok``.
"""
from __future__ import annotations

import torch

from . import mok
from .inputs import Workload, split_sources


def scale_words(rows: int, K: int) -> int:
    """32-bit words of an MX scale tile-layout buffer for a [rows, K] matrix."""
    return rows * K // 128


class MoELayer:
    def __init__(self, w: Workload, inputs: dict, *, training: bool = False, device="cuda",
                 **cfg_kw):
        self.w = w
        self.cfg = mok.Config.from_workload(w, **cfg_kw)
        self.device = torch.device(device)
        fwd, ctx, bwd = mok.workspace_size(self.cfg)
        self.ws = torch.empty(fwd, dtype=torch.uint8, device=self.device)
        self.ctx = torch.empty(ctx, dtype=torch.uint8, device=self.device) if training else None
        self.ctx_layout = mok.saved_ctx_layout(self.cfg)
        self.rows_pad = mok.max_padded_rows(self.cfg)
        x = inputs["x"]
        self.x = x
        self.x_src = split_sources(x, w.n_sources) if w.n_sources > 1 else [x]
        self.W_r = inputs["Wr"]
        self.bias = inputs.get("bias")
        self.weights = {"w_gate": inputs["Wg"], "w_up": inputs["Wu"], "w_down": inputs["Wd"]}
        if w.dtype == "mxfp8":
            self.quantize_weights()
        self.wstruct = mok.weights_struct(self.weights)
        self.out = torch.empty((w.T, w.d), dtype=torch.bfloat16, device=self.device)

    def quantize_weights(self, transposed: bool = False, stream=None):
        w, E, F, d = self.w, self.w.E, self.w.F, self.w.d
        dev = self.device
        q = self.weights
        for name, src, rows, K in (("gate", q["w_gate"], F, d), ("up", q["w_up"], F, d),
                                   ("down", q["w_down"], d, F)):
            codes = torch.empty((E, rows, K), dtype=torch.uint8, device=dev)
            scales = torch.empty(scale_words(E * rows, K), dtype=torch.int32, device=dev)
            mok.quantize_mx(src, E, rows, K, 0, codes, scales, stream)
            q["q_" + name], q["s_" + name] = codes, scales
            if transposed:
                codes_t = torch.empty((E, K, rows), dtype=torch.uint8, device=dev)
                scales_t = torch.empty(scale_words(E * K, rows), dtype=torch.int32, device=dev)
                mok.quantize_mx(src, E, rows, K, 1, codes_t, scales_t, stream)
                q["qt_" + name], q["st_" + name] = codes_t, scales_t
        self.wstruct = mok.weights_struct(q)

    def prepare_backward(self, stream=None):
        """Transposed weight copies the backward GEMMs read (K-major for dgrad)."""
        w, E, F, d = self.w, self.w.E, self.w.F, self.w.d
        q = self.weights
        if w.dtype == "mxfp8":
            if "qt_gate" not in q:
                self.quantize_weights(transposed=True, stream=stream)
        else:
            for name, src, rows, K in (("gate", q["w_gate"], F, d), ("up", q["w_up"], F, d),
                                       ("down", q["w_down"], d, F)):
                t = torch.empty((E, K, rows), dtype=torch.bfloat16, device=self.device)
                mok.transpose_bf16(src, E, rows, K, t, stream)
                q["wt_" + name] = t
            self.wstruct = mok.weights_struct(q)
        if not hasattr(self, "bws"):
            self.bws = torch.empty(mok.workspace_size(self.cfg)[2], dtype=torch.uint8,
                                   device=self.device)
            self.grads = {"d_gate": torch.empty((E, F, d), dtype=torch.bfloat16, device=self.device),
                          "d_up": torch.empty((E, F, d), dtype=torch.bfloat16, device=self.device),
                          "d_down": torch.empty((E, d, F), dtype=torch.bfloat16, device=self.device)}
            self.gstruct = mok.weight_grads_struct(self.grads)
            self.dX = torch.empty((w.T, w.d), dtype=torch.bfloat16, device=self.device)
            self.dgates = torch.empty((w.T, w.k), dtype=torch.float32, device=self.device)
            self.dlogits = torch.empty((w.T, w.E), dtype=torch.float32, device=self.device)
            self.dW_r = torch.empty((w.E, w.d), dtype=torch.float32, device=self.device)

    def backward(self, dY, stream=None, dlogits=True):
        assert self.ctx is not None, "backward needs a layer built with training=True"
        mok.moe_backward(self.cfg, self.x_src, self.W_r, self.ctx, dY, self.wstruct, self.dX,
                         self.gstruct, self.dgates, self.dlogits if dlogits else None, self.dW_r,
                         self.bws, stream)
        return self.dX

    def forward(self, stream=None):
        mok.moe_forward(self.cfg, self.x_src, self.W_r, self.bias, self.wstruct, self.out,
                        self.ctx, self.ws, stream)
        return self.out

    def status(self, stream=None) -> int:
        return mok.get_device_status(self.ws, stream)

    # -- views into the saved context (training) ------------------------------
    def ctx_view(self, field: str, dtype, shape):
        off = getattr(self.ctx_layout, field)
        n = 1
        for s in shape:
            n *= s
        nbytes = n * torch.tensor([], dtype=dtype).element_size()
        return self.ctx[off:off + nbytes].view(dtype).view(shape)
