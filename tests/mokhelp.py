"""Shared pieces of the GPU parity tests: conversions between torch device
tensors and the oracle's numpy arrays, the MX scale-layout permutation, and
the tolerance check.  Nothing here computes any step of the layer."""
from __future__ import annotations

import hashlib
import json
import os

import numpy as np
import torch

from combine_top_routing_gb300 import inputs as I
from combine_top_routing_gb300 import mok
from combine_top_routing_gb300.layer import MoELayer
from oracle import oracle as O

# Tolerances for BF16 / fp32-accumulated outputs and gradients (GPU vs oracle):
# relative L2 error, and max-abs error measured per element in units of
# max(1, |ref_i|, scale_i): absolute for O(1) values, relative for values
# above 1 (one BF16 ulp at |v| in [4, 8) is 0.031 > 2e-2), and, for the
# elements of a reduction, relative to the root-sum-square of its terms
# (scale_i, from the oracle's terms_rss family): a sum whose terms carry
# independent roundings is off by a multiple of that, however far the sum
# itself cancels.
REL_L2 = 5e-3
MAX_ABS = 2e-2
# MXFP8 weight gradients compared end to end (the oracle's own forward and
# backward): the GPU's h, dy, da, db and the oracle's can differ by one BF16
# ulp, and the weight-gradient GEMMs re-quantise them to MXFP8 along the token
# rows, so a fraction phi of the E4M3 codes can land one step (at most 2^-3 of
# the element) apart.  Independent flips add in quadrature: against the terms'
# root-sum-square the error is at most 2^-3 sqrt(phi); 2^-4 admits phi <= 1/4.
MAX_ABS_MX_CHAIN = 2.0 ** -4


def bf16_np(t: torch.Tensor) -> np.ndarray:
    """BF16 tensor (any device) -> fp64 numpy values."""
    bits = t.detach().contiguous().view(torch.int16).cpu().numpy().view(np.uint16)
    return O.bf16_values(bits)


def f32_np(t: torch.Tensor) -> np.ndarray:
    return t.detach().float().cpu().numpy().astype(np.float64)


def scales_to_canonical(words: torch.Tensor | np.ndarray, rows: int, K: int) -> np.ndarray:
    """MX scale tile layout (see include/mok.h) -> canonical [rows, K/32] bytes."""
    w = words.cpu().numpy() if isinstance(words, torch.Tensor) else words
    b = np.ascontiguousarray(w).view(np.uint8).reshape(K // 128, rows // 128, 32, 4, 4)
    # b[g, rb, r%32, (r%128)//32, byte]
    out = b.transpose(1, 3, 2, 0, 4).reshape(rows, K // 32)
    return out


def check_close(got: np.ndarray, ref: np.ndarray, rel=REL_L2, mabs=MAX_ABS, what="", scale=None):
    got = np.asarray(got, dtype=np.float64)
    ref = np.asarray(ref, dtype=np.float64)
    assert got.shape == ref.shape, (what, got.shape, ref.shape)
    assert np.all(np.isfinite(got)), f"{what}: non-finite values"
    err = np.linalg.norm(got - ref) / max(np.linalg.norm(ref), 1e-30)
    unit = np.maximum(1.0, np.abs(ref))
    if scale is not None:
        unit = np.maximum(unit, np.asarray(scale, dtype=np.float64))
    d = np.abs(got - ref)
    mx = float((d / unit).max()) if got.size else 0.0
    diag = os.environ.get("MOK_TEST_DIAG")
    if diag and got.size:
        i = int(np.argmax(d / unit))
        with open(diag, "a") as f:
            f.write(json.dumps({
                "test": os.environ.get("PYTEST_CURRENT_TEST", "").split(" ")[0], "what": what,
                "n": int(got.size), "rel_l2": float(err), "max_abs": float(d.max()),
                "max_units": mx, "ref_at_max": float(ref.reshape(-1)[i]),
                "unit_at_max": float(unit.reshape(-1)[i]),
                "max_units_1_ref": float((d / np.maximum(1.0, np.abs(ref))).max())}) + "\n")
    assert err <= rel and mx <= mabs, f"{what}: rel_l2={err:.3e} max_abs={mx:.3e}"
    return err, mx


def sha(t: torch.Tensor) -> str:
    return hashlib.sha256(t.contiguous().view(torch.uint8).cpu().numpy().tobytes()).hexdigest()


def make_layer(w: I.Workload, training=False, **kw) -> tuple[MoELayer, dict]:
    inp = I.make_inputs(w, device="cuda")
    return MoELayer(w, inp, training=training, **kw), inp


class Routed:
    """Runs mok_route_layout into fresh tensors."""

    def __init__(self, layer: MoELayer):
        w = layer.w
        dev = "cuda"
        self.ids = torch.empty((w.T, w.k), dtype=torch.int32, device=dev)
        self.gates = torch.empty((w.T, w.k), dtype=torch.float32, device=dev)
        self.sel = torch.empty((w.T, w.k), dtype=torch.float32, device=dev)
        self.logits = torch.empty((w.T, w.E), dtype=torch.float32, device=dev)
        self.counts = torch.empty(w.E, dtype=torch.int32, device=dev)
        self.offsets = torch.empty(w.E + 1, dtype=torch.int32, device=dev)
        self.pad_offsets = torch.empty(w.E + 1, dtype=torch.int32, device=dev)
        self.slot_pos = torch.empty((w.T, w.k), dtype=torch.int32, device=dev)
        self.row_tok = torch.empty(w.S, dtype=torch.int32, device=dev)
        self.row_j = torch.empty(w.S, dtype=torch.uint8, device=dev)
        mok.route_layout(layer.cfg, layer.x_src, layer.W_r, layer.bias, self.ids, self.gates,
                         self.sel, self.logits, self.counts, self.offsets, self.pad_offsets,
                         self.slot_pos, self.row_tok, self.row_j, layer.ws)


def expert_weights_np(inp: dict, e: int):
    return (bf16_np(inp["Wg"][e]), bf16_np(inp["Wu"][e]), bf16_np(inp["Wd"][e]))


def near_tie_tokens(logits_ref: np.ndarray, k: int, margin: float) -> np.ndarray:
    """Tokens whose k-th and (k+1)-th largest oracle logits are within margin."""
    s = -np.sort(-logits_ref, axis=1)
    if s.shape[1] <= k:
        return np.zeros(s.shape[0], dtype=bool)
    return (s[:, k - 1] - s[:, k]) < margin
