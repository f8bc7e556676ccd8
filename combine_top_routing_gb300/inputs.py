"""Seeded synthetic inputs for the MoE layer workloads.

This module only draws random tensors of the right shapes, dtypes and
distributions; it holds none of the layer's arithmetic, and both the CUDA
path and the CPU oracle take their inputs from it.

The pages run Kimi-2.5 / DeepSeek-V3-shaped layers (hidden 7168, expert
intermediate 2048: "Cursor's MoK achieves 2.37x performance boost on NVIDIA
GB300 NVL72", kucoin.com, §02, the minibatch paragraph) on training data we
do not have, so every tensor is drawn from the distributions below:

  x ~ N(0,1) as BF16;  W_g, W_u ~ N(0, 1/d), W_d ~ N(0, 1/F) as BF16
  (std = 1/sqrt(fan_in));  router W_r ~ N(0, 0.02^2) for the tiny layer and
  N(0, 1/d) otherwise (logits ~ N(0,1), near-uniform load), fp32;
  dY ~ N(0,1) as BF16.
  Skewed layer: per-expert logit bias b_e = -alpha * 1.2 * ln(rank_e), rank a
  seeded permutation of 1..E and alpha = 0.46, which puts about 20x the mean
  load on the hottest expert (measured on the drawn logits, reported by the
  benchmark).

Tensors are drawn with torch generators on the device that will hold them
(one generator per tensor, seeded from the workload seed), expert by expert
for the large weight tensors so that no fp32 copy of a whole weight tensor is
ever materialised.
"""
from __future__ import annotations

import dataclasses
import math

import torch


@dataclasses.dataclass(frozen=True)
class Workload:
    name: str
    T: int
    d: int
    E: int
    k: int
    F: int
    dtype: str            # "bf16" | "mxfp8"
    router: str           # "softmax" | "sigmoid"
    seed: int
    wr_std: float | None = None     # None: 1/sqrt(d)
    zipf_alpha: float = 0.0         # > 0: skewed per-expert logit bias
    n_sources: int = 1              # > 1: tokens live in this many source buffers
    ring_bytes: int = 0
    backward: bool = False

    @property
    def S(self) -> int:
        return self.T * self.k

    @property
    def source_rows(self) -> list[int]:
        assert self.T % self.n_sources == 0
        return [self.T // self.n_sources] * self.n_sources


WORKLOADS = {
    "tiny": Workload("tiny", T=128, d=128, E=8, k=2, F=256, dtype="bf16",
                     router="softmax", seed=0, wr_std=0.02),
    "mixtral_bf16": Workload("mixtral_bf16", T=8192, d=4096, E=8, k=2, F=14336,
                             dtype="bf16", router="softmax", seed=1),
    "dsv3_mxfp8": Workload("dsv3_mxfp8", T=16384, d=7168, E=256, k=8, F=2048,
                           dtype="mxfp8", router="sigmoid", seed=2),
    "dsv3_skew_ep": Workload("dsv3_skew_ep", T=16384, d=7168, E=256, k=8, F=2048,
                             dtype="mxfp8", router="sigmoid", seed=3, zipf_alpha=0.46,
                             n_sources=64, ring_bytes=256 << 20),
    "dsv3_fwdbwd": Workload("dsv3_fwdbwd", T=8192, d=7168, E=256, k=8, F=2048,
                            dtype="mxfp8", router="sigmoid", seed=4, backward=True),
}


def scaled(w: Workload, **kw) -> Workload:
    """A copy of a workload with some fields replaced (smaller test cases)."""
    return dataclasses.replace(w, **kw)


def _gen(device, seed: int, stream: int) -> torch.Generator:
    g = torch.Generator(device=device)
    g.manual_seed(seed * 1_000_003 + stream)
    return g


def _normal(shape, std, device, gen, dtype):
    return (torch.randn(shape, generator=gen, device=device, dtype=torch.float32) * std).to(dtype)


def make_inputs(w: Workload, device="cpu", with_weights=True) -> dict:
    """Draw every input tensor of workload ``w`` on ``device``."""
    dev = torch.device(device)
    out = {}
    out["x"] = _normal((w.T, w.d), 1.0, dev, _gen(dev, w.seed, 1), torch.bfloat16)
    wr_std = w.wr_std if w.wr_std is not None else 1.0 / math.sqrt(w.d)
    out["Wr"] = _normal((w.E, w.d), wr_std, dev, _gen(dev, w.seed, 2), torch.float32)
    if w.zipf_alpha > 0:
        g = torch.Generator(device="cpu")
        g.manual_seed(w.seed * 1_000_003 + 3)
        rank = torch.randperm(w.E, generator=g).to(torch.float64) + 1.0
        out["bias"] = (-w.zipf_alpha * 1.2 * torch.log(rank)).to(torch.float32).to(dev)
    else:
        out["bias"] = None
    if with_weights:
        Wg = torch.empty((w.E, w.F, w.d), dtype=torch.bfloat16, device=dev)
        Wu = torch.empty_like(Wg)
        Wd = torch.empty((w.E, w.d, w.F), dtype=torch.bfloat16, device=dev)
        gg, gu, gd = (_gen(dev, w.seed, s) for s in (4, 5, 6))
        for e in range(w.E):
            Wg[e] = _normal((w.F, w.d), 1 / math.sqrt(w.d), dev, gg, torch.bfloat16)
            Wu[e] = _normal((w.F, w.d), 1 / math.sqrt(w.d), dev, gu, torch.bfloat16)
            Wd[e] = _normal((w.d, w.F), 1 / math.sqrt(w.F), dev, gd, torch.bfloat16)
        out.update(Wg=Wg, Wu=Wu, Wd=Wd)
    out["dY"] = _normal((w.T, w.d), 1.0, dev, _gen(dev, w.seed, 7), torch.bfloat16)
    return out


def split_sources(x: torch.Tensor, n_sources: int) -> list[torch.Tensor]:
    """Token t = (T/n) * s + r lives in source buffer s at row r; each source is
    its own allocation, standing in for another rank's memory."""
    rows = x.shape[0] // n_sources
    return [x[s * rows:(s + 1) * rows].clone() for s in range(n_sources)]
