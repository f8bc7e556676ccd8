"""MoE-layer throughput on GB300: tokens/s of one forward layer (router top-k,
layout, pull dispatch, grouped SwiGLU FFN, weighted combine) through the C ABI,
and of the forward + backward layer.

    python bench.py [--gpus N] [--steps K] [--warmup W] [--workload NAME]
    python bench.py --impl reference ...   # the CPU oracle on the host cores

Default: the DeepSeek-V3-shaped MXFP8 forward (T 16384, d 7168, E 256, k 8,
F 2048); the same line carries the MXFP8 forward + backward at T 8192, the
Zipf-skewed layer's achieved expert load, and the Mixtral-shaped BF16 layer.

One JSON line on rank 0.  N > 1 runs under torch.distributed.run: every rank
runs its own independent layer on its own batch of T tokens (the layer is
per-token, so batches shard with no data-path collective: weak scaling); the
time is the max over ranks and the value the tokens of all ranks / that time.
Inputs are seeded synthetic tensors of the workload's shape (no dataset).
"""
from __future__ import annotations

import argparse
import json
import math
import os
import statistics
import subprocess
import sys
import tempfile
import time

ROOT = os.path.dirname(os.path.abspath(__file__))
sys.path.insert(0, ROOT)

METRIC = "MoE-layer tokens/s fwd & fwd+bwd on 1 GB300; % of FP8 TC / HBM roofline"
DEFAULT_WORKLOAD = "dsv3_mxfp8"
# forward + backward workload of each forward workload (the MXFP8 backward is
# quoted at T 8192), and the secondary BF16 layer reported beside the primary
FWD_BWD_OF = {"dsv3_mxfp8": "dsv3_fwdbwd", "dsv3_skew_ep": "dsv3_fwdbwd"}
SECONDARY = "mixtral_bf16"
# Tensor-pipe rate of tcgen05 MXFP8 (kind::mxf8f6f4, block-scaled, M 128 N 256)
# on shared-memory-resident tiles, one issuing thread per SM on all 152 SMs of
# this GB300, measured by a timing-only program; and the nameplate peaks.
MXFP8_PIPE_TFLOPS = 4850.0
NOMINAL = {"mxfp8_tflops": 4500.0, "bf16_tflops": 2250.0, "hbm_gbs": 8000.0}
L2_FLUSH_BYTES = 256 << 20


def _args():
    p = argparse.ArgumentParser()
    p.add_argument("--gpus", type=int, default=1)
    p.add_argument("--steps", type=int, default=50)
    p.add_argument("--warmup", type=int, default=5)
    p.add_argument("--impl", choices=["mok", "reference"], default="mok")
    p.add_argument("--workload", default=DEFAULT_WORKLOAD)
    p.add_argument("--no-cpu-baseline", action="store_true")
    p.add_argument("--no-backward", action="store_true")
    p.add_argument("--no-secondary", action="store_true",
                   help="skip the secondary (Mixtral-shaped BF16) layer and the skew report")
    p.add_argument("--sweep", action="store_true",
                   help="also time the fused forward over gather SM fraction x minibatch")
    p.add_argument("--cpu-sample-tokens", type=int, default=0)
    p.add_argument("--set", action="append", default=[], metavar="FIELD=VALUE",
                   help="override a workload field (e.g. T=2048, E=32) for profiling runs")
    return p.parse_args()


def _workload(args):
    from combine_top_routing_gb300 import inputs as I
    w = I.WORKLOADS[args.workload]
    over = {}
    for item in args.set:
        k, v = item.split("=", 1)
        over[k] = type(getattr(w, k))(v)
    return I.scaled(w, **over) if over else w


def _dist():
    rank = int(os.environ.get("RANK", "0"))
    world = int(os.environ.get("WORLD_SIZE", "1"))
    local = int(os.environ.get("LOCAL_RANK", "0"))
    return rank, world, local


def reduce_max(value: float, device=None) -> float:
    """Max of `value` over the ranks of the default process group (the job's
    time is its slowest rank's); the value itself when not distributed."""
    import torch
    import torch.distributed as dist
    if not (dist.is_available() and dist.is_initialized()) or dist.get_world_size() == 1:
        return value
    t = torch.tensor([value], dtype=torch.float64, device=device or "cpu")
    dist.all_reduce(t, op=dist.ReduceOp.MAX)
    return float(t.item())


def job_throughput(tokens_per_rank: int, world: int, ms_max: float) -> float:
    """Whole-job tokens/s: every rank's tokens over the slowest rank's time."""
    return world * tokens_per_rank / (ms_max / 1e3)


def _peaks():
    path = os.path.join(ROOT, "MEASURED_PEAKS.json")
    if os.path.exists(path):
        with open(path) as f:
            d = json.load(f)
        return d, "measured"
    return {"hbm_gbs": 6800.0, "bf16_tflops": 1900.0, "bf16_tflops_sustained": 1700.0}, "fallback"


class ClockSampler:
    """nvidia-smi clock / throttle sampling while the timed region runs."""

    FIELDS = ("timestamp,index,clocks.sm,clocks.max.sm,power.draw,clocks_event_reasons.active,"
              "clocks_event_reasons.hw_slowdown,clocks_event_reasons.hw_thermal_slowdown,"
              "clocks_event_reasons.sw_thermal_slowdown,clocks_event_reasons.sw_power_cap")

    def __init__(self, gpu_index: int):
        self.gpu = gpu_index
        self.proc = None
        self.file = None
        self.window = None  # (t0, t1) host wall-clock of the timed region

    def mark(self, t0: float, t1: float):
        self.window = (t0, t1)

    def __enter__(self):
        try:
            self.file = tempfile.NamedTemporaryFile("w+", suffix=".csv", delete=False)
            self.proc = subprocess.Popen(
                ["nvidia-smi", f"--id={self.gpu}", f"--query-gpu={self.FIELDS}",
                 "--format=csv,noheader,nounits", "-lms", "100"],
                stdout=self.file, stderr=subprocess.DEVNULL)
        except (OSError, FileNotFoundError):
            self.proc = None
        return self

    def __exit__(self, *exc):
        if self.proc is not None:
            self.proc.terminate()
            try:
                self.proc.wait(timeout=5)
            except subprocess.TimeoutExpired:
                self.proc.kill()

    def summary(self, sm_max_default):
        if self.proc is None or self.file is None:
            return {"sm_mhz": None, "sm_max_mhz": sm_max_default, "reasons": ["unsampled"]}
        self.file.flush()
        with open(self.file.name) as f:
            rows = [r.strip().split(",") for r in f if r.strip()]
        os.unlink(self.file.name)
        import datetime
        parsed = []
        for r in rows:
            if len(r) < 10:
                continue
            try:
                ts = datetime.datetime.strptime(r[0].strip(), "%Y/%m/%d %H:%M:%S.%f").timestamp()
                parsed.append((ts, float(r[2]), float(r[3]), r[6:10]))
            except ValueError:
                continue
        inside = parsed
        if self.window and parsed:
            t0, t1 = self.window
            inside = [p for p in parsed if t0 - 0.05 <= p[0] <= t1 + 0.05]
            if not inside:  # timed region shorter than the sampling period
                inside = [min(parsed, key=lambda p: abs(p[0] - 0.5 * (t0 + t1)))]
        names = ["hw_slowdown", "hw_thermal_slowdown", "sw_thermal_slowdown", "sw_power_cap"]
        reasons = set()
        for p in inside:
            for n, v in zip(names, p[3]):
                if v.strip().lower() == "active":
                    reasons.add(n)
        sm = [p[1] for p in inside]
        smax = [p[2] for p in inside]
        return {"sm_mhz": statistics.median(sm) if sm else None,
                "sm_max_mhz": max(smax) if smax else sm_max_default,
                "reasons": sorted(reasons), "samples": len(sm)}


def _layer_flops(w):
    return 6.0 * w.S * w.d * w.F


def _layer_bytes(w):
    """Algorithmic HBM bytes of one forward: every byte the method must move once."""
    e = 1 if w.dtype == "mxfp8" else 2
    sc = 1 / 32 if w.dtype == "mxfp8" else 0
    weights = w.E * 3 * w.F * w.d * (e + sc)
    x = w.T * w.d * 2
    xe = 2 * w.S * w.d * (e + sc)
    h = 2 * w.S * w.F * (e + sc)
    ystage = 2 * w.S * w.d * 2
    out = w.T * w.d * 2
    return weights + x + xe + h + ystage + out


# DRAM bytes (read + write) of one mok_moe_fused call -- the dispatch kernel (when
# the plan gathers first), the fused kernel and the combine kernel -- from one ncu
# capture (`--metrics dram__bytes_read.sum,dram__bytes_write.sum`) of a case small
# enough to capture: the same per-expert shape with the tokens and experts cut by
# `scale`, multiplied by `scale` (the weights, activations and staging all grow in
# proportion).  Keyed by workload and CTA pairs, with a hash of the kernels'
# sources at capture time (comments and blank lines left out): once their code
# changes, traffic is null.
FUSED_TRAFFIC = {
    # T 2048 / E 32 (1/8 of the tokens and experts): k_dispatch_by_token<1> 29.709 MB
    # read + 60.419 MB written, k_moe_fused_pair<1> 1628.526 + 244.993 MB,
    # k_combine<8> 234.963 + 17.933 MB
    ("dsv3_mxfp8", 1): {"bytes_small": 29708800 + 60418816 + 1628526080 + 244992512 + 234963200 + 17933312,
                        "scale": 8,
                        "case": "T 2048, 32 experts (1/8 of the tokens and experts); dispatch, fused and "
                                "combine kernels",
                        "src_sha": "ca1272697b0c8c80"},
    # full size (a few GB on the device): k_moe_fused_pair<0> 4407.417 MB read + 764.237 MB
    # written, k_combine<2> 134.295 + 30.839 MB (the split gather is inside the fused kernel)
    ("mixtral_bf16", 1): {"bytes_small": 4407416576 + 764236800 + 134294784 + 30838528, "scale": 1,
                          "case": "full size; fused and combine kernels",
                          "src_sha": "ca1272697b0c8c80"},
}
FUSED_SOURCES = ("mok_fused.cu", "mok_tc.cuh", "mok_ptx.cuh", "mok_internal.h", "mok_gather.cuh", "mok_move.cu")


def _fused_src_sha() -> str:
    import hashlib
    h = hashlib.sha256()
    for f in FUSED_SOURCES:
        with open(os.path.join(ROOT, "combine_top_routing_gb300", "csrc", f), encoding="utf-8") as fh:
            for line in fh:
                code = line.split("//", 1)[0].rstrip()
                if code:
                    h.update(code.encode() + b"\n")
    return h.hexdigest()[:16]


def _fused_traffic(workload: str, pairs: int):
    e = FUSED_TRAFFIC.get((workload, pairs))
    if e is None or e["src_sha"] != _fused_src_sha():
        return None
    return {"bytes": e["bytes_small"] * e["scale"], "captured": e["case"], "scale": e["scale"]}


def _dispatch_bytes(w):
    """Algorithmic HBM bytes of the pull dispatch: every token row read once,
    every slot row written once (codes + scales), the row index read."""
    e = 1 if w.dtype == "mxfp8" else 2
    sc = 1 / 32 if w.dtype == "mxfp8" else 0
    return w.T * w.d * 2 + w.S * w.d * (e + sc) + w.S * 4


def _combine_bytes(w):
    """Algorithmic HBM bytes of the weighted combine: every staged y row and
    gate read once, every output row written once."""
    return w.S * w.d * 2 + w.S * 4 + w.T * w.d * 2


def run_reference(args):
    """The oracle as it stands, timed on the host cores on a bounded token sample."""
    rank, world, _ = _dist()
    if rank != 0:
        return 0
    import numpy as np
    import torch

    from combine_top_routing_gb300 import inputs as I
    from oracle import oracle as O
    w = _workload(args)
    # inputs are drawn where the GPU arm draws them (same values); the oracle
    # converts each expert's weights to fp64 on the host when it uses them
    dev = "cuda" if torch.cuda.is_available() else "cpu"
    inp = I.make_inputs(w, device=dev)
    kind = O.SOFTMAX if w.router == "softmax" else O.SIGMOID

    def bf(t):
        return O.bf16_values(t.contiguous().view(torch.int16).cpu().numpy().view(np.uint16))

    # tokens per step: every step pays the fp64 conversion and MXFP8
    # quantisation of each expert its tokens touch (~0.3 s per expert at the
    # DeepSeek-V3 shape), so steps stay a few seconds: 256 tokens over 8
    # experts, 2 tokens (16 experts) over 256
    ntok = min(w.T, args.cpu_sample_tokens or (256 if w.E <= 16 else 2))
    rng = np.random.default_rng(0)
    x = bf(inp["x"])
    Wr = inp["Wr"].double().cpu().numpy()
    bias = None if inp["bias"] is None else inp["bias"].double().cpu().numpy()
    ge = lambda e: (bf(inp["Wg"][e]), bf(inp["Wu"][e]), bf(inp["Wd"][e]))

    def step():
        tok = np.sort(rng.choice(w.T, ntok, replace=False))
        O.forward(x, Wr, bias, ge, E=w.E, k=w.k, kind=kind, mode=w.dtype, tokens=tok)

    for _ in range(args.warmup):
        step()
    t0 = time.perf_counter()
    for _ in range(args.steps):
        step()
    dt = (time.perf_counter() - t0) / args.steps
    cores = len(os.sched_getaffinity(0))
    val = ntok / dt
    line = {
        "impl": "reference", "metric": METRIC, "value": val, "unit": "tokens/s",
        "n_gpus": args.gpus, "steps": args.steps, "warmup": args.warmup,
        "ms_per_step": dt * 1e3, "higher_is_better": True, "scaling": "weak",
        "vs_baseline": None, "dtype": "f64", "data": "synthetic",
        "config": {"workload": w.name, "T": w.T, "d_model": w.d, "experts": w.E, "top_k": w.k,
                   "d_ff": w.F, "gemm_dtype": w.dtype, "sample_tokens_per_step": ntok},
        "cpu_baseline": {"value": val, "unit": "tokens/s", "cores": cores, "kind": "oracle",
                         "cpu_model": _cpu_model(), "rate": "measured on a token sample, not extrapolated",
                         "sample": f"{ntok} random tokens of {w.name} (T {w.T}) per step (full layer "
                                   f"forward of those tokens, fp64 oracle)"},
        "e2e": {"value": val, "unit": "tokens/s", "h2d_bytes_per_step": 0, "d2h_bytes_per_step": 0},
    }
    print(json.dumps(line), flush=True)
    return 0


def _cpu_model() -> str:
    try:
        out = subprocess.run(["lscpu"], capture_output=True, text=True, timeout=10).stdout
        for line in out.splitlines():
            if line.lower().startswith("model name"):
                return line.split(":", 1)[1].strip()
    except (OSError, subprocess.SubprocessError):
        pass
    import platform
    return platform.processor() or platform.machine()


def cpu_baseline(w, inp_gpu, budget_s=20.0):
    """Oracle forward on a bounded token sample, on this host's cores: the rate
    measured on the sample (per-token work is uniform once routing is fixed)."""
    import numpy as np
    import torch

    from oracle import oracle as O
    kind = O.SOFTMAX if w.router == "softmax" else O.SIGMOID

    def bf(t):
        return O.bf16_values(t.contiguous().view(torch.int16).cpu().numpy().view(np.uint16))

    x = bf(inp_gpu["x"])
    Wr = inp_gpu["Wr"].double().cpu().numpy()
    bias = None if inp_gpu["bias"] is None else inp_gpu["bias"].double().cpu().numpy()
    ge = lambda e: (bf(inp_gpu["Wg"][e]), bf(inp_gpu["Wu"][e]), bf(inp_gpu["Wd"][e]))
    rng = np.random.default_rng(1)
    ntok, total_tok, t_total = 2, 0, 0.0
    while t_total < budget_s:
        tok = np.sort(rng.choice(w.T, ntok, replace=False))
        t0 = time.perf_counter()
        O.forward(x, Wr, bias, ge, E=w.E, k=w.k, kind=kind, mode=w.dtype, tokens=tok)
        t_total += time.perf_counter() - t0
        total_tok += ntok
        if t_total < budget_s / 4:
            ntok *= 2
    cores = len(os.sched_getaffinity(0))
    return {"value": total_tok / t_total, "unit": "tokens/s", "cores": cores, "kind": "oracle",
            "cpu_model": _cpu_model(), "rate": "measured on a token sample, not extrapolated",
            "sample": f"{total_tok} random tokens of {w.name} (T {w.T}) through the fp64 oracle "
                      f"forward, {t_total:.1f} s of CPU work; value = sampled tokens / that time"}


class L2Flush:
    """Writes a buffer twice the size of L2 between timed iterations, so that no
    iteration finds the previous one's data in L2."""

    def __init__(self):
        import torch
        self.buf = torch.empty(L2_FLUSH_BYTES // 4, dtype=torch.int32, device="cuda")

    def __call__(self):
        self.buf.fill_(0)


def time_flushed(fn, steps, stream, flush):
    """Mean CUDA-event time of `steps` calls of fn on `stream`, L2 flushed
    before each call (outside the timed events)."""
    import torch
    evs = [(torch.cuda.Event(enable_timing=True), torch.cuda.Event(enable_timing=True))
           for _ in range(steps)]
    for e0, e1 in evs:
        flush()
        e0.record(stream)
        fn()
        e1.record(stream)
    torch.cuda.synchronize()
    return sum(e0.elapsed_time(e1) for e0, e1 in evs) / steps


def _expert_load(w, dev="cuda"):
    """Achieved per-expert slot counts of workload w's routing (the router and
    layout through the C ABI; no expert weights needed)."""
    import torch

    from combine_top_routing_gb300 import inputs as I
    from combine_top_routing_gb300 import mok
    inp = I.make_inputs(w, device=dev, with_weights=False)
    cfg = mok.Config.from_workload(w)
    ws = torch.empty(mok.workspace_size(cfg)[0], dtype=torch.uint8, device=dev)
    x_src = I.split_sources(inp["x"], w.n_sources) if w.n_sources > 1 else [inp["x"]]
    ids = torch.empty((w.T, w.k), dtype=torch.int32, device=dev)
    gates = torch.empty((w.T, w.k), dtype=torch.float32, device=dev)
    counts = torch.empty(w.E, dtype=torch.int32, device=dev)
    offsets = torch.empty(w.E + 1, dtype=torch.int32, device=dev)
    pad = torch.empty(w.E + 1, dtype=torch.int32, device=dev)
    slot_pos = torch.empty((w.T, w.k), dtype=torch.int32, device=dev)
    row_tok = torch.empty(w.S, dtype=torch.int32, device=dev)
    row_j = torch.empty(w.S, dtype=torch.uint8, device=dev)
    mok.route_layout(cfg, x_src, inp["Wr"], inp["bias"], ids, gates, None, None, counts, offsets,
                     pad, slot_pos, row_tok, row_j, ws)
    c = counts.cpu().double()
    return {"workload": w.name, "hottest_over_mean": float(c.max() / c.mean()),
            "hottest_rows": int(c.max()), "coldest_rows": int(c.min()),
            "mean_rows": float(c.mean())}


def _layer_line(w, layer, stream, steps, flush, peaks):
    """Device-resident forward timing (L2 flushed between steps) of one layer."""
    import torch
    for _ in range(3):
        layer.forward()
    torch.cuda.synchronize()
    ms = time_flushed(layer.forward, steps, stream, flush)
    flops = _layer_flops(w)
    peak_tc = _tc_peak(w, peaks)
    return ms, {"tensor_frac": flops / (ms / 1e3) / 1e12 / peak_tc,
                "hbm_frac": _layer_bytes(w) / (ms / 1e3) / 1e9 / peaks.get("hbm_gbs", 6800.0)}


def _skewed_layer(w, stream, flush, peaks, world):
    """The Zipf-skewed, 64-source, 256 MB-ring layer: its forward with the
    automatic plan, and the gather share x minibatch sweep of the split gather,
    each point's output compared bit for bit with the automatic plan's."""
    import torch

    from combine_top_routing_gb300 import inputs as I
    from combine_top_routing_gb300 import mok
    from combine_top_routing_gb300.layer import MoELayer
    rank = int(os.environ.get("RANK", "0"))
    inp = I.make_inputs(I.scaled(w, seed=w.seed + 1000 * rank), device="cuda")
    layer = MoELayer(w, inp)
    ms, lr = _layer_line(w, layer, stream, 10, flush, peaks)
    ms = reduce_max(ms, "cuda")
    plan = mok.fused_plan(layer.cfg)
    ref = layer.out.clone()
    sweep = []
    for frac in (0.125, 0.25, 1 / 3):
        for mb in (64, 128, 256):
            layer.cfg.c.gather_sm_fraction = frac
            layer.cfg.c.minibatch_rows = mb
            layer.forward()
            torch.cuda.synchronize()
            same = bool(torch.equal(layer.out.view(torch.int16), ref.view(torch.int16)))
            sms = time_flushed(layer.forward, 5, stream, flush)
            if layer.status() != 0:
                raise RuntimeError("device status in the skewed sweep: " + mok.status_string(layer.status()))
            sweep.append({"gather_sm_fraction": round(frac, 4), "minibatch_rows": mb, "ms_per_step": sms,
                          "bit_identical_to_automatic_plan": same})
    out = {"forward_ms": ms, "value": job_throughput(w.T, world, ms), "unit": "tokens/s",
           "layer_roofline": lr, "fused_plan": plan, "sweep": sweep}
    del layer, inp, ref
    return out


def _tc_peak(w, peaks):
    """Measured dense tensor peak for the layer's GEMM dtype: the BF16 burst
    figure, x2 (the nominal FP8:BF16 ratio) for MXFP8."""
    return peaks.get("bf16_tflops", 1900.0) * (2.0 if w.dtype == "mxfp8" else 1.0)


def _fwd_bwd(w, stream, steps, flush, barrier, world):
    """Forward + backward of the training layer of workload w (saved context,
    weight gradients, router gradients), L2 flushed between steps."""
    import torch

    from combine_top_routing_gb300 import inputs as I
    from combine_top_routing_gb300 import mok
    from combine_top_routing_gb300.layer import MoELayer
    rank = int(os.environ.get("RANK", "0"))
    inp = I.make_inputs(I.scaled(w, seed=w.seed + 1000 * rank), device="cuda")
    tl = MoELayer(w, inp, training=True)
    tl.prepare_backward()

    def step():
        tl.forward()
        tl.backward(inp["dY"])

    for _ in range(3):
        step()
    torch.cuda.synchronize()
    barrier()
    ms = reduce_max(time_flushed(step, steps, stream, flush), "cuda")
    if tl.status() != 0:
        raise RuntimeError("device status after backward: " + mok.status_string(tl.status()))
    del tl, inp
    torch.cuda.empty_cache()
    return ms


def main():
    args = _args()
    if args.impl == "reference":
        return run_reference(args)
    rank, world, local = _dist()
    import torch
    import torch.distributed as dist

    from combine_top_routing_gb300 import inputs as I
    from combine_top_routing_gb300 import mok
    from combine_top_routing_gb300.layer import MoELayer

    torch.cuda.set_device(local)
    if world > 1:
        dist.init_process_group("nccl", device_id=torch.device("cuda", local))
    w = _workload(args)
    inp = I.make_inputs(I.scaled(w, seed=w.seed + 1000 * rank), device="cuda")
    layer = MoELayer(w, inp)
    stream = torch.cuda.current_stream()
    flush = L2Flush()

    def barrier():
        if world > 1:
            dist.barrier()

    # ---------------- device-resident timed region (L2 flushed between steps)
    peaks, peak_src = _peaks()
    with ClockSampler(local) as clk:
        for _ in range(max(3, args.warmup)):
            layer.forward()
        torch.cuda.synchronize()
        barrier()
        torch.cuda.synchronize()
        wall0 = time.time()
        ms = time_flushed(layer.forward, args.steps, stream, flush)
        clk.mark(wall0, time.time())
    barrier()
    status = layer.status()
    if status != 0:
        raise RuntimeError(f"device status {mok.status_string(status)}")
    ms = reduce_max(ms, "cuda")
    value = job_throughput(w.T, world, ms)
    flops = _layer_flops(w)
    peak_tc = _tc_peak(w, peaks)

    # ---------------- the dominant kernel (the fused forward) timed alone, same stream
    R = _route_for_ffn(layer)
    iters = max(5, min(50, args.steps))

    def timed(fn):
        for _ in range(2):
            fn()
        return time_flushed(fn, iters, stream, flush)

    def timed_n(fn, n):
        for _ in range(2):
            fn()
        return time_flushed(fn, n, stream, flush)

    # the HBM-bound steps on their own (separate kernels, same stream)
    disp_ms = timed(lambda: mok.dispatch(layer.cfg, layer.x_src, R.ids, R.offsets, R.pad_offsets,
                                         R.row_tok, R.row_j, R.xe, R.xs))
    disp_tok_ms = timed(lambda: mok.dispatch_by_token(layer.cfg, layer.x_src, R.ids, R.slot_pos, R.offsets,
                                                      R.pad_offsets, R.xe, R.xs))
    comb_ms = timed(lambda: mok.combine(layer.cfg, R.ystage, R.gates, layer.out))
    hbm_peak = peaks.get("hbm_gbs", 6800.0)
    hbm_steps = {}
    for name, ms_, nbytes in (("dispatch", disp_ms, _dispatch_bytes(w)),
                              ("dispatch_by_token", disp_tok_ms, _dispatch_bytes(w)),
                              ("combine", comb_ms, _combine_bytes(w))):
        gbs = nbytes / (ms_ / 1e3) / 1e9
        hbm_steps[name] = {"ms": ms_, "algorithmic_bytes": nbytes, "achieved_gbs": gbs,
                           "peak_gbs": hbm_peak, "frac": gbs / hbm_peak,
                           "frac_of_nominal_8tbs": gbs / NOMINAL["hbm_gbs"]}
    plan = mok.fused_plan(layer.cfg)
    fused_ms = timed(lambda: mok.moe_fused(layer.cfg, layer.x_src, layer.wstruct, R.ids, R.gates,
                                           R.counts, R.offsets, R.pad_offsets, R.slot_pos, R.row_tok, R.row_j,
                                           R.ystage, layer.out, layer.ws))
    ffn_ms = timed(lambda: _ffn(layer, R))
    fused_tflops = flops / (fused_ms / 1e3) / 1e12
    # router split, router GEMM, top-k, 4 layout passes, the fused kernel and the
    # combine kernel, and the dispatch kernel when the plan gathers first
    launches_per_step = 9 + (1 if plan["gather_ctas"] >= plan["ctas"] else 0)

    sweep = None
    if args.sweep:
        sweep = []
        for frac in (0.0625, 0.125, 0.25, 1 / 3):
            for mb in (64, 128, 256):
                layer.cfg.c.gather_sm_fraction = frac
                layer.cfg.c.minibatch_rows = mb
                sms = timed(layer.forward)
                if layer.status() != 0:
                    raise RuntimeError("device status in sweep: " + mok.status_string(layer.status()))
                sweep.append({"gather_sm_fraction": round(frac, 4), "minibatch_rows": mb,
                              "ms_per_step": sms})
        layer.cfg.c.gather_sm_fraction = 0.0
        layer.cfg.c.minibatch_rows = 0

    # ---------------- macrobatch pipelining: back-to-back calls, each call's
    # combine inside the next call's fused kernel (two workspaces alternating)
    chain = None
    if not args.no_secondary:
        n_chain = 4
        ws2 = torch.empty_like(layer.ws)
        outs = [torch.empty_like(layer.out) for _ in range(n_chain)]
        wss = [layer.ws if i % 2 == 0 else ws2 for i in range(n_chain)]

        def run_chain():
            mok.moe_forward_chain(layer.cfg, [layer.x_src] * n_chain, layer.W_r, layer.bias, layer.wstruct,
                                  outs, wss)

        def run_separate():
            for i in range(n_chain):
                mok.moe_forward(layer.cfg, layer.x_src, layer.W_r, layer.bias, layer.wstruct, outs[i], None,
                                wss[i])

        # the two arms alternate in rounds (the clock drifts under the power cap over
        # a long run); each arm's figure is its median over the rounds
        c_steps = max(3, min(args.steps, 5))
        rounds = 4
        chain_r, sep_r = [], []
        for _ in range(rounds):
            chain_r.append(timed_n(run_chain, c_steps) / n_chain)
            sep_r.append(timed_n(run_separate, c_steps) / n_chain)
        if layer.status() != 0 or mok.get_device_status(ws2) != 0:
            raise RuntimeError("device status after the chained calls")
        chain_ms = statistics.median(chain_r)
        sep_ms = statistics.median(sep_r)
        chain = {"calls": n_chain, "ms_per_call_chained": chain_ms, "ms_per_call_separate": sep_ms,
                 "saving_ms_per_call": sep_ms - chain_ms,
                 "saving_ms_per_round": [round(b - a, 4) for a, b in zip(chain_r, sep_r)],
                 "value_chained": job_throughput(w.T, world, reduce_max(chain_ms, "cuda")), "unit": "tokens/s",
                 "how": (f"mok_moe_forward_chain of {n_chain} calls vs {n_chain} mok_moe_forward calls, "
                         f"{rounds} alternating rounds of {c_steps} repeats each (median), "
                         "L2 flushed between repeats")}
        del ws2, outs
        torch.cuda.empty_cache()

    # ---------------- end to end through the C ABI with host buffers
    x_host = torch.empty_like(inp["x"], device="cpu").pin_memory()
    x_host.copy_(inp["x"].cpu())
    out_host = torch.empty((w.T, w.d), dtype=torch.bfloat16).pin_memory()
    e2e_steps = max(3, min(args.steps, 20))
    pipe = PipelinedE2E(layer, x_host, out_host)
    for i in range(2):
        pipe.step(i)
    torch.cuda.synchronize()
    barrier()
    torch.cuda.synchronize()
    t0 = time.perf_counter()
    for i in range(e2e_steps):
        pipe.step(i)
    torch.cuda.synchronize()
    e2e_ms = reduce_max((time.perf_counter() - t0) * 1e3 / e2e_steps, "cuda")
    if layer.status() != 0:
        raise RuntimeError("device status after the end-to-end steps: " + mok.status_string(layer.status()))
    e2e_val = job_throughput(w.T, world, e2e_ms)

    base = None
    if rank == 0 and not args.no_cpu_baseline:
        base = cpu_baseline(w, inp)
    del pipe, R, layer, inp
    torch.cuda.empty_cache()

    # ---------------- forward + backward (training layer: saved context)
    fb = None
    if not args.no_backward:
        wf = I.WORKLOADS[FWD_BWD_OF[w.name]] if w.name in FWD_BWD_OF else w
        fb_steps = max(3, min(args.steps, 20))
        fb_ms = _fwd_bwd(wf, stream, fb_steps, flush, barrier, world)
        fb = {"workload": wf.name, "T": wf.T, "gemm_dtype": wf.dtype,
              "value": job_throughput(wf.T, world, fb_ms), "unit": "tokens/s", "ms_per_step": fb_ms,
              "tensor_frac": 3 * _layer_flops(wf) / (fb_ms / 1e3) / 1e12 / _tc_peak(wf, peaks),
              "tensor_frac_of_nominal": 3 * _layer_flops(wf) / (fb_ms / 1e3) / 1e12 /
                                        NOMINAL["mxfp8_tflops" if wf.dtype == "mxfp8" else "bf16_tflops"],
              "steps": fb_steps, "l2": "flushed between timed steps"}

    # ---------------- skewed layer (load, forward, the gather-share x minibatch
    # sweep with its outputs compared bit for bit), secondary BF16 layer
    skew = secondary = None
    if not args.no_secondary:
        skew = _expert_load(I.WORKLOADS["dsv3_skew_ep"])
        torch.cuda.empty_cache()
        if w.name != "dsv3_skew_ep":
            skew.update(_skewed_layer(I.WORKLOADS["dsv3_skew_ep"], stream, flush, peaks, world))
            torch.cuda.empty_cache()
        if w.name != SECONDARY:
            w2 = I.WORKLOADS[SECONDARY]
            inp2 = I.make_inputs(I.scaled(w2, seed=w2.seed + 1000 * rank), device="cuda")
            l2 = MoELayer(w2, inp2)
            ms2, lr2 = _layer_line(w2, l2, stream, max(3, min(args.steps, 20)), flush, peaks)
            ms2 = reduce_max(ms2, "cuda")
            secondary = {"workload": w2.name, "T": w2.T, "gemm_dtype": w2.dtype, "pass": "forward",
                         "value": job_throughput(w2.T, world, ms2), "unit": "tokens/s",
                         "ms_per_step": ms2, "layer_roofline": lr2}
            if not args.no_backward:
                ms2b = _fwd_bwd(w2, stream, max(3, min(args.steps, 10)), flush, barrier, world)
                secondary["fwd_bwd"] = {"value": job_throughput(w2.T, world, ms2b), "unit": "tokens/s",
                                        "ms_per_step": ms2b,
                                        "tensor_frac": 3 * _layer_flops(w2) / (ms2b / 1e3) / 1e12 /
                                                       _tc_peak(w2, peaks)}
            del l2, inp2
            torch.cuda.empty_cache()

    if rank == 0:
        clocks = clk.summary(peaks.get("sm_max_mhz"))
        mx = w.dtype == "mxfp8"
        line = {
            "metric": METRIC, "value": value, "unit": "tokens/s", "n_gpus": world,
            "steps": args.steps, "warmup": max(3, args.warmup), "ms_per_step": ms,
            "higher_is_better": True, "scaling": "weak", "vs_baseline": None,
            "dtype": "mxfp8(e4m3+e8m0)/fp32-acc" if mx else "bf16/fp32-acc",
            "data": "synthetic",
            "config": {"workload": w.name, "T": w.T, "d_model": w.d, "experts": w.E,
                       "top_k": w.k, "d_ff": w.F, "gemm_dtype": w.dtype,
                       "router": w.router, "pass": "forward",
                       "l2": f"flushed between timed iterations ({L2_FLUSH_BYTES >> 20} MB written "
                             "outside the timed events)",
                       "parallelism": f"replicas x{world}"},
            "roofline": {"bound": "tensor", "achieved": fused_tflops, "peak": peak_tc,
                         "unit": "TFLOP/s", "frac": fused_tflops / peak_tc,
                         "traffic": None, "traffic_unit": "DRAM bytes per launch",
                         "kernel": (("k_dispatch_by_token (pull dispatch) + " if plan["gather_ctas"] >= plan["ctas"]
                                     else "")
                                    + ("k_moe_fused_pair" if plan["cta_pairs"] else "k_moe_fused")
                                    + (" (FFN1 + FFN2)" if plan["gather_ctas"] >= plan["ctas"]
                                       else " (pull dispatch by its gather CTAs + FFN1 + FFN2)")
                                    + " + k_combine, one mok_moe_fused call"),
                         "algorithmic": "6*S*d*F flops per launch",
                         "peak_source": f"{peak_src} bf16 burst"
                                        + (" x2 (nominal fp8:bf16 ratio)" if mx else ""),
                         "frac_of_tensor_pipe_measured": (fused_tflops / MXFP8_PIPE_TFLOPS) if mx else None,
                         "frac_of_nominal": fused_tflops / NOMINAL["mxfp8_tflops" if mx else "bf16_tflops"],
                         "ms_per_launch": fused_ms},
            "expert_ffn_separate_kernels": {"ms": ffn_ms,
                                            "tflops": flops / (ffn_ms / 1e3) / 1e12},
            "hbm_steps": hbm_steps,
            "fused_plan": plan,
            "sweep": sweep,
            "layer_roofline": {"tensor_frac": flops / (ms / 1e3) / 1e12 / peak_tc,
                               "tensor_frac_of_nominal": flops / (ms / 1e3) / 1e12 /
                                   NOMINAL["mxfp8_tflops" if mx else "bf16_tflops"],
                               "hbm_frac": _layer_bytes(w) / (ms / 1e3) / 1e9 /
                                           peaks.get("hbm_gbs", 6800.0),
                               "hbm_frac_of_nominal": _layer_bytes(w) / (ms / 1e3) / 1e9 / NOMINAL["hbm_gbs"]},
            "fwd_bwd": fb,
            "expert_load_skewed": skew,
            "macrobatch_chain": chain,
            "secondary": secondary,
            "e2e": {"value": e2e_val, "unit": "tokens/s",
                    "h2d_bytes_per_step": w.T * w.d * 2, "d2h_bytes_per_step": w.T * w.d * 2,
                    "how": "mok_moe_forward per step from pinned host x to pinned host out; copy-in, "
                           "layer and copy-out on three streams with two device buffers (host wall "
                           "time over the steps)"},
            "gpu_launches": launches_per_step * args.steps,
            "clocks": clocks,
            "cpu_baseline": base,
        }
        tr = _fused_traffic(w.name, plan["cta_pairs"])
        if tr is not None:
            line["roofline"]["traffic"] = tr["bytes"]
            line["roofline"]["traffic_how"] = (f"ncu dram__bytes_read.sum + dram__bytes_write.sum of one "
                                               f"mok_moe_fused call at {tr['captured']}, x{tr['scale']}")
        print(json.dumps(line), flush=True)
    if world > 1:
        dist.destroy_process_group()
    return 0


def _route_for_ffn(layer):
    """Route once so that the FFN alone can be timed on fixed layout buffers."""
    import torch
    w = layer.w
    class R:
        pass
    r = R()
    dev = "cuda"
    r.ids = torch.empty((w.T, w.k), dtype=torch.int32, device=dev)
    r.gates = torch.empty((w.T, w.k), dtype=torch.float32, device=dev)
    r.counts = torch.empty(w.E, dtype=torch.int32, device=dev)
    r.offsets = torch.empty(w.E + 1, dtype=torch.int32, device=dev)
    r.pad_offsets = torch.empty(w.E + 1, dtype=torch.int32, device=dev)
    r.slot_pos = torch.empty((w.T, w.k), dtype=torch.int32, device=dev)
    r.row_tok = torch.empty(w.S, dtype=torch.int32, device=dev)
    r.row_j = torch.empty(w.S, dtype=torch.uint8, device=dev)
    from combine_top_routing_gb300 import mok
    from combine_top_routing_gb300.layer import scale_words
    mok.route_layout(layer.cfg, layer.x_src, layer.W_r, layer.bias, r.ids, r.gates, None, None,
                     r.counts, r.offsets, r.pad_offsets, r.slot_pos, r.row_tok, r.row_j, layer.ws)
    rows = layer.rows_pad
    if w.dtype == "mxfp8":
        r.xe = torch.empty((rows, w.d), dtype=torch.uint8, device=dev)
        r.xs = torch.empty(scale_words(rows, w.d), dtype=torch.int32, device=dev)
    else:
        r.xe = torch.empty((rows, w.d), dtype=torch.bfloat16, device=dev)
        r.xs = None
    mok.dispatch(layer.cfg, layer.x_src, r.ids, r.offsets, r.pad_offsets, r.row_tok, r.row_j,
                 r.xe, r.xs)
    r.ystage = torch.empty((w.T, w.k, w.d), dtype=torch.bfloat16, device=dev)
    return r


def _ffn(layer, r):
    from combine_top_routing_gb300 import mok
    mok.expert_ffn(layer.cfg, r.xe, r.xs, layer.wstruct, r.offsets, r.pad_offsets, r.row_tok,
                   r.row_j, r.ystage, None, None, None, layer.ws)


class PipelinedE2E:
    """End to end through the C ABI from pinned host memory: every step copies
    its input rows host -> device, runs the layer (mok_moe_forward) and copies
    its output device -> host.  Three streams (copy in, compute, copy out) and
    two device input / output buffers let step i+1's upload and step i-1's
    read-back overlap step i's layer; events order every buffer's reuse."""

    def __init__(self, layer, x_host, out_host):
        import torch
        self.layer, self.x_host, self.out_host = layer, x_host, out_host
        w = layer.w
        self.s_c = torch.cuda.current_stream()
        self.s_in, self.s_out = torch.cuda.Stream(), torch.cuda.Stream()
        rows = w.T // w.n_sources
        self.src = [[torch.empty((rows, w.d), dtype=torch.bfloat16, device="cuda") for _ in range(w.n_sources)]
                    for _ in range(2)]
        self.rows = rows
        self.out = [torch.empty_like(layer.out) for _ in range(2)]
        self.ev_in = [torch.cuda.Event() for _ in range(2)]
        self.ev_used = [torch.cuda.Event() for _ in range(2)]
        self.ev_read = [torch.cuda.Event() for _ in range(2)]
        self.used = [False, False]

    def step(self, i):
        import torch
        from combine_top_routing_gb300 import mok
        b = i % 2
        lay = self.layer
        with torch.cuda.stream(self.s_in):
            if self.used[b]:
                self.s_in.wait_event(self.ev_used[b])  # the layer that read this buffer is done
            for s, buf in enumerate(self.src[b]):
                buf.copy_(self.x_host[s * self.rows:(s + 1) * self.rows], non_blocking=True)
            self.ev_in[b].record(self.s_in)
        self.s_c.wait_event(self.ev_in[b])
        if self.used[b]:
            self.s_c.wait_event(self.ev_read[b])  # this output buffer has been read back
        mok.moe_forward(lay.cfg, self.src[b], lay.W_r, lay.bias, lay.wstruct, self.out[b], None, lay.ws,
                        stream=self.s_c)
        self.ev_used[b].record(self.s_c)
        with torch.cuda.stream(self.s_out):
            self.s_out.wait_event(self.ev_used[b])
            self.out_host.copy_(self.out[b], non_blocking=True)
            self.ev_read[b].record(self.s_out)
        self.used[b] = True


if __name__ == "__main__":
    sys.exit(main())
