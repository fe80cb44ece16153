#!/usr/bin/env python3
"""Benchmark of the ternary-weight linear layer on GB300.

Default workload (``stack7b``): the 7B-shaped 28-layer stack in the fused
layout -- per model layer one fused QKV call (N = 3584 + 512 + 512, K = 3584),
o (3584 x 3584), the fused gate/up call (2 x 18944 rows, K = 3584) with the
SiLU-gated product in its epilogue, and down (3584 x 18944) reading that
product -- bf16 x, per-channel fp16 scales.  One bench step is one pass of the
stack at every M in {1, 16, 64, 256, 2048} (5 x 112 calls), each pass captured
as a CUDA graph and replayed; the stack's per-layer weights are distinct
(1.63 GB packed per pass, far above the 129 MB L2, so no flush is needed).
The other four workloads are timed after the step and reported per M in
``config.configs``.

Prints one JSON line (rank 0).  Under torchrun every rank runs its own replica
(no collective on the data path): value = sum of ranks' work / max rank time.

  python bench.py [--gpus N] [--steps K] [--warmup W] [--workload stack7b]
  python bench.py --impl reference ...   # the CPU oracle on a bounded sample
"""
from __future__ import annotations

import argparse
import dataclasses
import json
import os
import statistics
import subprocess
import sys
import threading
import time

import numpy as np
import torch

ROOT = os.path.dirname(os.path.abspath(__file__))
sys.path.insert(0, ROOT)

from ternary_weight_linear_02_gb300 import dist_util, synth  # noqa: E402
from ternary_weight_linear_02_gb300.workloads import (CONFIGS, algorithmic_bytes, flops,  # noqa: E402
                                                      layer_calls, out_cols, packed_bytes)

METRIC = "packed-weight HBM GB/s and % of roofline per ternary_linear; µs/decode-step"
FALLBACK_PEAKS = {"hbm_gbs": 6800.0, "bf16_tflops": 1900.0, "bf16_tflops_sustained": 1700.0}
SUB_CONFIGS = ("linear1k", "decode7b", "embed06b", "layers27b")


# ----------------------------------------------------------------------------- helpers
def dist_env():
    rank = int(os.environ.get("RANK", "0"))
    world = int(os.environ.get("WORLD_SIZE", "1"))
    local = int(os.environ.get("LOCAL_RANK", str(rank)))
    return rank, world, local


def peaks():
    p = os.path.join(ROOT, "MEASURED_PEAKS.json")
    if os.path.exists(p):
        with open(p) as f:
            d = json.load(f)
        return d, "measured"
    return dict(FALLBACK_PEAKS), "fallback"


class ClockSampler:
    """nvidia-smi clock / throttle samples, kept only inside [t0, t1]."""

    FIELDS = ("index,clocks.sm,clocks.max.sm,power.draw,clocks_event_reasons.active,"
              "clocks_event_reasons.hw_slowdown,clocks_event_reasons.hw_thermal_slowdown,"
              "clocks_event_reasons.sw_thermal_slowdown,clocks_event_reasons.sw_power_cap")

    def __init__(self, gpu_index: int):
        self.samples = []
        self.t0 = self.t1 = None
        try:
            self.proc = subprocess.Popen(
                ["nvidia-smi", f"--query-gpu={self.FIELDS}", "--format=csv,noheader,nounits",
                 "-lms", "100", "-i", str(gpu_index)],
                stdout=subprocess.PIPE, stderr=subprocess.DEVNULL, text=True)
        except Exception:
            self.proc = None
            return
        self.th = threading.Thread(target=self._read, daemon=True)
        self.th.start()

    def _read(self):
        for line in self.proc.stdout:
            self.samples.append((time.time(), line.strip()))

    def window(self, t0, t1):
        self.t0, self.t1 = t0, t1

    def stop(self):
        if self.proc is None:
            return None
        time.sleep(0.25)
        self.proc.terminate()
        try:
            self.proc.wait(timeout=5)
        except Exception:
            self.proc.kill()
        rows = [s for (t, s) in self.samples if self.t0 is not None and self.t0 <= t <= self.t1 + 0.15]
        sm, smax, reasons = [], None, set()
        names = ["hw_slowdown", "hw_thermal_slowdown", "sw_thermal_slowdown", "sw_power_cap"]
        for r in rows:
            f = [c.strip() for c in r.split(",")]
            if len(f) < 9:
                continue
            try:
                sm.append(float(f[1]))
                smax = float(f[2])
            except ValueError:
                continue
            for name, v in zip(names, f[5:9]):
                if v.lower() == "active":
                    reasons.add(name)
        return {"sm_mhz": statistics.median(sm) if sm else None, "sm_max_mhz": smax,
                "reasons": sorted(reasons), "samples": len(sm)}


def bench_config(key: str, depth: int = 0):
    """The config as benchmarked: its depth times its weight rotation (so one
    pass streams more than twice the L2), or an explicit depth."""
    cfg = CONFIGS[key]
    return dataclasses.replace(cfg, depth=depth if depth > 0 else cfg.depth * cfg.rotate)


# ----------------------------------------------------------------------------- workload
class Workload:
    """Device-resident inputs of one config: per model layer, per projection,
    packed weights and scales; per M, every call's input and output buffer.
    The independent inputs of one M pass are slices of one flat buffer and so are
    the outputs, so an end-to-end step moves them in one copy each way."""

    def __init__(self, cfg, Ms, dev):
        self.cfg, self.Ms, self.dev = cfg, tuple(Ms), dev
        self.calls = layer_calls(cfg)
        self.w = []  # [depth][layer] -> (packed, scale)
        for d in range(cfg.depth):
            row = []
            for l in cfg.layers:
                packed = synth.packed_codes(l.N, l.K, synth.seed_for(cfg.key, d, l.name, "w"), dev,
                                            cfg.p_reserved)
                groups = 0 if cfg.group_size == 0 else l.K // cfg.group_size
                scale = synth.scales(l.N, groups, cfg.s_lo, cfg.s_hi,
                                     synth.seed_for(cfg.key, d, l.name, "s"), dev)
                row.append((packed, scale))
            self.w.append(row)
        self.xflat, self.oflat, self.x, self.y = {}, {}, {}, {}
        for M in self.Ms:
            nx = cfg.depth * sum(M * cfg.layers[c.layer].K for c in self.calls if c.src < 0)
            no = cfg.depth * sum(M * out_cols(cfg, c) for c in self.calls)
            self.xflat[M] = torch.empty(nx, dtype=cfg.x_dtype, device=dev)
            self.oflat[M] = torch.empty(no, dtype=cfg.x_dtype, device=dev)
            xs, ys, ox, oo = [], [], 0, 0
            for d in range(cfg.depth):
                xr, yr = [], []
                for j, c in enumerate(self.calls):
                    l = cfg.layers[c.layer]
                    n = out_cols(cfg, c)
                    yr.append(self.oflat[M][oo:oo + M * n].view(M, n))
                    oo += M * n
                    if c.src < 0:
                        xv = self.xflat[M][ox:ox + M * l.K].view(M, l.K)
                        xv.copy_(synth.activations(M, l.K, cfg.x_dtype,
                                                   synth.seed_for(cfg.key, d, l.name, j, "x", M), dev))
                        ox += M * l.K
                        xr.append(xv)
                    else:
                        xr.append(yr[c.src])
                xs.append(xr)
                ys.append(yr)
            self.x[M], self.y[M] = xs, ys

    def run(self, tl, M, masks=None):
        """One pass of the stack at M tokens (every call with static weights);
        masks[d][layer]: zero-block maps to skip zero blocks with."""
        cfg = self.cfg
        for d in range(cfg.depth):
            for j, c in enumerate(self.calls):
                packed, scale = self.w[d][c.layer]
                kw = {} if masks is None else {"mask": masks[d][c.layer]}
                if c.kind == "silu_mul":
                    tl.linear_silu_mul(self.x[M][d][j], packed, scale, cfg.group_size,
                                       out=self.y[M][d][j], static_weights=True, **kw)
                else:
                    tl.linear(self.x[M][d][j], packed, scale, cfg.group_size,
                              out=self.y[M][d][j], static_weights=True, **kw)

    def calls_per_pass(self):
        return self.cfg.depth * len(self.calls)


def capture(fn, stream):
    g = torch.cuda.CUDAGraph()
    with torch.cuda.stream(stream):
        with torch.cuda.graph(g, stream=stream):
            fn()
    return g


def time_passes(graphs, stream, steps, warmup, barrier):
    """Replay the graphs in order `steps` times; CUDA events between graphs on the
    launching stream.  Returns (total ms, per-graph ms, wall t0, wall t1)."""
    with torch.cuda.stream(stream):
        for _ in range(warmup):
            for g in graphs:
                g.replay()
    torch.cuda.synchronize()
    barrier()
    torch.cuda.synchronize()
    ev = [[torch.cuda.Event(enable_timing=True) for _ in range(len(graphs) + 1)]
          for _ in range(steps)]
    t0 = time.time()
    with torch.cuda.stream(stream):
        for s in range(steps):
            ev[s][0].record(stream)
            for i, g in enumerate(graphs):
                g.replay()
                ev[s][i + 1].record(stream)
    torch.cuda.synchronize()
    t1 = time.time()
    barrier()
    per = [sum(ev[s][i].elapsed_time(ev[s][i + 1]) for s in range(steps)) for i in range(len(graphs))]
    return sum(per), per, t0, t1


def bound_of(M):
    return "hbm" if M <= 32 else ("tensor" if M >= 256 else "hbm+tensor")


def per_m_entry(cfg, M, ms, pk, calls):
    """Per-M figures of one pass that took `ms` milliseconds."""
    t = ms * 1e-3
    ab = algorithmic_bytes(cfg, M)
    fl = flops(cfg, M)
    e = {"us_per_pass": round(ms * 1e3, 2), "us_per_call": round(ms * 1e3 / calls, 3),
         "packed_GBps": round(packed_bytes(cfg) / t / 1e9, 1),
         "algorithmic_GBps": round(ab / t / 1e9, 1),
         "frac_of_hbm": round(ab / t / 1e9 / pk["hbm_gbs"], 4),
         "eff_TFLOPs": round(fl / t / 1e12, 2),
         "frac_of_bf16_burst": round(fl / t / 1e12 / pk["bf16_tflops"], 4),
         "frac_of_bf16_sustained": round(fl / t / 1e12 / pk["bf16_tflops_sustained"], 4),
         "bound": bound_of(M)}
    return e


def kernel_of(M):
    """The kernel family the automatic dispatch runs at M (K % 64 == 0)."""
    if M <= 8:
        return "decode kernel (warp MMAs, TMA-staged weights) and tcgen05 skinny kernel, per layer"
    if M <= 32:
        return "tcgen05 skinny kernel"
    return "tcgen05 tile kernel"


def roofline_of(cfg, M, ms, pk, pk_src, traffic):
    """The roofline object for the pass at M: every launch of one pass is the same
    kernel family, so per-launch work / average launch time = pass work / pass time."""
    t = ms * 1e-3
    calls = cfg.depth * len(layer_calls(cfg))
    if bound_of(M) == "tensor":
        ach = flops(cfg, M) / t / 1e12
        peak = pk["bf16_tflops"]
        return {"bound": "tensor", "achieved": ach, "peak": peak, "unit": "TFLOP/s",
                "frac": ach / peak, "traffic": traffic, "M": M,
                "kernel": f"{kernel_of(M)}, every launch of the M={M} pass ({calls} launches)",
                "peak_note": f"bf16_tflops (burst) of {pk_src} peaks; "
                             f"{ach / pk['bf16_tflops_sustained']:.3f} of the sustained figure"}
    ach = algorithmic_bytes(cfg, M) / t / 1e9
    peak = pk["hbm_gbs"]
    return {"bound": "hbm", "achieved": ach, "peak": peak, "unit": "GB/s", "frac": ach / peak,
            "traffic": traffic, "M": M,
            "kernel": f"{kernel_of(M)}, every launch of the M={M} pass ({calls} launches)",
            "peak_note": f"hbm_gbs of {pk_src} peaks"}


# ----------------------------------------------------------------------------- CPU oracle
def oracle_sample(cfg, Ms, budget_s: float, threads: int):
    """Time the CPU oracle, as it stands, on a bounded sample of the workload: for
    every call of one model layer and every M, the first R output rows
    (R = 256 for M <= 16, fewer for larger M so the sample stays bounded), cycled
    until about budget_s seconds of work.  Returns (estimated packed-weight GB/s of
    the whole pass set, description, seconds): the sampled time per row is scaled
    to every row of every layer of the stack."""
    import oracle
    oracle.build()
    name = "f16" if cfg.x_dtype == torch.float16 else "bf16"
    items = []
    for j, c in enumerate(layer_calls(cfg)):
        l = cfg.layers[c.layer]
        for M in Ms:
            rows = min(l.N, max(8, 256 * 16 // max(M, 16)))
            if c.kind == "silu_mul":  # rows pairs: gate rows then the matching up rows
                rows = 2 * min(l.N // 2, max(4, rows // 2))
            p = synth.packed_codes(rows, l.K, synth.seed_for("cpu", l.name, l.K), "cpu").numpy()
            groups = 0 if cfg.group_size == 0 else l.K // cfg.group_size
            s = synth.scales(rows, groups, cfg.s_lo, cfg.s_hi, 1, "cpu")
            sb = s.view(torch.int16).numpy().view(np.uint16)
            x = synth.activations(M, l.K, cfg.x_dtype, synth.seed_for("cpu", l.K, M), "cpu")
            xb = x.contiguous().view(torch.int16).numpy().view(np.uint16)
            # share of the call this sample stands for: weight rows sampled / rows of the call
            frac = rows / l.N
            items.append((c.kind, xb, p, sb, frac, l, M, f"{l.name}@M{M}[{rows} rows]"))
    spent = {i: 0.0 for i in range(len(items))}
    runs = {i: 0 for i in range(len(items))}
    total, passes = 0.0, 0
    while total < budget_s or passes == 0:
        for i, (kind, xb, p, sb, frac, l, M, _) in enumerate(items):
            t0 = time.perf_counter()
            if kind == "silu_mul":
                oracle.silu_mul_from_bits(xb, name, p, sb, cfg.group_size, threads)
            else:
                oracle.linear_from_bits(xb, name, p, sb, cfg.group_size, threads)
            dt = time.perf_counter() - t0
            spent[i] += dt
            runs[i] += 1
            total += dt
        passes += 1
    # estimated CPU seconds of one pass at each M = depth * sum over calls (time / frac)
    est = 0.0
    for i, (_, _, _, _, frac, _, _, _) in enumerate(items):
        est += cfg.depth * (spent[i] / runs[i]) / frac
    gbs = packed_bytes(cfg) * len(Ms) / est / 1e9
    desc = (f"oracle fp64 C with {threads} thread(s) on {len(items)} row slices of {cfg.key} "
            f"({', '.join(i[7] for i in items)}), {passes} passes, {total:.1f} s of CPU work; "
            f"per-row time scaled to the full {cfg.depth}-layer pass at each M "
            "(extrapolated); value = packed bytes of the step / estimated CPU time")
    return gbs, desc, total


# ----------------------------------------------------------------------------- comparators
def time_comparators(wl, tl, stream, reps):
    """The same stack and inputs on the pages' route 1, with cuBLAS (torch.matmul)
    doing the product: (a) weights dequantised once to the activation dtype at load
    (t * scale), (b) dequantised on the fly every call (ternary_unpack, then t * scale
    in torch, then the matmul).  The gated gate/up call forms silu(g) * u with torch
    after its matmul.  Reported as the same packed-weight GB/s for comparison."""
    cfg = wl.cfg
    dt = cfg.x_dtype

    def dequant(packed, scale, l):
        t, _ = tl.unpack(packed)
        if cfg.group_size == 0:
            w = t.to(torch.float32) * scale.to(torch.float32)[:, None]
        else:
            w = (t.to(torch.float32).view(l.N, -1, cfg.group_size)
                 * scale.to(torch.float32)[:, :, None]).view(l.N, l.K)
        return w.to(dt)

    def product(x, w, c, out):
        if c.kind == "silu_mul":
            y = torch.matmul(x, w.t())
            n = y.shape[1] // 2
            torch.mul(torch.nn.functional.silu(y[:, :n]), y[:, n:], out=out)
        else:
            torch.matmul(x, w.t(), out=out)

    res = {}
    # (a) dequantise once at load
    W = [[dequant(p, s, cfg.layers[i]) for i, (p, s) in enumerate(row)] for row in wl.w]
    torch.cuda.synchronize()
    per = {}
    for M in wl.Ms:
        def step(M=M):
            for d in range(cfg.depth):
                for j, c in enumerate(wl.calls):
                    product(wl.x[M][d][j], W[d][c.layer], c, wl.y[M][d][j])
        step()
        g = capture(step, stream)
        _, pm, _, _ = time_passes([g], stream, reps, 2, lambda: None)
        per[str(M)] = per_m_brief(cfg, M, pm[0] / reps)
        del g
    res["dequant_at_load"] = {"kind": f"weights dequantised once to {dt_name(dt)} (t * scale), "
                                      "torch.matmul (cuBLAS)", "per_M": per}
    del W
    torch.cuda.synchronize()
    torch.cuda.empty_cache()
    # (b) dequantise on the fly, every call
    per = {}
    for M in wl.Ms:
        def step(M=M):
            for d in range(cfg.depth):
                for j, c in enumerate(wl.calls):
                    p, s = wl.w[d][c.layer]
                    product(wl.x[M][d][j], dequant(p, s, cfg.layers[c.layer]), c, wl.y[M][d][j])
        step()
        g = capture(step, stream)
        _, pm, _, _ = time_passes([g], stream, reps, 2, lambda: None)
        per[str(M)] = per_m_brief(cfg, M, pm[0] / reps)
        del g
        torch.cuda.empty_cache()
    res["dequant_on_the_fly"] = {"kind": "every call: ternary_unpack to int8, t * scale in torch to "
                                         f"{dt_name(dt)}, torch.matmul (cuBLAS)", "per_M": per}
    return res


def time_sparse(tl, stream, dev, reps, p_zero=0.3, Ms=(1, 16, 256)):
    """Zero-block skipping on block-sparse weights: the 7B stack's layer shapes
    (6 model layers, 350 MB packed) with each 128-row x 64-k block zeroed with
    probability p_zero, timed without and with the zero-block maps."""
    cfg = bench_config("stack7b", depth=6)
    wl = Workload(cfg, Ms, dev)
    for d in range(cfg.depth):
        for i, (p, sc) in enumerate(wl.w[d]):
            wl.w[d][i] = (synth.block_sparse(p, p_zero, synth.seed_for("sparse", d, i) & 0xFFFFFFFF), sc)
    masks, zero, total = [], 0, 0
    for row in wl.w:
        mrow = []
        for p, _ in row:
            m, z = tl.block_mask(p)
            mrow.append(m)
            zero += int(z.item())
            total += ((p.shape[0] + 127) // 128) * ((p.shape[1] * 4 + 63) // 64)
        masks.append(mrow)
    for M in Ms:
        wl.run(tl, M)
        wl.run(tl, M, masks)
    torch.cuda.synchronize()
    out = {"workload": describe(cfg, Ms), "zero_block_fraction": round(zero / max(total, 1), 4),
           "block": "128 rows x 64 k", "per_M": {}}
    for M in Ms:
        gd = capture(lambda M=M: wl.run(tl, M), stream)
        gm = capture(lambda M=M: wl.run(tl, M, masks), stream)
        _, per, _, _ = time_passes([gd, gm], stream, reps, 3, lambda: None)
        out["per_M"][str(M)] = {"dense_us": round(per[0] / reps * 1e3, 2),
                                "masked_us": round(per[1] / reps * 1e3, 2),
                                "speedup": round(per[0] / per[1], 3)}
        del gd, gm
    del wl, masks
    torch.cuda.synchronize()
    torch.cuda.empty_cache()
    return out


def per_m_brief(cfg, M, ms):
    t = ms * 1e-3
    return {"us_per_pass": round(ms * 1e3, 2), "packed_GBps": round(packed_bytes(cfg) / t / 1e9, 1),
            "eff_TFLOPs": round(flops(cfg, M) / t / 1e12, 2)}


def dt_name(dt):
    return "bf16" if dt == torch.bfloat16 else "f16"


def time_config(key, tl, stream, dev, reps, pk, pk_src):
    """Compact per-M figures of one config (its own stack, rotated past the L2)."""
    cfg = bench_config(key)
    wl = Workload(cfg, cfg.Ms, dev)
    for M in cfg.Ms:
        wl.run(tl, M)
    torch.cuda.synchronize()
    graphs = [capture(lambda M=M: wl.run(tl, M), stream) for M in cfg.Ms]
    _, per, _, _ = time_passes(graphs, stream, reps, 3, lambda: None)
    calls = wl.calls_per_pass()
    out = {"workload": describe(cfg, cfg.Ms), "calls_per_pass": calls, "reps": reps, "per_M": {}}
    for M, ms in zip(cfg.Ms, per):
        e = per_m_entry(cfg, M, ms / reps, pk, calls)
        out["per_M"][str(M)] = e
    del graphs, wl
    torch.cuda.synchronize()
    torch.cuda.empty_cache()
    return out


def describe(cfg, Ms):
    calls = layer_calls(cfg)
    parts = []
    for c in calls:
        l = cfg.layers[c.layer]
        tag = "silu(gate)*up of " if c.kind == "silu_mul" else ""
        src = f" <- call {c.src}" if c.src >= 0 else ""
        parts.append(f"{tag}{l.name} {l.N}x{l.K}{src}")
    return (f"{cfg.key}: {cfg.title}; {cfg.depth} model layers (distinct weights); per layer "
            + ", ".join(parts) + f"; M in {list(Ms)}; {dt_name(cfg.x_dtype)} x; "
            + ("per-channel" if cfg.group_size == 0 else f"group-{cfg.group_size}") + " fp16 scales")


# ----------------------------------------------------------------------------- main
def main():
    ap = argparse.ArgumentParser()
    ap.add_argument("--gpus", type=int, default=1)
    ap.add_argument("--steps", type=int, default=20)
    ap.add_argument("--warmup", type=int, default=5)
    ap.add_argument("--impl", default="ours", choices=["ours", "reference"])
    ap.add_argument("--workload", default="stack7b", choices=sorted(CONFIGS))
    ap.add_argument("--ms", default="", help="comma list restricting M values")
    ap.add_argument("--cpu-budget", type=float, default=12.0,
                    help="seconds of CPU oracle work for cpu_baseline (all threads)")
    ap.add_argument("--no-cpu", action="store_true", help="skip the cpu_baseline leg")
    ap.add_argument("--no-e2e", action="store_true")
    ap.add_argument("--no-configs", action="store_true", help="skip the other configs' figures")
    ap.add_argument("--no-comparator", action="store_true", help="skip the cuBLAS comparators")
    ap.add_argument("--depth", type=int, default=0,
                    help="override the number of model layers (small cases for profiling)")
    ap.add_argument("--reps", type=int, default=0,
                    help="replays per pass for the other configs and comparators (default 10)")
    args = ap.parse_args()

    rank, world, local = dist_env()
    cfg = bench_config(args.workload, args.depth)
    Ms = tuple(int(v) for v in args.ms.split(",")) if args.ms else cfg.Ms
    threads = os.cpu_count() or 1
    workload_name = describe(cfg, Ms)
    pk, pk_src = peaks()

    if args.impl == "reference":
        if rank != 0:
            return 0
        # the oracle, as it stands, on a bounded sample per step
        per_step = max(1.0, min(20.0, 150.0 / max(1, args.steps + args.warmup)))
        vals = []
        for i in range(args.warmup + args.steps):
            v, desc, spent = oracle_sample(cfg, Ms, per_step, threads)
            if i >= args.warmup:
                vals.append((v, spent))
        value = statistics.median(v for v, _ in vals)
        ms = packed_bytes(cfg) * len(Ms) / (value * 1e9) * 1e3
        line = {"impl": "reference", "metric": METRIC, "value": value, "unit": "GB/s",
                "n_gpus": args.gpus, "steps": args.steps, "warmup": args.warmup,
                "ms_per_step": ms, "higher_is_better": True, "scaling": "weak",
                "vs_baseline": None, "dtype": "f64", "data": "synthetic",
                "config": {"workload": workload_name, "sample": desc},
                "cpu_baseline": {"value": value, "unit": "GB/s", "cores": threads, "kind": "oracle",
                                 "sample": desc},
                "e2e": {"value": value, "unit": "GB/s", "h2d_bytes_per_step": 0,
                        "d2h_bytes_per_step": 0}}
        print(json.dumps(line), flush=True)
        return 0

    import ternary_weight_linear_02_gb300 as tl
    if world > 1:
        import torch.distributed as dist
        dist.init_process_group("nccl", device_id=torch.device("cuda", local))
        barrier = lambda: dist.barrier()  # noqa: E731
    else:
        barrier = lambda: None  # noqa: E731
    torch.cuda.set_device(local)
    dev = torch.device("cuda", local)
    tl.build()
    tl.load()

    wl = Workload(cfg, Ms, dev)
    torch.cuda.synchronize()
    for M in Ms:  # first calls on the device outside capture (create the status word)
        wl.run(tl, M)
    torch.cuda.synchronize()

    stream = torch.cuda.Stream(dev)
    stream.wait_stream(torch.cuda.current_stream(dev))
    graphs = [capture(lambda M=M: wl.run(tl, M), stream) for M in Ms]

    clocks = ClockSampler(local)
    time.sleep(0.3)
    ms_total, per_ms, t0, t1 = time_passes(graphs, stream, args.steps, args.warmup, barrier)
    clocks.window(t0, t1)
    clk = clocks.stop()
    ms_step = dist_util.max_over_ranks(ms_total / args.steps, dev)

    pb = packed_bytes(cfg) * len(Ms)
    value = dist_util.job_throughput(pb, ms_step, world) / 1e9
    calls = wl.calls_per_pass()
    per_m = {str(M): per_m_entry(cfg, M, ms / args.steps, pk, calls) for M, ms in zip(Ms, per_ms)}
    traffic = read_traffic(cfg.key)
    # the dominant kernel: the pass with the largest share of the step
    dom = max(range(len(Ms)), key=lambda i: per_ms[i])
    roofline = roofline_of(cfg, Ms[dom], per_ms[dom] / args.steps, pk, pk_src, traffic)
    roofline["share_of_step"] = round(per_ms[dom] / ms_total, 4)
    per_m_roof = {str(M): roofline_of(cfg, M, ms / args.steps, pk, pk_src, None)
                  for M, ms in zip(Ms, per_ms)}
    decode_us = {str(M): per_m[str(M)]["us_per_pass"] for M in Ms if M <= 32}

    # end to end: pinned host inputs -> device, the pass, device outputs -> pinned host
    # (one copy each way per M pass: every call's own input / output is a slice)
    e2e = None
    if not args.no_e2e:
        hx = {M: wl.xflat[M].cpu().pin_memory() for M in Ms}
        ho = {M: torch.empty(wl.oflat[M].shape, dtype=cfg.x_dtype).pin_memory() for M in Ms}
        h2d = sum(t.numel() * t.element_size() for t in hx.values())
        d2h = sum(t.numel() * t.element_size() for t in ho.values())

        def e2e_pass(M):
            wl.xflat[M].copy_(hx[M], non_blocking=True)
            wl.run(tl, M)
            ho[M].copy_(wl.oflat[M], non_blocking=True)

        ge = [capture(lambda M=M: e2e_pass(M), stream) for M in Ms]
        e_ms, _, _, _ = time_passes(ge, stream, args.steps, args.warmup, barrier)
        e_step = dist_util.max_over_ranks(e_ms / args.steps, dev)
        e2e = {"value": dist_util.job_throughput(pb, e_step, world) / 1e9, "unit": "GB/s",
               "ms_per_step": e_step, "h2d_bytes_per_step": h2d, "d2h_bytes_per_step": d2h,
               "path": "ternary_weight_linear_02_gb300.linear / linear_silu_mul (C ABI through "
                       "ctypes), pinned host inputs copied in and outputs copied out in the "
                       "timed region"}
        del ge

    reps = args.reps if args.reps > 0 else 10
    comparator = None
    if not args.no_comparator and world == 1:
        comparator = time_comparators(wl, tl, stream, max(3, reps // 2))

    # a kernel wait that gave up (bounded waits) leaves a non-zero status word:
    # the outputs of that call are not valid, so the line says so
    torch.cuda.synchronize()
    dev_status = tl.device_status(clear=True)
    if dev_status != 0:
        print(f"bench: device status {tl.status_string(dev_status)} after the timed runs",
              file=sys.stderr)
    del graphs, wl
    torch.cuda.synchronize()
    torch.cuda.empty_cache()

    configs = None
    if not args.no_configs and args.workload == "stack7b" and not args.depth:
        configs = {k: time_config(k, tl, stream, dev, reps, pk, pk_src) for k in SUB_CONFIGS}
        st2 = tl.device_status(clear=True)
        if st2 != 0:
            print(f"bench: device status {tl.status_string(st2)} after the other configs",
                  file=sys.stderr)
            dev_status = dev_status or st2

    sparse = None
    if not args.no_configs and args.workload == "stack7b" and not args.depth and world == 1:
        sparse = time_sparse(tl, stream, dev, reps)

    cpu = None
    if rank == 0 and world == 1 and not args.no_cpu:
        v, desc, _ = oracle_sample(cfg, Ms, args.cpu_budget, threads)
        v1, desc1, _ = oracle_sample(cfg, Ms, args.cpu_budget / 2, 1)
        cpu = {"value": v, "unit": "GB/s", "cores": threads, "kind": "oracle", "sample": desc,
               "single_thread": {"value": v1, "unit": "GB/s", "cores": 1, "sample": desc1}}

    line = {
        "metric": METRIC, "value": value, "unit": "GB/s", "n_gpus": world, "steps": args.steps,
        "warmup": args.warmup, "ms_per_step": ms_step, "higher_is_better": True,
        "scaling": "weak", "vs_baseline": None, "dtype": dt_name(cfg.x_dtype), "data": "synthetic",
        "config": {"workload": workload_name, "Ms": list(Ms), "calls_per_step": calls * len(Ms),
                   "packed_bytes_per_step": pb,
                   "algorithmic_bytes_per_step": sum(algorithmic_bytes(cfg, M) for M in Ms),
                   "l2": "inputs larger than L2: distinct per-layer weights, "
                         f"{packed_bytes(cfg) / 1e9:.2f} GB packed per pass",
                   "us_per_decode_step": decode_us,
                   "per_M": per_m, "roofline_per_M": per_m_roof, "peaks_source": pk_src,
                   "configs": configs},
        "roofline": roofline,
        "cpu_baseline": cpu,
        "e2e": e2e,
        "gpu_launches": calls * len(Ms) * args.steps,
        "comparator": comparator,
        "sparse_skip": sparse,
        "clocks": clk,
        "device_status": tl.status_string(dev_status),
    }
    if rank == 0:
        print(json.dumps(line), flush=True)
    if world > 1:
        import torch.distributed as dist
        dist.destroy_process_group()
    return 0


def read_traffic(key):
    """Per-launch DRAM traffic from the committed ncu summary for this
    workload, if its kernel fingerprint matches the current sources."""
    path = os.path.join(ROOT, "profiles", f"traffic_{key}.txt")
    if not os.path.exists(path):
        return None
    vals = {}
    for line in open(path):
        if ":" in line and not line.startswith("#"):
            k, v = line.split(":", 1)
            vals[k.strip()] = v.strip()
    try:
        from ternary_weight_linear_02_gb300 import _build
        want = _build._fingerprint()[:16]
    except Exception:
        return None
    if vals.get("kernel_fingerprint") != want:
        return None
    try:
        return float(vals["dram_bytes_per_launch"])
    except (KeyError, ValueError):
        return None


if __name__ == "__main__":
    sys.exit(main())
