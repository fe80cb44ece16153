#!/usr/bin/env python3
"""Benchmark of the ternary-weight linear layer on GB300.

Default workload: the 7B-shaped decode set (N,K) in {(4096,4096) q/k/v/o,
(11008,4096) gate/up, (4096,11008) down}, bf16 x, per-channel fp16 scales,
M in {1,4,8,16}, run as decode steps through a 32-layer stack whose every
layer has its own weights (1.62 GB of packed weights per M, far above the
129 MB L2, so no flush is needed).  One bench step = one decode pass at each
M (4 x 224 = 896 ternary_linear calls), captured once as a CUDA graph and
replayed.

Prints one JSON line (rank 0).  Under torchrun every rank runs its own replica
(the layer shards across GPUs only as independent replicas here; no
collective is on the data path): value = sum of ranks' work / max rank time.

  python bench.py [--gpus N] [--steps K] [--warmup W] [--workload decode7b]
  python bench.py --impl reference ...   # the CPU oracle on a bounded sample
"""
from __future__ import annotations

import argparse
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
from ternary_weight_linear_02_gb300.workloads import CONFIGS, algorithmic_bytes, flops, packed_bytes  # noqa: E402

METRIC = "packed-weight HBM GB/s and % of roofline per ternary_linear; µs/decode-step"
FALLBACK_PEAKS = {"hbm_gbs": 6800.0, "bf16_tflops": 1900.0, "bf16_tflops_sustained": 1700.0}


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


# ----------------------------------------------------------------------------- workload
class Stack:
    """Device-resident inputs of one config: per model layer, per projection,
    packed weights and scales; per M, x and out buffers for every call."""

    def __init__(self, cfg, Ms, dev):
        self.cfg, self.Ms, self.dev = cfg, Ms, dev
        self.w = []  # [depth][proj] -> (packed, scale)
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
        # per M: every call's x and out are slices of one flat buffer, so an
        # end-to-end step moves all of a pass's inputs / outputs in one copy each
        self.x, self.out, self.xflat, self.oflat = {}, {}, {}, {}
        for M in Ms:
            nx = sum(M * l.K for l in cfg.layers) * cfg.depth
            no = sum(M * l.N for l in cfg.layers) * cfg.depth
            self.xflat[M] = torch.empty(nx, dtype=cfg.x_dtype, device=dev)
            self.oflat[M] = torch.empty(no, dtype=cfg.x_dtype, device=dev)
            xs, outs, ox, oo = [], [], 0, 0
            for d in range(cfg.depth):
                xr, orow = [], []
                for l in cfg.layers:
                    xv = self.xflat[M][ox:ox + M * l.K].view(M, l.K)
                    xv.copy_(synth.activations(M, l.K, cfg.x_dtype,
                                               synth.seed_for(cfg.key, d, l.name, "x", M), dev))
                    xr.append(xv)
                    orow.append(self.oflat[M][oo:oo + M * l.N].view(M, l.N))
                    ox += M * l.K
                    oo += M * l.N
                xs.append(xr)
                outs.append(orow)
            self.x[M], self.out[M] = xs, outs

    def calls_per_step(self):
        return len(self.Ms) * self.cfg.depth * len(self.cfg.layers)

    def run_step(self, tl):
        cfg = self.cfg
        for M in self.Ms:
            for d in range(cfg.depth):
                for j, l in enumerate(cfg.layers):
                    packed, scale = self.w[d][j]
                    tl.linear(self.x[M][d][j], packed, scale, cfg.group_size,
                              out=self.out[M][d][j], static_weights=True)


class FusedStack:
    """The same weights in the fused layout a vLLM-style model runs: per layer
    one QKV call (q, k, v rows stacked), o, one gate/up call with the SiLU-gated
    product in its epilogue (ternary_linear_silu_mul), and down reading that
    product -- 4 calls per layer instead of 7, the same packed bytes."""

    NAMES = ("q", "k", "v", "o", "gate", "up", "down")

    def __init__(self, stack):
        cfg = stack.cfg
        names = [l.name for l in cfg.layers]
        self.ok = all(n in names for n in self.NAMES)
        if not self.ok:
            return
        ix = {n: i for i, n in enumerate(names)}
        self.cfg, self.stack = cfg, stack
        self.w = []
        for d in range(cfg.depth):
            w = stack.w[d]
            qkv = tuple(torch.cat([w[ix[n]][t] for n in "qkv"]) for t in (0, 1))
            gu = tuple(torch.cat([w[ix["gate"]][t], w[ix["up"]][t]]) for t in (0, 1))
            self.w.append((qkv, w[ix["o"]], gu, w[ix["down"]]))
        self.ix = ix
        self.bufs = {}
        for M in stack.Ms:
            layer = []
            for d in range(cfg.depth):
                qkv_n = self.w[d][0][0].shape[0]
                o_n = self.w[d][1][0].shape[0]
                h_n = self.w[d][2][0].shape[0] // 2
                dn_n = self.w[d][3][0].shape[0]
                layer.append(tuple(torch.empty((M, n), dtype=cfg.x_dtype, device=stack.dev)
                                   for n in (qkv_n, o_n, h_n, dn_n)))
            self.bufs[M] = layer

    def calls_per_layer(self):
        return 4

    def run_m(self, tl, M):
        cfg, st, ix = self.cfg, self.stack, self.ix
        for d in range(cfg.depth):
            (qkv, o, gu, dn), (y_qkv, y_o, h, y_dn) = self.w[d], self.bufs[M][d]
            gs = cfg.group_size
            tl.linear(st.x[M][d][ix["q"]], qkv[0], qkv[1], gs, out=y_qkv, static_weights=True)
            tl.linear(st.x[M][d][ix["o"]], o[0], o[1], gs, out=y_o, static_weights=True)
            tl.linear_silu_mul(st.x[M][d][ix["gate"]], gu[0], gu[1], gs, out=h, static_weights=True)
            tl.linear(h, dn[0], dn[1], gs, out=y_dn, static_weights=True)


def capture(fn, stream):
    g = torch.cuda.CUDAGraph()
    with torch.cuda.stream(stream):
        with torch.cuda.graph(g, stream=stream):
            fn()
    return g


def time_graph(g, stream, steps, warmup, barrier):
    with torch.cuda.stream(stream):
        for _ in range(warmup):
            g.replay()
    torch.cuda.synchronize()
    barrier()
    torch.cuda.synchronize()
    e0 = torch.cuda.Event(enable_timing=True)
    e1 = torch.cuda.Event(enable_timing=True)
    t0 = time.time()
    with torch.cuda.stream(stream):
        e0.record(stream)
        for _ in range(steps):
            g.replay()
        e1.record(stream)
    torch.cuda.synchronize()
    t1 = time.time()
    barrier()
    return e0.elapsed_time(e1), t0, t1


# ----------------------------------------------------------------------------- CPU oracle
def oracle_sample(cfg, Ms, budget_s: float, threads: int):
    """Time the CPU oracle, as it stands, on a bounded sample of the workload:
    for every distinct (N, K) projection shape and every M, the first R output
    rows (R = min(N, 256)), cycled until about budget_s seconds of work.
    Returns (packed-weight GB/s of the sample, description, seconds)."""
    import oracle
    oracle.build()
    shapes = []
    for l in cfg.layers:
        if (l.N, l.K) not in [(a, b) for a, b, _ in shapes]:
            shapes.append((l.N, l.K, l.name))
    name = "f16" if cfg.x_dtype == torch.float16 else "bf16"
    items = []
    for N, K, lname in shapes:
        rows = min(N, 256)
        p = synth.packed_codes(rows, K, synth.seed_for("cpu", N, K), "cpu").numpy()
        groups = 0 if cfg.group_size == 0 else K // cfg.group_size
        s = synth.scales(rows, groups, cfg.s_lo, cfg.s_hi, 1, "cpu")
        sb = s.view(torch.int16).numpy().view(np.uint16)
        for M in Ms:
            x = synth.activations(M, K, cfg.x_dtype, synth.seed_for("cpu", K, M), "cpu")
            xb = x.contiguous().view(torch.int16).numpy().view(np.uint16)
            items.append((xb, p, sb, rows * K // 4, f"{N}x{K}@M{M}[{rows} rows]"))
    done_bytes, spent, passes = 0, 0.0, 0
    while spent < budget_s or passes == 0:
        for xb, p, sb, nbytes, _ in items:
            t0 = time.perf_counter()
            oracle.linear_from_bits(xb, name, p, sb, cfg.group_size, threads)
            spent += time.perf_counter() - t0
            done_bytes += nbytes
        passes += 1
    gbs = done_bytes / spent / 1e9
    desc = (f"oracle fp64 C with {threads} threads on {len(items)} slices of {cfg.key} "
            f"({', '.join(i[4] for i in items)}), {passes} passes, {spent:.1f} s of CPU work; "
            "value = packed bytes of the slices / CPU time")
    return gbs, desc, spent


# ----------------------------------------------------------------------------- main
def main():
    ap = argparse.ArgumentParser()
    ap.add_argument("--gpus", type=int, default=1)
    ap.add_argument("--steps", type=int, default=1000)
    ap.add_argument("--warmup", type=int, default=10)
    ap.add_argument("--impl", default="ours", choices=["ours", "reference"])
    ap.add_argument("--workload", default="decode7b", choices=sorted(CONFIGS))
    ap.add_argument("--ms", default="", help="comma list restricting M values")
    ap.add_argument("--cpu-budget", type=float, default=12.0,
                    help="seconds of CPU oracle work for cpu_baseline")
    ap.add_argument("--no-cpu", action="store_true", help="skip the cpu_baseline leg")
    ap.add_argument("--no-e2e", action="store_true")
    ap.add_argument("--depth", type=int, default=0,
                    help="override the number of model layers (small cases for profiling)")
    ap.add_argument("--per-m-reps", type=int, default=0,
                    help="graph replays for each per-M timing (default: max(20, steps/4))")
    ap.add_argument("--comparator", action="store_true",
                    help="also time the same stack with weights dequantised once to bf16 "
                         "(t * scale) and torch.matmul (cuBLAS)")
    args = ap.parse_args()

    rank, world, local = dist_env()
    cfg = CONFIGS[args.workload]
    if args.depth > 0:
        import dataclasses
        cfg = dataclasses.replace(cfg, depth=args.depth)
    Ms = tuple(int(v) for v in args.ms.split(",")) if args.ms else cfg.Ms
    threads = os.cpu_count() or 1
    workload_name = (f"{cfg.key}: {cfg.title}; depth {cfg.depth}; "
                     + ", ".join(f"{l.name} {l.N}x{l.K}" for l in cfg.layers) + f"; M in {list(Ms)}")
    xdt = "bf16" if cfg.x_dtype == torch.bfloat16 else "f16"

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
        ms = statistics.median(s for _, s in vals) * 1e3
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

    stack = Stack(cfg, Ms, dev)
    torch.cuda.synchronize()
    # first call on the device outside capture (creates the status word)
    stack.run_step(tl)
    torch.cuda.synchronize()

    stream = torch.cuda.Stream(dev)
    stream.wait_stream(torch.cuda.current_stream(dev))
    g = capture(lambda: stack.run_step(tl), stream)

    clocks = ClockSampler(local)
    time.sleep(0.3)
    ms_total, t0, t1 = time_graph(g, stream, args.steps, args.warmup, barrier)
    clocks.window(t0, t1)
    clk = clocks.stop()
    ms_step = dist_util.max_over_ranks(ms_total / args.steps, dev)

    pb = packed_bytes(cfg) * len(Ms)
    ab = sum(algorithmic_bytes(cfg, M) for M in Ms)
    value = dist_util.job_throughput(pb, ms_step, world) / 1e9
    calls = stack.calls_per_step()
    pk, pk_src = peaks()
    peak = pk["hbm_gbs"]
    achieved = ab / (ms_step * 1e-3) / 1e9  # every launch of the step is the linear kernel
    per_m = {}
    for M in Ms:  # per-M decode-step time: time one M pass alone
        reps = args.per_m_reps if args.per_m_reps > 0 else max(20, args.steps // 4)
        gm = capture(lambda M=M: Stack.run_step(_OneM(stack, M), tl), stream)
        mt, _, _ = time_graph(gm, stream, reps, 3, lambda: None)
        mt /= reps
        per_m[str(M)] = {"us_per_decode_step": round(mt * 1e3, 2),
                         "packed_GBps": round(packed_bytes(cfg) / (mt * 1e-3) / 1e9, 1),
                         "frac_of_hbm": round(algorithmic_bytes(cfg, M) / (mt * 1e-3) / 1e9 / peak, 4),
                         "eff_TFLOPs": round(flops(cfg, M) / (mt * 1e-3) / 1e12, 2)}
        del gm

    # the same layers in the fused layout (QKV, o, gate/up + SiLU product, down)
    fused = None
    fs = FusedStack(stack)
    if fs.ok:
        fused = {"calls_per_layer": fs.calls_per_layer(),
                 "layout": "QKV stacked; gate/up stacked with silu(gate)*up in its epilogue "
                           "(ternary_linear_silu_mul); down reads that product",
                 "per_M": {}}
        for M in Ms:
            reps = args.per_m_reps if args.per_m_reps > 0 else max(20, args.steps // 4)
            gf = capture(lambda M=M: fs.run_m(tl, M), stream)
            ft, _, _ = time_graph(gf, stream, reps, 3, lambda: None)
            ft /= reps
            fused["per_M"][str(M)] = {
                "us_per_decode_step": round(ft * 1e3, 2),
                "packed_GBps": round(packed_bytes(cfg) / (ft * 1e-3) / 1e9, 1),
                "packed_frac_of_hbm": round(packed_bytes(cfg) / (ft * 1e-3) / 1e9 / peak, 4)}
            del gf
        del fs

    # end to end: pinned host x -> device, the calls, device out -> pinned host
    # (one copy per M pass in each direction: every call's x / out is a slice)
    e2e = None
    if not args.no_e2e:
        hx = {M: stack.xflat[M].cpu().pin_memory() for M in Ms}
        ho = {M: torch.empty(stack.oflat[M].shape, dtype=cfg.x_dtype).pin_memory() for M in Ms}
        h2d = sum(t.numel() * t.element_size() for t in hx.values())
        d2h = sum(t.numel() * t.element_size() for t in ho.values())

        def e2e_step():
            for M in Ms:
                stack.xflat[M].copy_(hx[M], non_blocking=True)
            stack.run_step(tl)
            for M in Ms:
                ho[M].copy_(stack.oflat[M], non_blocking=True)

        ge = capture(e2e_step, stream)
        e_ms, _, _ = time_graph(ge, stream, args.steps, args.warmup, barrier)
        e_step = dist_util.max_over_ranks(e_ms / args.steps, dev)
        e2e = {"value": dist_util.job_throughput(pb, e_step, world) / 1e9, "unit": "GB/s",
               "ms_per_step": e_step, "h2d_bytes_per_step": h2d, "d2h_bytes_per_step": d2h}
        del ge

    comparator = None
    if args.comparator:
        comparator = time_comparator(stack, tl, stream, Ms, args)

    # a kernel wait that gave up (bounded waits) leaves a non-zero status word:
    # the outputs of that call are not valid, so the line says so
    torch.cuda.synchronize()
    dev_status = tl.device_status(clear=True)
    if dev_status != 0:
        print(f"bench: device status {tl.status_string(dev_status)} after the timed runs", file=sys.stderr)

    cpu = None
    if rank == 0 and world == 1 and not args.no_cpu:
        v, desc, _ = oracle_sample(cfg, Ms, args.cpu_budget, threads)
        cpu = {"value": v, "unit": "GB/s", "cores": threads, "kind": "oracle", "sample": desc}

    traffic = read_traffic(cfg.key)
    line = {
        "metric": METRIC, "value": value, "unit": "GB/s", "n_gpus": world, "steps": args.steps,
        "warmup": args.warmup, "ms_per_step": ms_step, "higher_is_better": True,
        "scaling": "weak", "vs_baseline": None, "dtype": xdt, "data": "synthetic",
        "config": {"workload": workload_name, "Ms": list(Ms), "calls_per_step": calls,
                   "packed_bytes_per_step": pb, "algorithmic_bytes_per_step": ab,
                   "l2": "inputs larger than L2: distinct per-layer weights, "
                         f"{packed_bytes(cfg) / 1e9:.2f} GB packed per M pass",
                   "per_M": per_m, "fused_layout": fused, "peaks_source": pk_src},
        "roofline": {"bound": "hbm", "achieved": achieved, "peak": peak, "unit": "GB/s",
                     "frac": achieved / peak, "traffic": traffic,
                     "kernel": "ternary_linear kernels (every launch of the step)",
                     "peak_note": f"hbm_gbs of {pk_src} peaks"},
        "cpu_baseline": cpu,
        "e2e": e2e,
        "gpu_launches": calls * args.steps,
        "comparator": comparator,
        "clocks": clk,
        "device_status": tl.status_string(dev_status),
    }
    if rank == 0:
        print(json.dumps(line), flush=True)
    if world > 1:
        import torch.distributed as dist
        dist.destroy_process_group()
    return 0


def time_comparator(stack, tl, stream, Ms, args):
    """The same decode stack with each layer's weights dequantised once to bf16
    (t from ternary_unpack, times the scale) and run with torch.matmul (cuBLAS):
    the dequantise-at-load route the pages compare against.  Reported as the same
    packed-weight GB/s (packed bytes of the step / step time) for comparison."""
    cfg = stack.cfg
    W = []
    for d in range(cfg.depth):
        row = []
        for j, l in enumerate(cfg.layers):
            packed, scale = stack.w[d][j]
            t, _ = tl.unpack(packed)
            if cfg.group_size == 0:
                w = t.to(torch.float32) * scale.to(torch.float32)[:, None]
            else:
                w = (t.to(torch.float32).view(l.N, -1, cfg.group_size)
                     * scale.to(torch.float32)[:, :, None]).view(l.N, l.K)
            row.append(w.to(cfg.x_dtype))
            del t, w
        W.append(row)
    torch.cuda.synchronize()
    res = {"kind": "weights dequantised once to " + ("bf16" if cfg.x_dtype == torch.bfloat16 else "fp16")
           + " (t * scale) + torch.matmul (cuBLAS), same stack and inputs", "unit": "GB/s", "per_M": {}}
    tot_ms = 0.0
    for M in Ms:
        def step(M=M):
            for d in range(cfg.depth):
                for j in range(len(cfg.layers)):
                    torch.matmul(stack.x[M][d][j], W[d][j].t(), out=stack.out[M][d][j])
        step()
        g = capture(step, stream)
        reps = args.per_m_reps if args.per_m_reps > 0 else max(20, args.steps // 4)
        mt, _, _ = time_graph(g, stream, reps, 3, lambda: None)
        mt /= reps
        tot_ms += mt
        res["per_M"][str(M)] = {"us_per_decode_step": round(mt * 1e3, 2),
                                "packed_GBps": round(packed_bytes(cfg) / (mt * 1e-3) / 1e9, 1),
                                "bf16_weight_GBps": round(packed_bytes(cfg) * 8 / (mt * 1e-3) / 1e9, 1)}
        del g
    res["value"] = packed_bytes(cfg) * len(Ms) / (tot_ms * 1e-3) / 1e9
    del W
    torch.cuda.empty_cache()
    return res


class _OneM:
    """A view of a Stack restricted to one M (for the per-M timings)."""

    def __init__(self, stack, M):
        self.cfg, self.Ms, self.w, self.x, self.out = stack.cfg, (M,), stack.w, stack.x, stack.out


def read_traffic(key):
    """Per-launch DRAM traffic from the committed ncu summary for this
    workload, if its kernel fingerprint matches the current sources."""
    path = os.path.join(ROOT, "profiles", f"traffic_{key}.txt")
    if not os.path.exists(path):
        return None
    want = None
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
