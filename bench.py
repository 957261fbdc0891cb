#!/usr/bin/env python3
"""Benchmark of the top-k MoE layer forward on B300.

One step = one pass of the whole layer over one batch: router GEMM + biased top-k +
gates, histogram + scan + permute, grouped SwiGLU GEMMs (+ shared expert), gated
combine, and the +-gamma bias step.  Headline workload: the DeepSeek-V3-shaped layer
(N=4096 tokens, d_model=7168, 256 routed experts of d_ff=2048 plus one shared expert,
top-8, sigmoid scores normalised over the chosen 8), the largest single-GPU layer of the
five; the line's `per_config` object measures the other four (handbook, Mixtral-shaped,
Zipf-skewed at k=8 and k=4, all-fp32 tiny) the same way.

  python bench.py [--gpus N] [--steps K] [--warmup W] [--config NAME] [--impl reference]

Prints one JSON line (rank 0).  Under torchrun every rank runs an independent replica on
its own token batch (weak scaling); the per-expert counts are all-reduced before the
bias step so every replica keeps the same bias.
"""
from __future__ import annotations

import argparse
import json
import os
import platform
import statistics
import subprocess
import sys
import tempfile
import time

import numpy as np
import torch

ROOT = os.path.dirname(os.path.abspath(__file__))
sys.path.insert(0, ROOT)

from mixture_experts_layer_scores_b300 import moe, synth  # noqa: E402

METRIC = "MoE-layer fwd tokens/s; grouped-GEMM TFLOP/s & permute GB/s vs B300 peak"
FALLBACK_PEAKS = {"hbm_gbs": 6400.0, "bf16_tflops": 1800.0, "bf16_tflops_sustained": 1400.0}
DEFAULT_CONFIG = "deepseek_v3"
# (label, configuration, experts per token): the workloads of the line's per_config object
WORKLOADS = [("deepseek_v3", "deepseek_v3", 8), ("handbook", "handbook", 8), ("mixtral", "mixtral", 2),
             ("skewed_k8", "skewed", 8), ("skewed_k4", "skewed", 4), ("tiny", "tiny", 2)]
# fp32 FMA peak of the all-fp32 layer's CUDA-core kernels: 148 SMs x 128 lanes x 2 flops x 2.032 GHz
F32_ALU_TFLOPS = 148 * 128 * 2 * 2.032e9 / 1e12
# tokens of the workload the oracle runs per timed sample (about a second of host work each)
ORACLE_SAMPLE_TOKENS = {"tiny": 512, "handbook": 512, "mixtral": 16, "deepseek_v3": 6, "skewed": 512}


def peaks():
    p = os.path.join(ROOT, "MEASURED_PEAKS.json")
    if os.path.exists(p):
        with open(p) as f:
            d = json.load(f)
        return d, "measured"
    return FALLBACK_PEAKS, "fallback"


def recorded_traffic(cfg, gather):
    """ncu DRAM bytes of one grouped SwiGLU call (the row-gathering variant when `gather`), if
    recorded for this workload and the kernel sources are unchanged since (else None)."""
    import hashlib
    if synth.CONFIGS.get(cfg.name) != cfg:  # a scaled workload: the record is for the full size
        return None
    suffix = "_gather" if gather else ""
    path = os.path.join(ROOT, "profiles", f"grouped_gemm_{cfg.name}{suffix}_traffic.txt")
    if not os.path.exists(path):
        return None
    kv = {}
    with open(path) as f:
        for line in f:
            if "=" in line and not line.startswith("#"):
                k, v = line.strip().split("=", 1)
                kv[k] = v
    h = hashlib.sha256()
    for src in kv.get("sources", "").split():
        with open(os.path.join(ROOT, src), "rb") as f:
            h.update(f.read())
    if h.hexdigest() != kv.get("sources_sha256"):
        return None
    return int(kv["dram_bytes_per_call"])


def workload_name(cfg, k=None):
    k = cfg.k if k is None else k
    s = f"{cfg.name}: N={cfg.N} D={cfg.D} E={cfg.E} F={cfg.F} k={k} {cfg.score_fn}"
    if cfg.shared:
        s += f" +{cfg.shared} shared(F={cfg.F_shared})"
    if cfg.zipf_s:
        s += f" zipf({cfg.zipf_s})"
    if cfg.dtype != "bf16":
        s += f" all-{cfg.dtype}"
    return s


def config_dict(cfg, k, world):
    """The `config` object of both arms' lines: the workload only (the same dict in both)."""
    wbytes = 3 * cfg.E * cfg.D * cfg.F * (2 if cfg.dtype == "bf16" else 4)
    return {"workload": workload_name(cfg, k), "tokens_per_gpu": cfg.N,
            "l2": "no flush: every step streams %.0f MB of expert weights (L2 126 MB)" % (wbytes / 1e6)
                  if wbytes > 126e6 else "no flush: the whole layer fits in L2 (%.1f MB of weights)" % (wbytes / 1e6),
            "parallelism": f"replicas x{world}" if world > 1 else "single GPU"}


def router_bound(alg, us, pk, tensor_cores):
    """The router's roofline time and its fraction of the measured time: the slower of its
    bytes at the measured HBM bandwidth and its multiply-adds at the peak of the unit that runs
    them -- on tensor cores three bf16 products per fp32 weight (the exact three-plane split),
    on CUDA cores one fp32 FMA each."""
    t_bytes = alg["router_bytes"] / (pk["hbm_gbs"] * 1e9)
    if tensor_cores:
        flops, peak, unit = 3.0 * alg["router_flops"], pk["bf16_tflops"] * 1e12, "bf16 tensor (burst), 3 planes"
    else:
        flops, peak, unit = alg["router_flops"], F32_ALU_TFLOPS * 1e12, "fp32 FMA"
    t_flops = flops / peak
    bound = max(t_bytes, t_flops)
    return {"bound": "tensor" if t_flops > t_bytes else "hbm", "bound_us": round(bound * 1e6, 2),
            "bound_time_frac": bound / (us * 1e-6), "compute": unit}


def algorithmic(cfg, k=None, copy_rows=False):
    """Algorithmic flops and bytes of each step (only what the method must move).  The
    permute moves token rows only when the first GEMM does not gather them itself."""
    k = cfg.k if k is None else k
    N, D, E, F, S = cfg.N, cfg.D, cfg.E, cfg.F, cfg.shared
    R = N * k
    b = 2 if cfg.dtype == "bf16" else 4
    Fs = cfg.F_shared
    return dict(
        router_flops=2.0 * N * D * E,
        router_bytes=N * D * b + E * D * 4 + N * E * 4 + N * k * 8 + N,
        permute_bytes=(N * D * b + R * D * b if copy_rows else 0) + 12.0 * R,
        permute_copy_bytes=N * D * b + R * D * b + 12.0 * R,
        gemm_flops=6.0 * R * D * F,
        gemm_bytes=3.0 * E * D * F * b + R * D * b + 2.0 * R * F * b + R * D * b,
        shared_flops=6.0 * N * D * Fs * S,
        shared_bytes=(3.0 * D * Fs * b + N * D * b + 2.0 * N * Fs * b + N * D * b) * S,
        combine_bytes=R * D * b + 8.0 * R + (2 + S) * N * D * b,
    )


class ClockSampler:
    """nvidia-smi samples (every 20 ms) of SM clock, power and throttle reasons; summary()
    keeps the samples whose timestamps fall inside a host-time window (the timed region)."""

    FIELDS = ("timestamp,index,clocks.sm,clocks.max.sm,power.draw,clocks_event_reasons.active,"
              "clocks_event_reasons.hw_slowdown,clocks_event_reasons.hw_thermal_slowdown,"
              "clocks_event_reasons.sw_thermal_slowdown,clocks_event_reasons.sw_power_cap")

    def __init__(self, gpu_index):
        self.gpu = gpu_index
        self.proc = None
        self.path = None

    def __enter__(self):
        fd, self.path = tempfile.mkstemp(suffix=".csv")
        os.close(fd)
        try:
            self.proc = subprocess.Popen(
                ["nvidia-smi", f"--query-gpu={self.FIELDS}", "--format=csv,noheader,nounits", "-lms", "20",
                 "-i", str(self.gpu)], stdout=open(self.path, "w"), stderr=subprocess.DEVNULL)
        except (FileNotFoundError, OSError):
            self.proc = None
        time.sleep(0.3)
        return self

    def __exit__(self, *a):
        if self.proc is not None:
            self.proc.terminate()
            try:
                self.proc.wait(timeout=5)
            except subprocess.TimeoutExpired:
                self.proc.kill()

    def _rows(self):
        if getattr(self, "_parsed", None) is not None:
            return self._parsed
        import datetime
        rows = []
        names = ["hw_slowdown", "hw_thermal_slowdown", "sw_thermal_slowdown", "sw_power_cap"]
        with open(self.path) as f:
            for line in f:
                p = [x.strip() for x in line.split(",")]
                if len(p) < 10:
                    continue
                try:
                    ts = datetime.datetime.strptime(p[0], "%Y/%m/%d %H:%M:%S.%f").timestamp()
                    sm, smax = float(p[2]), float(p[3])
                except ValueError:
                    continue
                try:
                    pw = float(p[4])
                except ValueError:
                    pw = None
                act = {nm for nm, v in zip(names, p[6:10]) if v.lower() == "active"}
                rows.append((ts, sm, smax, pw, act))
        os.unlink(self.path)
        self._parsed = rows
        return rows

    def summary(self, window=None):
        if self.proc is None or (getattr(self, "_parsed", None) is None and not os.path.exists(self.path)):
            return {"sm_mhz": None, "sm_max_mhz": None, "reasons": ["nvidia-smi unavailable"]}
        rows = self._rows()
        scope = "timed region"
        if window is not None:
            inside = [r for r in rows if window[0] <= r[0] <= window[1]]
            if not inside:  # region shorter than the sampling period: the samples around it
                inside = sorted(rows, key=lambda r: abs(r[0] - 0.5 * (window[0] + window[1])))[:3]
                scope = "nearest samples to the timed region"
            rows = inside
        if not rows:
            return {"sm_mhz": None, "sm_max_mhz": None, "reasons": ["no samples"]}
        pw = [r[3] for r in rows if r[3] is not None]
        return {"sm_mhz": statistics.median(r[1] for r in rows), "sm_max_mhz": max(r[2] for r in rows),
                "reasons": sorted(set().union(*[r[4] for r in rows])), "samples": len(rows), "scope": scope,
                "power_w_median": statistics.median(pw) if pw else None, "power_w_max": max(pw) if pw else None}


REJECT_REASONS = ("hw_slowdown", "hw_thermal_slowdown", "sw_thermal_slowdown")


def clock_problem(summary):
    """Why a timed region's clock record makes its number invalid, or None: a hardware or
    thermal slowdown seen during it, or SM clocks far below their maximum with no reason
    active (a clock left locked low).  sw_power_cap alone is normal under a long load."""
    bad = [r for r in summary.get("reasons", []) if r in REJECT_REASONS]
    if bad:
        return ", ".join(bad)
    sm, smax = summary.get("sm_mhz"), summary.get("sm_max_mhz")
    if sm and smax and not summary.get("reasons") and sm < 0.6 * smax:
        return f"SM clock {sm:.0f} of {smax:.0f} MHz with no reason active"
    return None


def sustained_gemm(wl, calls=20, reps=25):
    """The layer's expert call (the grouped SwiGLU, with the shared expert's tiles when the
    layer runs them there) in a sustained loop -- a CUDA graph of `calls` back-to-back calls,
    replayed `reps` times (about 2 s on the DeepSeek-V3 layer) -- on three inputs that move the
    same bytes: the layer's routed counts, perfectly balanced counts (N k / E rows per expert:
    no padded row tiles) and all-zero activations with the routed counts.  With the power draw
    and SM clock that nvidia-smi reports over each loop: where the GPU holds its power limit,
    the differences show what the call's speed follows there."""
    L, cfg = wl.layer, wl.cfg
    wl.run()  # one forward: counts, offsets, permuted rows
    torch.cuda.synchronize()
    real = L.offsets.clone()
    R = cfg.N * wl.k
    balanced = torch.arange(0, R + 1, R // cfg.E, dtype=torch.int32, device=real.device) \
        if R % cfg.E == 0 else None
    zeros = torch.zeros_like(wl.xn)

    def tiles(off):
        c = (off[1:] - off[:-1]).long()
        return {"row_tiles": int(((c + 127) // 128).sum()), "half_tiles": int(((c % 128 > 0) & (c % 128 <= 64)).sum())}

    out = {}
    for name, off, xs, zero in (("routed counts", real, wl.xn, False), ("balanced counts", balanced, wl.xn, False),
                                ("zero activations", real, zeros, True)):
        if off is None:
            continue
        L.offsets.copy_(off)
        saved = None
        if zero and L.x_perm is not None:
            saved = L.x_perm.clone()
            L.x_perm.zero_()
        s = torch.cuda.Stream()
        s.wait_stream(torch.cuda.current_stream())

        def call():
            L.experts(xs, stream=s)
            L.shared_expert(xs, stream=s)
        with torch.cuda.stream(s):
            call()
        s.synchronize()
        g = torch.cuda.CUDAGraph()
        with torch.cuda.graph(g, stream=s):
            for _ in range(calls):
                call()
        torch.cuda.current_stream().wait_stream(s)
        g.replay()
        g.replay()
        torch.cuda.synchronize()
        e0, e1 = torch.cuda.Event(enable_timing=True), torch.cuda.Event(enable_timing=True)
        with ClockSampler(torch.cuda.current_device()) as clk:
            t0 = time.time()
            e0.record()
            for _ in range(reps):
                g.replay()
            e1.record()
            torch.cuda.synchronize()
            t1 = time.time()
        st = moe.last_device_status()
        if st != 0:
            raise SystemExit(f"device status {moe.STATUS.get(st, st)} in the sustained loop ({name})")
        out[name] = dict(tiles(off), ms_per_call=e0.elapsed_time(e1) / (calls * reps), clocks=clk.summary((t0, t1)))
        del g
        if saved is not None:
            L.x_perm.copy_(saved)
        time.sleep(1.0)
    L.offsets.copy_(real)
    return out


def cpu_model():
    try:
        with open("/proc/cpuinfo") as f:
            for line in f:
                if line.startswith("model name"):
                    return line.split(":", 1)[1].strip()
    except OSError:
        pass
    return platform.processor() or "unknown"


# ------------------------------------------------------------------------------------------
# CUDA arm
# ------------------------------------------------------------------------------------------

class Workload:
    """One layer (weights, tokens, reusable buffers) and its step: forward + bias step."""

    # "bias": the separate bias step of replicas (empty on one GPU, where the permute does it)
    STAGES = ("router", "permute", "grouped_swiglu", "shared", "combine", "bias")

    def __init__(self, cfg, k, dev, rank=0, world=1, gather=None, fuse_shared=True, router_shared=False):
        self.cfg, self.k, self.dev, self.world = cfg, k, dev, world
        self.xn, self.h = synth.make_tokens(cfg, dev, seed=cfg.seed + 1000 * rank)
        w_r, b = synth.make_router(cfg, dev)
        wg, wu, wd = synth.make_experts(cfg, dev)
        sh = synth.make_shared(cfg, dev)
        dt = torch.bfloat16 if cfg.dtype == "bf16" else torch.float32
        self.layer = moe.MoELayer(moe.LayerWeights(w_r, b, wg, wu, wd, sh), cfg.N, k, cfg.score_fn,
                                  cfg.gamma, dtype=dt, gather=gather, fuse_shared=fuse_shared,
                                  router_shared=router_shared)

    def run(self, xn=None, h=None, events=None, out=None):
        L = self.layer
        xn = self.xn if xn is None else xn
        h = self.h if h is None else h
        rec = (lambda i: events[i].record()) if events is not None else (lambda i: None)
        rec(0)
        L.route(xn)
        rec(1)
        # one replica: the +-gamma step rides in the permute's launches; replicas sum the
        # counts first (the global load histogram), then step the bias
        L.permute(xn, update_bias=self.world == 1)
        rec(2)
        L.experts(xn)
        rec(3)
        L.shared_expert(xn)
        rec(4)
        out = L.combine(h, out=out)
        rec(5)
        if self.world > 1:
            L.bias_step(moe.global_counts(L.counts))
        rec(6)
        return out

    @property
    def launches(self):
        return self.layer.kernels_per_forward(fused_bias=self.world == 1)


def _timed(fn, steps):
    """Device ms for `steps` calls of fn on the current stream (events at the ends only)."""
    t0 = torch.cuda.Event(enable_timing=True)
    t1 = torch.cuda.Event(enable_timing=True)
    torch.cuda.synchronize()
    t0.record()
    for _ in range(steps):
        fn()
    t1.record()
    torch.cuda.synchronize()
    return t0.elapsed_time(t1)


def time_device(wl, steps, warmup, world):
    """The headline: K forwards + bias steps back to back, events at the ends only.  On one
    GPU each step replays a CUDA graph of the layer (MoELayer.capture); with replicas the
    steps launch eagerly, since the counts all-reduce sits between the forward and the bias
    step.  Returns (ms for the K steps, launch mode)."""
    for _ in range(warmup):
        wl.run()
    fwd, mode = wl.run, "eager"
    if world == 1:
        fwd, mode = wl.layer.capture(wl.xn, wl.h), "cuda graph of the layer (MoELayer.capture)"
        for _ in range(warmup):
            fwd()
    torch.cuda.synchronize()
    if world > 1:
        torch.distributed.barrier()
    h0 = time.time()
    ms = _timed(fwd, steps)
    h1 = time.time()
    if world > 1:
        torch.distributed.barrier()
    return ms, mode, (h0, h1)


def stage_times(wl, steps, world):
    """Per-stage device µs over `steps` steps run back to back, as in the headline, with
    timing events between the stages.  On one GPU the steps are one CUDA graph holding all
    `steps` forwards one after another (every step with its own events, captured as event
    nodes), replayed once to warm it and once to time it.  The event nodes cut the
    programmatic overlap of the kernels on both sides of each, so the stage sum runs a
    little above the headline step.  With replicas: eager steps."""
    evs = [[torch.cuda.Event(enable_timing=True, external=True) for _ in range(7)] for _ in range(steps)]
    if world == 1:
        s = torch.cuda.Stream()
        s.wait_stream(torch.cuda.current_stream())
        g = torch.cuda.CUDAGraph()
        with torch.cuda.graph(g, stream=s):
            for e in evs:
                wl.run(events=e)
        torch.cuda.current_stream().wait_stream(s)
        g.replay()  # warm: the graph's first replay happens before the timed one
        torch.cuda.synchronize()
        run = g.replay
        how = "one CUDA graph of the back-to-back steps with event nodes between the stages, second replay"
    else:
        run = lambda: [wl.run(events=e) for e in evs]
        how = "eager steps with events between the stages"
    torch.cuda.synchronize()
    h0 = time.time()
    run()
    torch.cuda.synchronize()
    h1 = time.time()
    acc = {n: [e[j].elapsed_time(e[j + 1]) for e in evs] for j, n in enumerate(Workload.STAGES)}
    return {n: 1e3 * statistics.mean(v) for n, v in acc.items()}, how, (h0, h1)


def time_permute_copy(wl, steps):
    """The permute with the row copy (x_perm written) on the layer's routing, graph replays:
    the HBM-bound form of the step, measured also where the layer's GEMM gathers instead."""
    L, cfg = wl.layer, wl.cfg
    x_perm = torch.empty(cfg.N * wl.k, cfg.D, dtype=wl.xn.dtype, device=wl.xn.device)
    cnt, off = torch.empty_like(L.counts), torch.empty_like(L.offsets)
    rm, pt = torch.empty_like(L.row_map), torch.empty_like(L.perm_token)
    fn = lambda: moe.moe_permute(wl.xn, L.idx, L.E, cnt, off, rm, pt, x_perm, L.workspace)
    fn()
    s = torch.cuda.Stream()
    s.wait_stream(torch.cuda.current_stream())
    g = torch.cuda.CUDAGraph()
    with torch.cuda.graph(g, stream=s):
        fn()
    torch.cuda.current_stream().wait_stream(s)
    g.replay()
    us = 1e3 * _timed(g.replay, steps) / steps
    del x_perm
    return us


def time_e2e(wl, steps, warmup, world):
    """The layer fed from and drained to pinned host memory every step, the way a serving
    loop runs it: two sets of device buffers, host-to-device copies of step i+1 and the
    device-to-host copy of step i-1 on their own streams while step i computes."""
    cfg = wl.cfg
    hx = wl.xn.cpu().pin_memory()
    hh = wl.h.cpu().pin_memory()
    nb = 2
    hout = [torch.empty(cfg.N, cfg.D, dtype=wl.xn.dtype).pin_memory() for _ in range(nb)]
    dx = [torch.empty_like(wl.xn) for _ in range(nb)]
    dh = [torch.empty_like(wl.h) for _ in range(nb)]
    dout = [torch.empty(cfg.N, cfg.D, dtype=wl.xn.dtype, device=wl.xn.device) for _ in range(nb)]
    comp = torch.cuda.current_stream()
    for b in range(nb):
        dx[b].copy_(wl.xn)
        dh[b].copy_(wl.h)
    if world == 1:  # one graph per buffer set, as in the device-timed leg
        graphs = [wl.layer.capture(dx[b], dh[b], out=dout[b]) for b in range(nb)]
        fwd = lambda b: graphs[b]()
    else:
        fwd = lambda b: wl.run(dx[b], dh[b], out=dout[b])
    s_in, s_out = torch.cuda.Stream(), torch.cuda.Stream()
    ev = lambda: [torch.cuda.Event() for _ in range(nb)]
    in_ready, used, out_ready, out_copied = ev(), ev(), ev(), ev()

    def run(n):
        for i in range(n):
            b = i % nb
            with torch.cuda.stream(s_in):
                if i >= nb:
                    s_in.wait_event(used[b])  # step i-2 no longer reads these inputs
                dx[b].copy_(hx, non_blocking=True)
                dh[b].copy_(hh, non_blocking=True)
                in_ready[b].record(s_in)
            comp.wait_event(in_ready[b])
            if i >= nb:
                comp.wait_event(out_copied[b])  # step i-2's output has reached the host
            fwd(b)
            used[b].record(comp)
            out_ready[b].record(comp)
            with torch.cuda.stream(s_out):
                s_out.wait_event(out_ready[b])
                hout[b].copy_(dout[b], non_blocking=True)
                out_copied[b].record(s_out)
        for b in range(min(n, nb)):
            comp.wait_event(out_copied[b])

    run(warmup)
    torch.cuda.synchronize()
    if world > 1:
        torch.distributed.barrier()
    t0 = torch.cuda.Event(enable_timing=True)
    t1 = torch.cuda.Event(enable_timing=True)
    t0.record(comp)
    s_in.wait_event(t0)
    s_out.wait_event(t0)
    run(steps)
    t1.record(comp)
    torch.cuda.synchronize()
    if world > 1:
        torch.distributed.barrier()
    ms = t0.elapsed_time(t1)
    b = hx.element_size()
    return ms, 2 * cfg.N * cfg.D * b, cfg.N * cfg.D * b


def fresh_layer(wl, k):
    """A layer on the workload's weights with the initial bias and k experts per token."""
    cfg, w = wl.cfg, wl.layer.w
    b0 = synth.make_router(cfg, wl.dev)[1]
    dt = torch.bfloat16 if cfg.dtype == "bf16" else torch.float32
    return moe.MoELayer(moe.LayerWeights(w.w_router, b0, w.w_gate, w.w_up, w.w_down, w.shared), cfg.N, k,
                        cfg.score_fn, cfg.gamma, dtype=dt)


def load_balance_trace(wl, steps=50):
    """max/mean expert load of each of `steps` forwards, each on a fresh seeded batch
    (seed * 1000 + t) and each followed by the +-gamma bias step, from the initial bias
    (untimed)."""
    L = fresh_layer(wl, wl.k)
    trace = []
    for t in range(steps):
        xn, h = synth.make_tokens(wl.cfg, wl.dev, seed=wl.cfg.seed * 1000 + t)
        L.forward(xn, h)
        trace.append(round(float(L.mom.item()), 4))
    return {"gamma": wl.cfg.gamma, "steps": steps, "batches": "fresh seeded batch per step",
            "max_over_mean_per_step": trace}


def roofline_of(flops, bytes_, us, pk, long_run, dtype):
    """The bound of a kernel from its algorithmic flops and bytes (whichever takes longer at
    the measured peaks), and its achieved fraction of that bound."""
    if dtype != "bf16":
        ach = flops / (us * 1e-6) / 1e12
        return {"bound": "alu", "achieved": ach, "peak": F32_ALU_TFLOPS, "unit": "TFLOP/s",
                "frac": ach / F32_ALU_TFLOPS, "peak_kind": "fp32 FMA rate: 148 SMs x 128 lanes x 2.032 GHz"}
    pt = pk["bf16_tflops_sustained"] if long_run else pk["bf16_tflops"]
    t_tensor = flops / (pt * 1e12)
    t_hbm = bytes_ / (pk["hbm_gbs"] * 1e9)
    if t_tensor >= t_hbm:
        ach = flops / (us * 1e-6) / 1e12
        return {"bound": "tensor", "achieved": ach, "peak": pt, "unit": "TFLOP/s", "frac": ach / pt,
                "peak_kind": "bf16 " + ("sustained" if long_run else "burst"),
                "frac_of_burst": ach / pk["bf16_tflops"]}
    ach = bytes_ / (us * 1e-6) / 1e9
    return {"bound": "hbm", "achieved": ach, "peak": pk["hbm_gbs"], "unit": "GB/s", "frac": ach / pk["hbm_gbs"],
            "peak_kind": "HBM copy", "tensor_frac": flops / (us * 1e-6) / 1e12 / pt}


def measure(wl, steps, warmup, world, pk, e2e_steps):
    """Every number of one workload: headline graph replays, stage times, roofline, e2e."""
    cfg, k, L = wl.cfg, wl.k, wl.layer
    total_ms, mode, window = time_device(wl, steps, warmup, world)
    total_ms = max_over_ranks(total_ms, world)
    st = moe.last_device_status()
    if st != 0:
        raise SystemExit(f"device status {moe.STATUS.get(st, st)} after {cfg.name} k={k}")
    stage_us, how, stage_window = stage_times(wl, steps, world)
    ms = total_ms / steps
    alg = algorithmic(cfg, k, copy_rows=not L.gather)
    long_run = total_ms >= 1000.0
    alg_r = dict(alg)

    def gemm_roofline(sustained):
        """The grouped SwiGLU call against the sustained (power-capped) or burst bf16 peak."""
        a = dict(alg_r)

        def bound_s(flops, bytes_):  # the roofline time of one phase: the slower of its two bounds
            pt = pk["bf16_tflops_sustained"] if sustained else pk["bf16_tflops"]
            return max(flops / (pt * 1e12), bytes_ / (pk["hbm_gbs"] * 1e9))
        t_phases = bound_s(a["gemm_flops"], a["gemm_bytes"])
        if L.fuse_shared:  # the shared expert's tiles run in the routed experts' launches, after theirs
            sf, sb = a["shared_flops"], a["shared_bytes"]
            if L.router_shared:  # only its second GEMM: W_down, H read, output written
                Fs = cfg.F_shared
                sf, sb = sf / 3.0, (cfg.D * Fs + cfg.N * Fs + cfg.N * cfg.D) * 2.0
            t_phases += bound_s(sf, sb)
            a["gemm_flops"] += sf
            a["gemm_bytes"] += sb
        r = roofline_of(a["gemm_flops"], a["gemm_bytes"], stage_us["grouped_swiglu"], pk, sustained, cfg.dtype)
        if L.fuse_shared and cfg.dtype == "bf16":
            r["bound_time_frac"] = t_phases / (stage_us["grouped_swiglu"] * 1e-6)
            r["bound_time_note"] = ("(routed experts' roofline time + shared expert's roofline time) / measured "
                                    "time: the shared tiles follow the routed ones in each launch")
        return r, a
    gemm, alg = gemm_roofline(long_run)
    gbs = lambda b, us: b / (us * 1e-6) / 1e9
    hbm = pk["hbm_gbs"]
    copy_us = time_permute_copy(wl, steps)
    res = {
        "workload": workload_name(cfg, k), "tokens_per_s": cfg.N * world / (ms * 1e-3), "ms_per_step": ms,
        "timed_window": window, "stage_window": stage_window,
        "steps": steps, "launch": mode, "gemm1_rows": "gathered from xn" if L.gather else "permuted copy x_perm",
        "stage_us": {n: round(v, 2) for n, v in stage_us.items()},
        "stage_sum_us": round(sum(stage_us.values()), 2), "stage_us_from": how,
        "_gemm_sustained": gemm_roofline(True)[0],
        "grouped_gemm": dict(gemm, kernel="moe_grouped_swiglu_shared_h (routed + the shared expert's GEMM2; its "
                             "GEMM1 in the router launch)" if L.router_shared
                             else "moe_grouped_swiglu_shared (routed + shared expert)" if L.fuse_shared
                             else ("moe_grouped_swiglu_gather" if L.gather else "moe_grouped_swiglu"),
                             launches="GEMM1+SwiGLU and GEMM2", us=round(stage_us["grouped_swiglu"], 2),
                             tflops=alg["gemm_flops"] / (stage_us["grouped_swiglu"] * 1e-6) / 1e12,
                             algorithmic_gflop=alg["gemm_flops"] / 1e9,
                             algorithmic_gb=alg["gemm_bytes"] / 1e9),
        "router": dict({"gbs": gbs(alg["router_bytes"], stage_us["router"]),
                        "frac_hbm": gbs(alg["router_bytes"], stage_us["router"]) / hbm,
                        "algorithmic_mb": alg["router_bytes"] / 1e6, "launches": 3 if L.tc_router else 1},
                       **router_bound(alg, stage_us["router"], pk, L.tc_router)),
        "permute": {"moves_rows": not L.gather, "us": round(stage_us["permute"], 2),
                    "gbs": gbs(alg["permute_bytes"], stage_us["permute"]) if not L.gather else None,
                    "frac_hbm": gbs(alg["permute_bytes"], stage_us["permute"]) / hbm if not L.gather else None,
                    "index_only_mb": 12.0 * cfg.N * k / 1e6 if L.gather else None},
        "permute_with_row_copy": {"us": round(copy_us, 2), "gbs": gbs(alg["permute_copy_bytes"], copy_us),
                                  "frac_hbm": gbs(alg["permute_copy_bytes"], copy_us) / hbm,
                                  "algorithmic_mb": alg["permute_copy_bytes"] / 1e6},
        "combine": {"gbs": gbs(alg["combine_bytes"], stage_us["combine"]),
                    "frac_hbm": gbs(alg["combine_bytes"], stage_us["combine"]) / hbm,
                    "algorithmic_mb": alg["combine_bytes"] / 1e6},
        "gpu_launches_per_step": wl.launches,
    }
    if cfg.shared and not L.fuse_shared:
        res["shared_expert"] = roofline_of(alg["shared_flops"], alg["shared_bytes"], stage_us["shared"], pk,
                                           long_run, cfg.dtype)
    e2e_ms, bi, bo = time_e2e(wl, e2e_steps, warmup, world)
    e2e_ms = max_over_ranks(e2e_ms, world)
    res["e2e"] = {"value": cfg.N * world / (e2e_ms / e2e_steps * 1e-3), "unit": "tokens/s",
                  "h2d_bytes_per_step": bi, "d2h_bytes_per_step": bo}
    return res, total_ms


def settle_peak(res, stage_clocks):
    """A tensor-bound GEMM timed in a stage pass whose clock record shows sw_power_cap ran at
    the power-capped clock: compare it with the measured sustained bf16 peak (taken under the
    same cap) rather than the burst one; the burst fraction stays in frac_of_burst."""
    sus = res.pop("_gemm_sustained")
    g = res["grouped_gemm"]
    if g.get("bound") == "tensor" and "sw_power_cap" in (stage_clocks.get("reasons") or []) \
            and g.get("peak_kind", "").endswith("burst"):
        keep = {k2: g[k2] for k2 in ("kernel", "launches", "us", "tflops", "algorithmic_gflop", "algorithmic_gb")}
        res["grouped_gemm"] = dict(sus, **keep, peak_reason="stage pass under sw_power_cap")


def max_over_ranks(x, world):
    if world == 1:
        return x
    t = torch.tensor([x], dtype=torch.float64, device="cuda")
    torch.distributed.all_reduce(t, op=torch.distributed.ReduceOp.MAX)
    return float(t.item())


# ------------------------------------------------------------------------------------------
# CPU oracle (the reference arm and the cpu_baseline leg)
# ------------------------------------------------------------------------------------------

class OracleSample:
    """The oracle on the first n tokens of a workload, timed.

    The oracle's own functions run in its layer order: route, counts, scan, stable
    permutation, every visited expert's SwiGLU on its rows, the shared expert, the combine,
    the bias step.  Expert weights are regenerated once per expert (synth.make_expert: the
    same bits as the GPU's) and widened to float64 outside the timed sections, one expert
    at a time, so the largest layer (22.6 GB of bf16 weights) never sits in host memory.
    """

    def __init__(self, cfg, k, n):
        from oracle import moe_oracle as O
        self.O, self.cfg, self.k, self.n = O, cfg, k, n
        xn, h = synth.make_tokens(cfg, "cpu", rows=np.arange(n))
        self.x = xn.double().numpy()
        self.h = h.double().numpy()
        w_r, b = synth.make_router(cfg, "cpu")
        self.w_r, self.b = w_r.numpy(), b.numpy()
        # the experts the sample visits (the routing is recomputed, timed, in every run)
        idx = O.route(self.x, self.w_r, self.b, k, cfg.score_fn)["idx"]
        self.used = sorted({int(e) for e in idx.ravel()})
        self.weights = {e: synth.make_expert(cfg, e, "cpu") for e in self.used}
        self.shared = None
        if cfg.shared:
            self.shared = tuple(t.double().numpy() for t in synth.make_expert(cfg, 0, "cpu", shared=True))

    def run(self):
        """One pass; returns the seconds spent inside the oracle's functions."""
        O, cfg, k = self.O, self.cfg, self.k
        clock = time.perf_counter
        t0 = clock()
        r = O.route(self.x, self.w_r, self.b, k, cfg.score_fn)
        counts = O.expert_counts(r["idx"], cfg.E)
        offsets = O.exclusive_scan(counts)
        row_map, perm = O.stable_permutation(r["idx"], offsets)
        x_perm = self.x[perm]
        y = np.zeros((len(perm), cfg.D))
        spent = clock() - t0
        for e in self.used:
            a, b = int(offsets[e]), int(offsets[e + 1])
            if b > a:
                wg, wu, wd = (t.double().numpy() for t in self.weights[e])  # untimed widening
                t0 = clock()
                y[a:b] = O.swiglu_expert(x_perm[a:b], wg, wu, wd)
                spent += clock() - t0
        t0 = clock()
        ysh = O.swiglu_expert(self.x, *self.shared) if self.shared else None
        O.combine(y, row_map, r["gate"], residual=self.h, shared_y=ysh)
        O.bias_update(self.b, counts, r["idx"].size, cfg.gamma)
        return spent + clock() - t0

    def describe(self):
        return (f"first {self.n} of {self.cfg.N} tokens, k={self.k}: the oracle (numpy float64) routes them over "
                f"all {self.cfg.E} experts and runs the {len(self.used)} experts they visit"
                + (" and the shared expert" if self.cfg.shared else "")
                + "; weights regenerated and widened to float64 outside the timed sections")


def blas_threads():
    try:
        from threadpoolctl import threadpool_info
        n = [i.get("num_threads", 1) for i in threadpool_info() if i.get("user_api") == "blas"]
        return max(n) if n else 1
    except Exception:  # noqa: BLE001
        return os.cpu_count() or 1


def cpu_baseline(cfg, k, budget_s=10.0, max_runs=80):
    """The oracle, as it stands, on the reference arm's token sample, repeated for about
    `budget_s` seconds of oracle time (host cores)."""
    s = OracleSample(cfg, k, min(cfg.N, ORACLE_SAMPLE_TOKENS[cfg.name]))
    spent, runs = 0.0, 0
    while runs < max_runs and (spent < budget_s or runs < 2):
        spent += s.run()
        runs += 1
    return {"value": s.n * runs / spent, "unit": "tokens/s", "cores": blas_threads(), "cpu": cpu_model(),
            "kind": "oracle", "sample": s.describe() + f"; {runs} runs, {spent:.1f} s"}


def reference_arm(args, cfg, k):
    rank = int(os.environ.get("RANK", "0"))
    if rank != 0:
        return
    s = OracleSample(cfg, k, min(cfg.N, ORACLE_SAMPLE_TOKENS[cfg.name]))
    times = []
    for i in range(args.warmup + args.steps):
        dt = s.run()
        if i >= args.warmup:
            times.append(dt)
    tot = sum(times)
    val = s.n * len(times) / tot
    line = {"impl": "reference", "metric": METRIC, "value": val, "unit": "tokens/s", "n_gpus": args.gpus,
            "steps": args.steps, "warmup": args.warmup, "ms_per_step": 1e3 * tot / len(times),
            "higher_is_better": True, "scaling": "weak", "vs_baseline": None, "dtype": "f64",
            "data": "synthetic (seeded SplitMix64 / Irwin-Hall Gaussian tokens and weights)",
            "config": config_dict(cfg, k, args.gpus),
            "cpu_baseline": {"value": val, "unit": "tokens/s", "cores": blas_threads(), "cpu": cpu_model(),
                             "kind": "oracle", "sample": s.describe() + " per step"},
            "e2e": {"value": val, "unit": "tokens/s", "h2d_bytes_per_step": 0, "d2h_bytes_per_step": 0}}
    print(json.dumps(line), flush=True)


# ------------------------------------------------------------------------------------------

def main():
    ap = argparse.ArgumentParser()
    ap.add_argument("--gpus", type=int, default=1)
    ap.add_argument("--steps", type=int, default=20)
    ap.add_argument("--warmup", type=int, default=5)
    ap.add_argument("--config", default=DEFAULT_CONFIG, choices=sorted(synth.CONFIGS))
    ap.add_argument("--k", type=int, default=0, help="experts per token (default: the configuration's)")
    ap.add_argument("--impl", default="cuda", choices=["cuda", "reference"])
    ap.add_argument("--e2e-steps", type=int, default=20)
    ap.add_argument("--no-cpu-baseline", action="store_true")
    ap.add_argument("--no-per-config", action="store_true", help="measure the headline workload only")
    ap.add_argument("--override", default="",
                    help="comma-separated size overrides of the configuration, e.g. N=512,E=32 (a scaled "
                         "workload of the same recipe, for small profiling captures)")
    rows = ap.add_mutually_exclusive_group()
    rows.add_argument("--permute-copy", action="store_true",
                      help="the permute writes the permuted rows x_perm and GEMM1 loads them by TMA")
    ap.add_argument("--shared-separate", action="store_true",
                    help="run the shared expert in launches of its own instead of inside the routed experts' launches")
    ap.add_argument("--router-shared", action="store_true",
                    help="the shared expert's first GEMM in the router's launch (moe_router_topk_split_shared)")
    ap.add_argument("--sustained-gemm", action="store_true",
                    help="print only the expert call timed in a sustained loop on routed counts, "
                         "balanced counts and zero activations, with power and SM clock")
    rows.add_argument("--gather", action="store_true",
                      help="GEMM1 gathers its rows from xn through perm_token (default: the layer "
                           "chooses by size)")
    args = ap.parse_args()
    cfg = synth.CONFIGS[args.config]
    if args.override:
        kw = {kv.split("=")[0]: int(kv.split("=")[1]) for kv in args.override.split(",")}
        cfg = synth.scaled(cfg, **kw)
    k = args.k or cfg.k
    if args.impl == "reference":
        reference_arm(args, cfg, k)
        return
    if args.warmup < 3:
        raise SystemExit("--warmup must be >= 3")

    world = int(os.environ.get("WORLD_SIZE", "1"))
    rank = int(os.environ.get("RANK", "0"))
    local = int(os.environ.get("LOCAL_RANK", "0"))
    torch.cuda.set_device(local)
    if world > 1:
        torch.distributed.init_process_group("nccl", device_id=torch.device("cuda", local))
    dev = torch.device("cuda", local)
    pk, pk_kind = peaks()
    gather = True if args.gather else (False if args.permute_copy else None)

    wl = Workload(cfg, k, dev, rank, world, gather=gather, fuse_shared=not args.shared_separate,
                  router_shared=args.router_shared)
    torch.cuda.synchronize()
    if args.sustained_gemm:
        if rank == 0:
            print(json.dumps({"sustained_gemm": sustained_gemm(wl), "config": config_dict(cfg, k, world),
                              "gemm1_rows": "gathered from xn" if wl.layer.gather else "permuted copy x_perm"}))
        return
    with ClockSampler(local) as clk:
        head, total_ms = measure(wl, args.steps, args.warmup, world, pk, args.e2e_steps)
    clocks = clk.summary(head.pop("timed_window"))
    head["clocks_stage_pass"] = clk.summary(head.pop("stage_window"))
    settle_peak(head, head["clocks_stage_pass"])
    remeasured = clock_problem(clocks)
    # every rank measures again if any rank's record is invalid (the timing has barriers)
    if max_over_ranks(1.0 if remeasured else 0.0, world) > 0:
        remeasured = remeasured or "another rank's clock record"
        with ClockSampler(local) as clk:
            head, total_ms = measure(wl, args.steps, args.warmup, world, pk, args.e2e_steps)
        clocks = clk.summary(head.pop("timed_window"))
        head["clocks_stage_pass"] = clk.summary(head.pop("stage_window"))
        settle_peak(head, head["clocks_stage_pass"])

    g = head["grouped_gemm"]
    gemm_ms = g["us"] * 1e-3
    roof = {k2: g[k2] for k2 in ("bound", "achieved", "peak", "unit", "frac", "peak_kind", "peak_reason",
                                 "frac_of_burst", "bound_time_frac", "bound_time_note") if k2 in g}
    roof.update({"kernel": f"{g['kernel']} ({g['launches']} launches, one call)",
                 # the record is the default call's (with the shared expert's first GEMM)
                 "traffic": None if wl.layer.router_shared else recorded_traffic(cfg, wl.layer.gather),
                 "traffic_unit": "bytes per call (ncu)",
                 "peak_source": pk_kind, "timed": head["stage_us_from"],
                 "algorithmic": (f"{g['algorithmic_gb']:.2f} GB" if g["bound"] == "hbm"
                                 else f"{g['algorithmic_gflop']:.1f} GFLOP") + " per call",
                 "call_ms": gemm_ms})
    line = {
        "metric": METRIC, "value": head["tokens_per_s"], "unit": "tokens/s", "n_gpus": world, "steps": args.steps,
        "warmup": args.warmup, "ms_per_step": head["ms_per_step"], "higher_is_better": True, "scaling": "weak",
        "vs_baseline": None, "dtype": "bf16" if cfg.dtype == "bf16" else "f32",
        "data": "synthetic (seeded SplitMix64 / Irwin-Hall Gaussian tokens and weights)",
        "config": config_dict(cfg, k, world),
        "launch": head["launch"], "gemm1_rows": head["gemm1_rows"],
        "roofline": roof,
        "grouped_gemm_tflops": g["tflops"],
        "router": head["router"], "permute": head["permute"], "permute_with_row_copy": head["permute_with_row_copy"],
        "combine": head["combine"],
        "stage_us": head["stage_us"], "stage_sum_us": head["stage_sum_us"], "stage_us_from": head["stage_us_from"],
        "clocks_stage_pass": head["clocks_stage_pass"],
        "gpu_launches": wl.launches * args.steps,
        "clocks": dict(clocks, remeasured_after=remeasured) if remeasured else clocks,
        "e2e": head["e2e"],
    }
    if "shared_expert" in head:
        line["shared_expert"] = head["shared_expert"]
    if rank == 0:
        line["load_balance"] = load_balance_trace(wl)
    del wl
    torch.cuda.empty_cache()
    if not args.no_per_config:
        per = {}
        for label, name, kk in WORKLOADS:
            c2 = synth.CONFIGS[name]
            if name == cfg.name and kk == k:
                continue
            w2 = Workload(c2, kk, dev, rank, world, gather=gather if c2.dtype == "bf16" else None)
            with ClockSampler(local) as clk2:
                r2, _ = measure(w2, args.steps, args.warmup, world, pk, args.e2e_steps)
            r2["clocks"] = clk2.summary(r2.pop("timed_window"))
            r2["clocks_stage_pass"] = clk2.summary(r2.pop("stage_window"))
            settle_peak(r2, r2["clocks_stage_pass"])
            if rank == 0 and c2.bias_steps > 1:
                r2["load_balance"] = load_balance_trace(w2, c2.bias_steps)
            if rank == 0 and world == 1 and not args.no_cpu_baseline:
                r2["cpu_baseline"] = cpu_baseline(c2, kk, budget_s=3.0, max_runs=10)
            per[label] = r2
            del w2
            torch.cuda.empty_cache()
        line["per_config"] = per
    if rank == 0 and world == 1 and not args.no_cpu_baseline:
        line["cpu_baseline"] = cpu_baseline(cfg, k)
    if rank == 0:
        print(json.dumps(line), flush=True)
    if world > 1:
        torch.distributed.destroy_process_group()


if __name__ == "__main__":
    main()
