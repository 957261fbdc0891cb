#!/usr/bin/env python3
"""Benchmark of the top-k MoE layer forward on B300.

One step = one pass of the whole layer over one batch: router GEMM + biased top-k +
gates, histogram + scan + permute, grouped SwiGLU GEMMs (+ shared expert), gated
combine, and the +-gamma bias step.  Default workload: the handbook teaching-model
layer (N=8192 tokens, d_model=2048, 64 experts of d_ff=1024, top-8, softmax gates).

  python bench.py [--gpus N] [--steps K] [--warmup W] [--config NAME] [--impl reference]

Prints one JSON line (rank 0).  Under torchrun every rank runs an independent replica on
its own token batch (weak scaling); the per-expert counts are all-reduced before the
bias step so every replica keeps the same bias.
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

import numpy as np
import torch

ROOT = os.path.dirname(os.path.abspath(__file__))
sys.path.insert(0, ROOT)

from mixture_experts_layer_scores_b300 import moe, synth  # noqa: E402

METRIC = "MoE-layer fwd tokens/s; grouped-GEMM TFLOP/s & permute GB/s vs B300 peak"
FALLBACK_PEAKS = {"hbm_gbs": 6400.0, "bf16_tflops": 1800.0, "bf16_tflops_sustained": 1400.0}


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


def workload_name(cfg):
    s = f"{cfg.name}: N={cfg.N} D={cfg.D} E={cfg.E} F={cfg.F} k={cfg.k} {cfg.score_fn}"
    if cfg.shared:
        s += f" +{cfg.shared} shared(F={cfg.F_shared})"
    return s


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
        gemm_flops=6.0 * R * D * F,
        gemm_bytes=3.0 * E * D * F * b + R * D * b + 2.0 * R * F * b + R * D * b,
        shared_flops=6.0 * N * D * Fs * S,
        combine_bytes=R * D * b + 8.0 * R + (2 + S) * N * D * b,
    )


class ClockSampler:
    """nvidia-smi samples of SM clock and throttle reasons while the timed region runs."""

    def __init__(self, gpu_index):
        self.gpu = gpu_index
        self.proc = None
        self.path = None

    def __enter__(self):
        fd, self.path = tempfile.mkstemp(suffix=".csv")
        os.close(fd)
        q = ("index,clocks.sm,clocks.max.sm,power.draw,clocks_event_reasons.active,"
             "clocks_event_reasons.hw_slowdown,clocks_event_reasons.hw_thermal_slowdown,"
             "clocks_event_reasons.sw_thermal_slowdown,clocks_event_reasons.sw_power_cap")
        try:
            self.proc = subprocess.Popen(
                ["nvidia-smi", f"--query-gpu={q}", "--format=csv,noheader,nounits", "-lms", "100",
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

    def summary(self):
        if self.proc is None or not os.path.exists(self.path):
            return {"sm_mhz": None, "sm_max_mhz": None, "reasons": ["nvidia-smi unavailable"]}
        sm, smax, reasons = [], [], set()
        names = ["hw_slowdown", "hw_thermal_slowdown", "sw_thermal_slowdown", "sw_power_cap"]
        with open(self.path) as f:
            for line in f:
                p = [x.strip() for x in line.split(",")]
                if len(p) < 9:
                    continue
                try:
                    sm.append(float(p[1]))
                    smax.append(float(p[2]))
                except ValueError:
                    continue
                for nm, v in zip(names, p[5:9]):
                    if v.lower() == "active":
                        reasons.add(nm)
        os.unlink(self.path)
        if not sm:
            return {"sm_mhz": None, "sm_max_mhz": None, "reasons": ["no samples"]}
        return {"sm_mhz": statistics.median(sm), "sm_max_mhz": max(smax), "reasons": sorted(reasons),
                "samples": len(sm)}


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


# ------------------------------------------------------------------------------------------
# CUDA arm
# ------------------------------------------------------------------------------------------

class Step:
    """One layer forward + bias step with CUDA events between the stages."""

    STAGES = ("router", "permute", "grouped_swiglu", "shared", "combine", "bias")

    def __init__(self, cfg, dev, rank, world, gather=None):
        self.cfg, self.dev, self.world = cfg, dev, world
        seed_tok = cfg.seed + 1000 * rank
        xn, h = synth.make_tokens(cfg, dev, seed=seed_tok)
        self.xn, self.h = xn, h
        w_r, b = synth.make_router(cfg, dev)
        wg, wu, wd = synth.make_experts(cfg, dev)
        sh = synth.make_shared(cfg, dev)
        self.layer = moe.MoELayer(moe.LayerWeights(w_r, b, wg, wu, wd, sh), cfg.N, cfg.k,
                                  cfg.score_fn, cfg.gamma, gather=gather)
        self.ev = None

    def run(self, xn=None, h=None, events=None, out=None):
        L = self.layer
        xn = self.xn if xn is None else xn
        h = self.h if h is None else h
        rec = (lambda i: events[i].record()) if events is not None else (lambda i: None)
        rec(0)
        L.route(xn)
        rec(1)
        L.permute(xn)
        rec(2)
        L.experts(xn)
        rec(3)
        L.shared_expert(xn)
        rec(4)
        out = L.combine(h, out=out)
        rec(5)
        world = moe.global_counts(L.counts)  # global load histogram for the bias step
        L.bias_step(world)
        rec(6)
        return out

    @property
    def launches(self):
        return self.layer.kernels_per_forward


def time_device(step, steps, warmup, world):
    """The headline: K forwards + bias steps back to back, with events at the ends only.  On
    one GPU each step replays a CUDA graph of the layer (MoELayer.capture); with replicas the
    steps launch eagerly, since the counts all-reduce sits between the forward and the bias
    step.  Then K more eager steps with events between the stages give the per-stage times
    (the grouped GEMM's among them, for the roofline).  Returns (ms for the K headline
    steps, stage µs, launch mode)."""
    for _ in range(warmup):
        step.run()
    fwd, mode = step.run, "eager"
    if world == 1:
        fwd, mode = step.layer.capture(step.xn, step.h), "cuda graph of the layer (MoELayer.capture)"
        for _ in range(warmup):
            fwd()
    torch.cuda.synchronize()
    t0 = torch.cuda.Event(enable_timing=True)
    t1 = torch.cuda.Event(enable_timing=True)
    if world > 1:
        torch.distributed.barrier()
    torch.cuda.synchronize()
    t0.record()
    for _ in range(steps):
        fwd()
    t1.record()
    torch.cuda.synchronize()
    if world > 1:
        torch.distributed.barrier()
    total_ms = t0.elapsed_time(t1)
    evs = [[torch.cuda.Event(enable_timing=True) for _ in range(7)] for _ in range(steps)]
    for i in range(steps):
        step.run(events=evs[i])
    torch.cuda.synchronize()
    stage_us = {}
    for j, name in enumerate(Step.STAGES):
        stage_us[name] = 1e3 * statistics.mean(e[j].elapsed_time(e[j + 1]) for e in evs)
    return total_ms, stage_us, mode


def time_e2e(step, steps, warmup, world):
    """The layer fed from and drained to pinned host memory every step, the way a serving
    loop runs it: two sets of device buffers, host-to-device copies of step i+1 and the
    device-to-host copy of step i-1 on their own streams while step i computes."""
    cfg = step.cfg
    hx = step.xn.cpu().pin_memory()
    hh = step.h.cpu().pin_memory()
    nb = 2
    hout = [torch.empty(cfg.N, cfg.D, dtype=step.xn.dtype).pin_memory() for _ in range(nb)]
    dx = [torch.empty_like(step.xn) for _ in range(nb)]
    dh = [torch.empty_like(step.h) for _ in range(nb)]
    dout = [torch.empty(cfg.N, cfg.D, dtype=step.xn.dtype, device=step.xn.device) for _ in range(nb)]
    comp = torch.cuda.current_stream()
    for b in range(nb):
        dx[b].copy_(step.xn)
        dh[b].copy_(step.h)
    if world == 1:  # one graph per buffer set, as in the device-timed leg
        graphs = [step.layer.capture(dx[b], dh[b], out=dout[b]) for b in range(nb)]
        fwd = lambda b: graphs[b]()
    else:
        fwd = lambda b: step.run(dx[b], dh[b], out=dout[b])
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


def fresh_layer(step, k):
    """A layer on the step's weights and tokens with the initial bias and k experts per token."""
    cfg, w = step.cfg, step.layer.w
    b0 = synth.make_router(cfg, step.dev)[1]
    return moe.MoELayer(moe.LayerWeights(w.w_router, b0, w.w_gate, w.w_up, w.w_down, w.shared), cfg.N, k,
                        cfg.score_fn, cfg.gamma)


def load_balance_trace(step, steps=50):
    """max/mean expert load after each of `steps` forwards with the +-gamma bias step, from the
    initial bias (untimed)."""
    L = fresh_layer(step, step.cfg.k)
    trace = []
    for _ in range(steps):
        L.forward(step.xn, step.h)
        trace.append(round(float(L.mom.item()), 4))
    return {"gamma": step.cfg.gamma, "steps": steps, "max_over_mean_per_step": trace}


def time_fewer_experts(step, k, steps, warmup):
    """The same weights served with k experts per token instead of cfg.k (gates renormalise
    over the k chosen): tokens/s over `steps` timed forwards."""
    cfg, xn, h = step.cfg, step.xn, step.h
    L = fresh_layer(step, k)
    for _ in range(warmup):
        L.forward(xn, h)
    fwd = L.capture(xn, h)  # replayed as in the headline leg
    for _ in range(warmup):
        fwd()
    torch.cuda.synchronize()
    e0, e1 = torch.cuda.Event(enable_timing=True), torch.cuda.Event(enable_timing=True)
    e0.record()
    for _ in range(steps):
        fwd()
    e1.record()
    torch.cuda.synchronize()
    ms = e0.elapsed_time(e1) / steps
    return {"k": k, "tokens_per_s": cfg.N / (ms * 1e-3), "ms_per_step": ms}


def max_over_ranks(x, world):
    if world == 1:
        return x
    t = torch.tensor([x], dtype=torch.float64, device="cuda")
    torch.distributed.all_reduce(t, op=torch.distributed.ReduceOp.MAX)
    return float(t.item())


# ------------------------------------------------------------------------------------------
# CPU oracle (the reference arm and the cpu_baseline leg)
# ------------------------------------------------------------------------------------------

def oracle_sample(cfg, n_tok):
    """Inputs for the first n_tok tokens of the workload, plus the full weights (CPU)."""
    rows = np.arange(n_tok)
    xn, h = synth.make_tokens(cfg, "cpu", rows=rows)
    w_r, b = synth.make_router(cfg, "cpu")
    wg, wu, wd = synth.make_experts(cfg, "cpu")
    sh = synth.make_shared(cfg, "cpu")
    f = lambda t: t.to(torch.float32).numpy()
    return dict(xn=f(xn), h=f(h), w_r=w_r.numpy(), b=b.numpy(), wg=f(wg), wu=f(wu), wd=f(wd),
                sh=None if sh is None else tuple(f(t) for t in sh))


def run_oracle(cfg, s):
    from oracle import moe_oracle
    return moe_oracle.moe_layer(s["xn"], s["h"], s["w_r"], s["b"], s["wg"], s["wu"], s["wd"], cfg.k,
                                cfg.score_fn, shared=s["sh"], gamma=cfg.gamma)


def blas_threads():
    try:
        from threadpoolctl import threadpool_info
        n = [i.get("num_threads", 1) for i in threadpool_info() if i.get("user_api") == "blas"]
        return max(n) if n else 1
    except Exception:  # noqa: BLE001
        return os.cpu_count() or 1


def cpu_baseline(cfg, budget_s=20.0):
    """The oracle, as it stands, on a bounded token sample of the workload (host cores)."""
    n = min(cfg.N, 64)
    s = oracle_sample(cfg, cfg.N)
    while True:
        sub = dict(s, xn=s["xn"][:n], h=s["h"][:n])
        t = time.perf_counter()
        run_oracle(cfg, sub)
        dt = time.perf_counter() - t
        if dt * 2 > budget_s or n >= cfg.N:
            break
        n = min(cfg.N, int(n * max(2.0, min(8.0, budget_s / 2 / max(dt, 1e-3)))))
    return {"value": n / dt, "unit": "tokens/s", "cores": blas_threads(), "kind": "oracle",
            "sample": f"first {n} of {cfg.N} tokens of the workload, all {cfg.E} experts "
                      f"(numpy float64, {dt:.1f} s)"}


def reference_arm(args, cfg):
    rank = int(os.environ.get("RANK", "0"))
    if rank != 0:
        return
    s = oracle_sample(cfg, cfg.N)
    n = min(cfg.N, 128)
    sub = dict(s, xn=s["xn"][:n], h=s["h"][:n])
    times = []
    for i in range(args.warmup + args.steps):
        t = time.perf_counter()
        run_oracle(cfg, sub)
        if i >= args.warmup:
            times.append(time.perf_counter() - t)
    tot = sum(times)
    val = n * len(times) / tot
    line = {"impl": "reference", "metric": METRIC, "value": val, "unit": "tokens/s", "n_gpus": args.gpus,
            "steps": args.steps, "warmup": args.warmup, "ms_per_step": 1e3 * tot / len(times),
            "higher_is_better": True, "scaling": "weak", "vs_baseline": None, "dtype": "f64",
            "data": "synthetic", "config": {"workload": workload_name(cfg)},
            "cpu_baseline": {"value": val, "unit": "tokens/s", "cores": blas_threads(), "kind": "oracle",
                             "sample": f"first {n} of {cfg.N} tokens per step, all {cfg.E} experts"},
            "e2e": {"value": val, "unit": "tokens/s", "h2d_bytes_per_step": 0, "d2h_bytes_per_step": 0}}
    print(json.dumps(line), flush=True)


# ------------------------------------------------------------------------------------------

def main():
    ap = argparse.ArgumentParser()
    ap.add_argument("--gpus", type=int, default=1)
    ap.add_argument("--steps", type=int, default=2000)
    ap.add_argument("--warmup", type=int, default=5)
    ap.add_argument("--config", default="handbook", choices=sorted(synth.CONFIGS))
    ap.add_argument("--impl", default="cuda", choices=["cuda", "reference"])
    ap.add_argument("--e2e-steps", type=int, default=50)
    ap.add_argument("--no-cpu-baseline", action="store_true")
    rows = ap.add_mutually_exclusive_group()
    rows.add_argument("--permute-copy", action="store_true",
                      help="the permute writes the permuted rows x_perm and GEMM1 loads them by TMA")
    rows.add_argument("--gather", action="store_true",
                      help="GEMM1 gathers its rows from xn through perm_token (default: the layer "
                           "chooses by size)")
    args = ap.parse_args()
    cfg = synth.CONFIGS[args.config]
    if args.impl == "reference":
        reference_arm(args, cfg)
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

    step = Step(cfg, dev, rank, world, gather=True if args.gather else (False if args.permute_copy else None))
    torch.cuda.synchronize()
    with ClockSampler(local) as clk:
        total_ms, stage_us, launch_mode = time_device(step, args.steps, args.warmup, world)
    clocks = clk.summary()
    remeasured = clock_problem(clocks)
    # every rank measures again if any rank's record is invalid (the timing has barriers)
    if max_over_ranks(1.0 if remeasured else 0.0, world) > 0:
        remeasured = remeasured or "another rank's clock record"
        with ClockSampler(local) as clk:
            total_ms, stage_us, launch_mode = time_device(step, args.steps, args.warmup, world)
        clocks = clk.summary()
    total_ms = max_over_ranks(total_ms, world)
    st = moe.last_device_status()
    if st != 0:
        raise SystemExit(f"device status {moe.STATUS.get(st, st)}")
    e2e_ms, bi, bo = time_e2e(step, args.e2e_steps, args.warmup, world)
    e2e_ms = max_over_ranks(e2e_ms, world)

    ms_step = total_ms / args.steps
    tokens = cfg.N * world
    value = tokens / (ms_step * 1e-3)
    alg = algorithmic(cfg, copy_rows=not step.layer.gather)
    pk, pk_kind = peaks()
    gemm_us = stage_us["grouped_swiglu"]
    gemm_tflops = alg["gemm_flops"] / (gemm_us * 1e-6) / 1e12
    perm_gbs = alg["permute_bytes"] / (stage_us["permute"] * 1e-6) / 1e9
    # a kernel timed inside a loop of a second or more runs under the power cap: compare it
    # with the sustained bf16 figure; shorter timed regions with the burst figure
    long_run = total_ms >= 1000.0
    peak_t = pk["bf16_tflops_sustained"] if long_run else pk["bf16_tflops"]
    peak_label = f"{pk_kind} bf16 {'sustained' if long_run else 'burst'}"
    line = {
        "metric": METRIC, "value": value, "unit": "tokens/s", "n_gpus": world, "steps": args.steps,
        "warmup": args.warmup, "ms_per_step": ms_step, "higher_is_better": True, "scaling": "weak",
        "vs_baseline": None, "dtype": "bf16" if cfg.dtype == "bf16" else "f32",
        "data": "synthetic (seeded SplitMix64 / Irwin-Hall Gaussian tokens and weights)",
        "config": {"workload": workload_name(cfg), "tokens_per_gpu": cfg.N,
                   "l2": "inputs larger than L2: every step streams %.0f MB of expert weights"
                         % (3 * cfg.E * cfg.D * cfg.F * 2 / 1e6),
                   "gemm1_rows": "gathered from xn" if step.layer.gather else "permuted copy x_perm",
                   "parallelism": f"replicas x{world}" if world > 1 else "single GPU",
                   "launch": launch_mode,
                   "stage_us_from": "a second pass of the same steps, eager, events between stages"},
        "roofline": {"kernel": ("moe_grouped_swiglu_gather" if step.layer.gather else "moe_grouped_swiglu")
                               + " (GEMM1+SwiGLU and GEMM2 launches)", "bound": "tensor",
                     "achieved": gemm_tflops, "peak": peak_t, "unit": "TFLOP/s",
                     "frac": gemm_tflops / peak_t, "traffic": recorded_traffic(cfg, step.layer.gather),
                     "traffic_unit": "bytes per call (ncu)", "peak_kind": peak_label,
                     "frac_of_burst": gemm_tflops / pk["bf16_tflops"]},
        "grouped_gemm_tflops": gemm_tflops,
        # with gathering, the permute moves no rows (GEMM1 reads them): only its index work
        "permute_gbs": perm_gbs,
        "permute_frac_hbm": None if step.layer.gather else perm_gbs / pk["hbm_gbs"],
        "permute_moves_rows": not step.layer.gather,
        "router_gbs": alg["router_bytes"] / (stage_us["router"] * 1e-6) / 1e9,
        "combine_gbs": alg["combine_bytes"] / (stage_us["combine"] * 1e-6) / 1e9,
        "stage_us": {k: round(v, 2) for k, v in stage_us.items()},
        "gpu_launches": step.launches * args.steps,
        "clocks": dict(clocks, remeasured_after=remeasured) if remeasured else clocks,
        "e2e": {"value": tokens / (e2e_ms / args.e2e_steps * 1e-3), "unit": "tokens/s",
                "h2d_bytes_per_step": bi, "d2h_bytes_per_step": bo},
    }
    if rank == 0:
        line["load_balance"] = load_balance_trace(step)
        if cfg.name == "skewed":  # serving with fewer experts per token than trained
            line["serving_fewer_experts"] = time_fewer_experts(step, 4, min(args.steps, 500), args.warmup)
    if rank == 0 and world == 1 and not args.no_cpu_baseline:
        line["cpu_baseline"] = cpu_baseline(cfg)
    if rank == 0:
        print(json.dumps(line), flush=True)
    if world > 1:
        torch.distributed.destroy_process_group()


if __name__ == "__main__":
    main()
