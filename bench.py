#!/usr/bin/env python
"""Benchmark of the routed-expert MoE FFN layer (router, permute, expert SwiGLU FFN, combine +
shared expert) on one GB300, through the library's C ABI.

One step = one pass of the whole layer over one batch of T tokens, inputs already in HBM.
Prints one JSON line. Headline workload: the DeepSeek-V3-shaped decode layer (T=256, d=7168,
256 routed + 1 shared experts, top-8, f=2048, bf16 weights). The same line carries a `sweep`
array: the token-batch sweep T in {1, 8, 64, 256, 1024, 4096, 16384} of the V3 shape with FP8
weights, the skewed-load prefill layer and the V4-Pro-shaped decode layers, each measured the
same way.

  python bench.py [--steps K] [--warmup W] [--config NAME] [--sweep default|all|none]
                  [--impl ours|reference]

The library is a one-GPU library: `--gpus` must be 1 (the layer does not shard without an
exchange step this build does not implement, and its prefill tiles load shared token rows into
both CTAs of a cluster pair, which is for one-GPU runs only).
--impl reference times the CPU oracle on the host cores instead.
"""
from __future__ import annotations

import argparse
import datetime
import hashlib
import json
import math
import os
import statistics
import subprocess
import sys
import time

ROOT = os.path.dirname(os.path.abspath(__file__))
sys.path.insert(0, ROOT)

METRIC = "MoE-layer tokens/s and achieved HBM GB/s (% roofline) vs token batch T, 1×GB300"
FALLBACK_HBM_GBS = 6800.0
FALLBACK_BF16_TFLOPS = 1900.0
FALLBACK_BF16_TFLOPS_SUSTAINED = 1700.0

SWEEP_T = (1, 8, 64, 256, 1024, 4096, 16384)
SWEEPS = {
    "default": [f"sweep_fp8_T{t}" for t in SWEEP_T] + ["skewed_prefill", "v4pro_decode",
                                                       "v4pro_decode_fp4"],
    "all": ([f"sweep_fp8_T{t}" for t in SWEEP_T] + [f"sweep_fp4_T{t}" for t in SWEEP_T]
            + ["skewed_prefill", "v4pro_decode", "v4pro_decode_fp4", "tiny"]),
    "none": [],
}


def parse_args(argv=None):
    p = argparse.ArgumentParser()
    p.add_argument("--gpus", type=int, default=1)
    p.add_argument("--steps", type=int, default=200)
    p.add_argument("--warmup", type=int, default=10)
    p.add_argument("--config", default="v3_decode")
    p.add_argument("--impl", choices=("ours", "reference"), default="ours")
    p.add_argument("--sweep", choices=tuple(SWEEPS), default="default",
                   help="workloads measured after the headline, each reported in `sweep`")
    p.add_argument("--sweep-min-ms", type=float, default=400.0,
                   help="shortest timed region of a sweep point (more steps for short layers)")
    p.add_argument("--no-cpu-baseline", action="store_true")
    p.add_argument("--no-graph", action="store_true",
                   help="launch the layer eagerly each step instead of replaying a CUDA graph")
    p.add_argument("--e2e-steps", type=int, default=None)
    p.add_argument("--graph-passes", type=int, default=8,
                   help="layer passes captured back to back in the timed CUDA graph (as a "
                        "model's layers follow one another in one graph)")
    p.add_argument("--T", type=int, default=None, help="override the token batch (profiling cases)")
    p.add_argument("--E", type=int, default=None, help="override the routed experts (profiling cases)")
    return p.parse_args(argv)


def workload_desc(cfg) -> str:
    w = {"bf16": "bf16 weights", "fp8": "FP8 E4M3 weights with fp32 128x128 block scales",
         "mxfp4": "MXFP4 weights (E2M1 codes, one E8M0 scale per 32 elements)"}[cfg.wdtype]
    r = "Zipf(s=1.1) popularity bias" if cfg.router == "zipf" else "plain router"
    return (f"{cfg.name}: T={cfg.T} tokens, d={cfg.d}, {cfg.E} routed + {cfg.n_shared} shared "
            f"experts, top-{cfg.k}, expert intermediate f={cfg.f}, SwiGLU, {w}, bf16 activations, "
            f"{r}, seed {cfg.seed}")


def config_record(cfg, **extra) -> dict:
    rec = {"workload": workload_desc(cfg), "T": cfg.T, "d": cfg.d, "E": cfg.E, "k": cfg.k,
           "f": cfg.f, "n_shared": cfg.n_shared, "weights": cfg.wdtype, "router": cfg.router,
           "parallelism": "one GPU"}
    rec.update(extra)
    return rec


def dtype_of(cfg) -> str:
    return {"bf16": "bf16", "fp8": "fp8_e4m3 weights, bf16 activations",
            "mxfp4": "mxfp4 (e2m1 + e8m0) weights, bf16 activations as two e4m3 terms"}[cfg.wdtype]


def measured_peaks():
    path = os.path.join(ROOT, "MEASURED_PEAKS.json")
    try:
        with open(path) as fh:
            return json.load(fh), "measured"
    except (OSError, ValueError):
        return {"hbm_gbs": FALLBACK_HBM_GBS, "bf16_tflops": FALLBACK_BF16_TFLOPS,
                "bf16_tflops_sustained": FALLBACK_BF16_TFLOPS_SUSTAINED}, "fallback"


def kernel_sources_sha(files) -> str:
    h = hashlib.sha256()
    for fn in files:
        with open(os.path.join(ROOT, fn), "rb") as fh:
            h.update(os.path.basename(fn).encode() + fh.read())
    return h.hexdigest()[:16]


def ncu_traffic(config_name: str):
    """DRAM bytes per launch of the gate/up kernel from a committed ncu capture, if it was taken
    on the kernel's current sources; else None."""
    path = os.path.join(ROOT, "profiles", "ncu_traffic.json")
    try:
        with open(path) as fh:
            ent = json.load(fh).get(config_name)
        if ent and ent.get("kernel_sources_sha") == kernel_sources_sha(ent["kernel_sources"]):
            return ent.get("dram_bytes_per_launch")
    except (OSError, ValueError, KeyError):
        pass
    return None


class ClockSampler:
    """nvidia-smi clocks and throttle reasons every 50 ms while a measurement runs. Each sample
    carries nvidia-smi's own timestamp, so the samples that fall inside the timed region are
    known (`mark_timed`)."""
    Q = ("timestamp,index,clocks.sm,clocks.max.sm,power.draw,clocks_event_reasons.active,"
         "clocks_event_reasons.hw_slowdown,clocks_event_reasons.hw_thermal_slowdown,"
         "clocks_event_reasons.sw_thermal_slowdown,clocks_event_reasons.sw_power_cap")
    REASONS = ["hw_slowdown", "hw_thermal_slowdown", "sw_thermal_slowdown", "sw_power_cap"]

    def __init__(self, dev_index: int):
        self.proc = None
        self.dev = dev_index
        self.lines = []
        self.timed = None

    def __enter__(self):
        try:
            import torch
            uuid = str(torch.cuda.get_device_properties(self.dev).uuid)
            sel = ["-i", uuid if uuid.startswith("GPU-") else "GPU-" + uuid]
        except Exception:
            sel = []
        try:
            self.proc = subprocess.Popen(["nvidia-smi", "--query-gpu=" + self.Q,
                                          "--format=csv,noheader,nounits", "-lms", "50"] + sel,
                                         stdout=subprocess.PIPE, stderr=subprocess.DEVNULL, text=True)
            time.sleep(0.3)  # the first sample comes after nvidia-smi has started
        except OSError:
            self.proc = None
        return self

    def mark_timed(self, t0: float, t1: float):
        """Host wall-clock bounds (time.time()) of the timed region."""
        self.timed = (t0, t1)

    def __exit__(self, *exc):
        if self.proc is not None:
            time.sleep(0.12)
            self.proc.terminate()
            try:
                out, _ = self.proc.communicate(timeout=5)
            except subprocess.TimeoutExpired:
                self.proc.kill()
                out, _ = self.proc.communicate()
            self.lines = [ln for ln in out.splitlines() if ln.strip()]
        return False

    def _samples(self):
        for ln in self.lines:
            parts = [p.strip() for p in ln.split(",")]
            if len(parts) < 10:
                continue
            try:
                ts = datetime.datetime.strptime(parts[0], "%Y/%m/%d %H:%M:%S.%f").timestamp()
                sm, mx = float(parts[2]), float(parts[3])
            except ValueError:
                continue
            reasons = {nm for nm, v in zip(self.REASONS, parts[6:10]) if v.lower() == "active"}
            yield ts, sm, mx, reasons

    def summary(self):
        """Median SM clock and every throttle reason seen while the measurement ran (the timed
        region and the phase and end-to-end loops that follow it on the same workload), and the
        same over the samples inside the timed region alone."""
        allv = list(self._samples())
        inside = [s for s in allv if self.timed and self.timed[0] - 0.05 <= s[0] <= self.timed[1] + 0.05]
        if not allv:
            return {"sm_mhz": None, "sm_max_mhz": None, "reasons": [], "samples": 0,
                    "samples_in_timed_region": 0}
        out = {"sm_mhz": statistics.median(s[1] for s in allv),
               "sm_max_mhz": max(s[2] for s in allv),
               "reasons": sorted(set().union(*(s[3] for s in allv))),
               "samples": len(allv), "samples_in_timed_region": len(inside),
               "window": "timed region + phase loop + end-to-end loop of this workload"}
        if inside:
            out["timed_region"] = {"sm_mhz": statistics.median(s[1] for s in inside),
                                   "reasons": sorted(set().union(*(s[3] for s in inside)))}
        return out


# ---------------------------------------------------------------------------------------------
# CPU oracle: the whole layer, step by step, on the host cores (cpu_baseline and --impl reference)
# ---------------------------------------------------------------------------------------------

def oracle_threads() -> int:
    os.environ.setdefault("OMP_NUM_THREADS", str(os.cpu_count() or 1))
    return int(os.environ["OMP_NUM_THREADS"])


def oracle_layer_seconds(cfg, x_rows, wg, bias, get_expert):
    """Runs the oracle's whole layer on the token rows x_rows [n, d] (bf16 bits): fp32 router
    logits over all E experts, top-k and gate weights, the permutation, every routed expert that
    received tokens on its rows, the shared expert on every token, and the combine. Weights come
    from get_expert(e) between the timed pieces (fetching or drawing them is input preparation,
    not the oracle's work). Returns (seconds of oracle work, experts run, y [n, d] fp64)."""
    import numpy as np

    import oracle
    n, k = x_rows.shape[0], cfg.k
    t0 = time.perf_counter()
    logits = oracle.router_logits(x_rows, wg, bias)
    idx, _, w64 = oracle.route(logits, k)
    off, perm, inv = oracle.permute(idx, cfg.E, cfg.n_shared)
    secs = time.perf_counter() - t0
    y_perm = np.zeros((n * k + cfg.n_shared * n, cfg.d), np.float64)
    run = 0
    for e in range(cfg.E + cfg.n_shared):
        lo, hi = (int(off[e]), int(off[e + 1])) if e < cfg.E else (n * k, n * k + n)
        if hi == lo:
            continue
        ew = get_expert(e)
        rows = x_rows[perm[lo:hi]] if e < cfg.E else x_rows
        t0 = time.perf_counter()
        y_perm[lo:hi] = oracle.expert_rows(rows, ew.w13, ew.w2, cfg.wdtype, ew.s13, ew.s2)
        secs += time.perf_counter() - t0
        run += 1
    t0 = time.perf_counter()
    y = oracle.combine(y_perm, inv, w64, n, k, cfg.n_shared)
    secs += time.perf_counter() - t0
    return secs, run, y


def device_expert_getter(cfg, dev):
    """Expert e's weights copied from the synthetic device inputs (the same bits the host
    generator draws) into host arrays."""
    import synth

    import torch

    def h(t, e):
        if t is None:
            return None
        if t.dtype == torch.bfloat16:
            return t[e].view(torch.int16).cpu().numpy().view("uint16")
        return t[e].cpu().numpy()

    def get(e):
        return synth.ExpertWeights(h(dev["w13"], e), h(dev["w2"], e), h(dev["s13"], e),
                                   h(dev["s2"], e))
    return get


def cpu_baseline_full_layer(cfg, dev) -> dict:
    """The oracle's whole layer on the full batch of the workload (every token), weights from
    the device inputs."""
    import torch

    import synth
    cores = oracle_threads()
    x = dev["x"].view(torch.int16).cpu().numpy().view("uint16")
    secs, run, _ = oracle_layer_seconds(cfg, x, synth.host_wg(cfg), synth.host_bias(cfg),
                                        device_expert_getter(cfg, dev))
    return {"value": cfg.T / secs, "unit": "tokens/s", "cores": cores, "kind": "oracle",
            "seconds": secs,
            "sample": (f"one whole layer of the workload, all {cfg.T} tokens: fp32 router over "
                       f"{cfg.E} experts, top-{cfg.k}, permutation, fp64 SwiGLU of the {run} "
                       f"experts run (hit + shared) on their rows, combine; weight copies to the "
                       f"host not timed")}


def run_reference(args, cfg, rank):
    """The CPU oracle as the reference arm: each step is the oracle's whole layer on a sample of
    the workload's tokens (the first n of the batch, every step the same), sized so that the
    whole run of warm-up and timed steps takes a few minutes; the weights of the experts that
    sample hits are drawn on the host once, before the first step."""
    if rank != 0:
        return
    import numpy as np

    import synth
    cores = oracle_threads()
    wg, bias = synth.host_wg(cfg), synth.host_bias(cfg)
    cache = {}

    def get(e):
        if e not in cache:
            cache[e] = synth.host_expert(cfg, e)
        return cache[e]

    # size the sample: seconds per token from one token (drawing its experts' weights on the
    # way), then n tokens per step for ~120 s over all steps, at most 8 tokens (host memory
    # for the weights of the experts they hit) and at most the batch
    x1 = synth.host_x(cfg, tokens=range(1))
    per_tok, _, _ = oracle_layer_seconds(cfg, x1, wg, bias, get)
    budget = 120.0 / max(1, args.steps + args.warmup)
    n = int(max(1, min(cfg.T, 8, budget / max(per_tok, 1e-9))))
    x = synth.host_x(cfg, tokens=range(n))
    times = []
    run = 0
    for i in range(args.warmup + args.steps):
        secs, run, y = oracle_layer_seconds(cfg, x, wg, bias, get)
        assert np.all(np.isfinite(y))
        if i >= args.warmup:
            times.append(secs)
    ms = statistics.mean(times) * 1e3
    value = n / (ms * 1e-3)
    sample = (f"first {n} of the {cfg.T} tokens each step, through the oracle's whole layer: "
              f"fp32 router over {cfg.E} experts, top-{cfg.k}, permutation, fp64 SwiGLU of the "
              f"{run} experts they hit (+ shared), combine")
    out = {"impl": "reference", "metric": METRIC, "value": value, "unit": "tokens/s",
           "n_gpus": args.gpus, "steps": args.steps, "warmup": args.warmup, "ms_per_step": ms,
           "higher_is_better": True, "scaling": "weak", "vs_baseline": None, "dtype": "f64",
           "data": "synthetic",
           "config": config_record(cfg, sample_tokens_per_step=n),
           "cpu_baseline": {"value": value, "unit": "tokens/s", "cores": cores, "kind": "oracle",
                            "sample": sample},
           "e2e": {"value": value, "unit": "tokens/s", "h2d_bytes_per_step": 0,
                   "d2h_bytes_per_step": 0}}
    print(json.dumps(out), flush=True)


# ---------------------------------------------------------------------------------------------
# GPU arm
# ---------------------------------------------------------------------------------------------

def load_config(name, T=None, E=None):
    import dataclasses

    import synth
    over = {k: v for k, v in (("T", T), ("E", E)) if v is not None}
    cfg = synth.get_config(name, **over)
    if over:
        cfg = dataclasses.replace(cfg, name=cfg.name + "".join(f"_{k}{v}" for k, v in over.items()))
    return cfg


def graph_passes(steps, passes, graph=True, exact=True) -> int:
    """Layer passes per replay of the timed graph: 1 without a graph; with exact (the headline,
    whose K passes are timed exactly), the largest divisor of steps up to the requested count."""
    if not graph:
        return 1
    passes = max(1, passes)
    if exact and steps % passes:
        passes = max(p for p in range(1, passes + 1) if steps % p == 0)
    return passes


def measure(cfg, steps, warmup, graph=True, e2e_steps=None, min_ms=None, keep_inputs=False,
            passes=1):
    """Times `steps` layer passes of one workload (CUDA events on the launching stream, inputs
    resident in HBM), then the gate/up and down phases averaged over as many replays, then the
    end-to-end loop. With min_ms, steps grows until the timed region lasts about min_ms. With
    passes > 1 the timed graph holds that many passes back to back (as a model's layers follow
    one another in one graph)."""
    import torch

    import routed_expert_ffn_moe_gb300 as moe
    import synth
    from routed_expert_ffn_moe_gb300 import roofline as R

    dev = synth.device_inputs(cfg)
    w = {k: dev[k] for k in ("wg", "bias", "w13", "w2", "s13", "s2")}
    x = dev["x"]                       # the layer's input buffer (also the e2e copy target)
    layer = moe.MoeLayer(cfg.T, cfg.d, cfg.E, cfg.k, cfg.f, cfg.n_shared, cfg.wdtype, w)
    stream = torch.cuda.current_stream()

    for _ in range(warmup):
        layer.forward(x)
    torch.cuda.synchronize()
    moe.moe_check_device_status(layer.ws)

    # One step = one layer pass (one moe_forward call), captured into a CUDA graph (the library
    # enqueues no synchronisation or allocation) and replayed; the graph holds `passes` of them.
    # The timed graph holds the layer's kernels alone (an event recorded between two kernels
    # would cut the programmatic launch overlap between them); a second graph of one pass,
    # captured with the library's phase events, times the gate/up and down passes.
    g = gp = g1 = None
    passes = graph_passes(steps, passes, graph, exact=not min_ms)
    moe.moe_profile_enable(True)    # resets the launch counter
    moe.moe_profile_enable(False)   # no phase events; launches are still counted
    if graph:
        g = torch.cuda.CUDAGraph()
        with torch.cuda.graph(g):
            for _ in range(passes):
                layer.forward(x)
        launches_per_step = moe.moe_profile_read()["kernel_launches"] // passes
        g1 = g
        if passes > 1:  # one pass a step for the end-to-end loop
            g1 = torch.cuda.CUDAGraph()
            with torch.cuda.graph(g1):
                layer.forward(x)
        moe.moe_profile_enable(True)
        gp = torch.cuda.CUDAGraph()
        with torch.cuda.graph(gp):
            layer.forward(x)
        moe.moe_profile_enable(False)
        for gr in (g, gp):
            for _ in range(2):
                gr.replay()
        torch.cuda.synchronize()
    else:
        layer.forward(x)
        torch.cuda.synchronize()
        launches_per_step = moe.moe_profile_read()["kernel_launches"]
        moe.moe_profile_enable(False)

    def step():
        if g is not None:
            g.replay()
        else:
            layer.forward(x)

    if min_ms:
        s0, s1 = torch.cuda.Event(enable_timing=True), torch.cuda.Event(enable_timing=True)
        s0.record(stream)
        for _ in range(3):
            step()
        s1.record(stream)
        torch.cuda.synchronize()
        est = s0.elapsed_time(s1) / (3 * passes)
        steps = int(min(5000, max(steps, math.ceil(min_ms / max(est, 1e-3)))))
    replays = -(-steps // passes)
    steps = replays * passes

    start, end = torch.cuda.Event(enable_timing=True), torch.cuda.Event(enable_timing=True)
    with ClockSampler(torch.cuda.current_device()) as clocks:
        torch.cuda.synchronize()
        t_host0 = time.time()
        start.record(stream)
        for _ in range(replays):
            step()
        end.record(stream)
        torch.cuda.synchronize()
        clocks.mark_timed(t_host0, time.time())
        ms = start.elapsed_time(end) / steps
        moe.moe_check_device_status(layer.ws)

        # Phases of the FFN (gate/up and down) averaged over `steps` more passes: each pass is
        # read back before the next so that every pass's own events are counted.
        # (The phase graph replays the events captured with it; eager passes get fresh ones.)
        up = dn = 0.0
        for _ in range(steps):
            if gp is not None:
                gp.replay()
            else:
                moe.moe_profile_enable(True)
                layer.forward(x)
            p = moe.moe_profile_read()
            up += p["ms_gate_up"] / max(1, p["ffn_calls"])
            dn += p["ms_down"] / max(1, p["ffn_calls"])
        moe.moe_profile_enable(False)
        ms_up, ms_dn = up / steps, dn / steps

        # End to end: pinned host x -> device, the layer, y -> pinned host, every step (one pass
        # a step).
        e2e_steps = e2e_steps or max(3, steps // 4)
        x_host = torch.empty(x.shape, dtype=x.dtype, pin_memory=True)
        x_host.copy_(x)
        y_host = torch.empty(layer.y.shape, dtype=layer.y.dtype, pin_memory=True)
        torch.cuda.synchronize()
        e0, e1 = torch.cuda.Event(enable_timing=True), torch.cuda.Event(enable_timing=True)
        e0.record(stream)
        for _ in range(e2e_steps):
            x.copy_(x_host, non_blocking=True)
            if g1 is not None:
                g1.replay()
            else:
                layer.forward(x)
            y_host.copy_(layer.y, non_blocking=True)
        e1.record(stream)
        torch.cuda.synchronize()
        ms_e2e = e0.elapsed_time(e1) / e2e_steps
    moe.moe_check_device_status(layer.ws)

    # ---- roofline of the dominant kernel (expert gate/up) and of the layer ---------------
    off = layer.expert_offsets.cpu().tolist()
    n_hit = sum(1 for e in range(cfg.E) if off[e + 1] > off[e])
    # In prefill-sized batches moe_forward runs the shared expert on a second stream beside the
    # routed path, and the phase events time the routed passes alone.
    overlap = cfg.n_shared == 1 and cfg.T > 0 and cfg.T * cfg.k > 32 * cfg.E
    n_run = n_hit + (0 if overlap else cfg.n_shared)
    slots_run = cfg.T * cfg.k + (0 if overlap else cfg.n_shared * cfg.T)
    peaks, peak_src = measured_peaks()
    hbm = float(peaks["hbm_gbs"])
    tc_peak = float(peaks.get("bf16_tflops_sustained", FALLBACK_BF16_TFLOPS_SUSTAINED)) * 1e12
    up_bytes = R.gate_up_bytes(cfg.d, cfg.f, cfg.wdtype, n_run)
    up_flops = 2.0 * slots_run * 2 * cfg.f * cfg.d
    layer_bytes = R.layer_bytes(cfg.T, cfg.d, cfg.E, cfg.f, cfg.n_shared, cfg.wdtype, n_hit)
    layer_flops = R.layer_flops(cfg.T, cfg.d, cfg.E, cfg.k, cfg.f, cfg.n_shared)
    t_floor = R.roofline_time(layer_flops, layer_bytes, tc_peak, hbm * 1e9)
    hbm_bound = layer_bytes / (hbm * 1e9) >= layer_flops / tc_peak
    # The dominant kernel is the gate/up pass. Where the layer is HBM-bound it is rated by its
    # algorithmic bytes against the measured copy bandwidth; where the layer is tensor-bound, by
    # its FLOPs (2 * slots * 2f * d) against the sustained bf16 tensor peak (FP8 and MXFP4
    # prefill tiles dequantise on chip and run bf16 or f16 MMAs).
    kern = "expert gate/up (SiLU x up fused)" + ("; routed experts only (the shared expert "
                                                 "runs beside it)" if overlap else "")
    if hbm_bound:
        achieved = up_bytes / (ms_up * 1e-3) / 1e9 if ms_up > 0 else 0.0
        roof = {"bound": "hbm", "kernel": kern, "achieved": achieved, "peak": hbm,
                "unit": "GB/s", "frac": achieved / hbm, "peak_source": peak_src,
                "algorithmic_bytes_per_launch": up_bytes, "launch_us": ms_up * 1e3}
    else:
        tflops = up_flops / (ms_up * 1e-3) / 1e12 if ms_up > 0 else 0.0
        roof = {"bound": "tensor", "kernel": kern, "achieved": tflops, "peak": tc_peak / 1e12,
                "unit": "TFLOP/s", "frac": tflops * 1e12 / tc_peak,
                "peak_source": peak_src + " (sustained bf16)",
                "algorithmic_flops_per_launch": up_flops,
                "algorithmic_bytes_per_launch": up_bytes, "launch_us": ms_up * 1e3}
    res = {
        "cfg": cfg, "ms": ms, "ms_e2e": ms_e2e, "steps": steps, "e2e_steps": e2e_steps,
        "n_hit": n_hit, "launches_per_step": launches_per_step,
        "graph": g is not None, "graph_passes": passes,
        "layer": {"us": ms * 1e3, "algorithmic_bytes": layer_bytes, "flops": layer_flops,
                  "achieved_GBps": layer_bytes / (ms * 1e-3) / 1e9,
                  "achieved_TFLOPs": layer_flops / (ms * 1e-3) / 1e12,
                  "roofline_frac": t_floor / (ms * 1e-3),
                  "roofline_bound": "hbm" if hbm_bound else "tensor"},
        "phases_us": {"gate_up": ms_up * 1e3, "down": ms_dn * 1e3, "replays_averaged": steps},
        "roofline": roof,
        "e2e": {"value": cfg.T / (ms_e2e * 1e-3), "unit": "tokens/s",
                "h2d_bytes_per_step": x.numel() * x.element_size(),
                "d2h_bytes_per_step": layer.y.numel() * layer.y.element_size()},
        "clocks": clocks.summary(),
    }
    if keep_inputs:
        res["dev"] = dev
    del g, gp, g1, layer, w, x, x_host, y_host
    if not keep_inputs:
        del dev
    torch.cuda.synchronize()
    torch.cuda.empty_cache()
    return res


def sweep_point(r) -> dict:
    cfg = r["cfg"]
    roof = r["roofline"]
    return {"workload": cfg.name, "T": cfg.T, "weights": cfg.wdtype, "router": cfg.router,
            "us_per_layer": r["layer"]["us"], "tokens_per_s": cfg.T / (r["ms"] * 1e-3),
            "layer_roofline_frac": r["layer"]["roofline_frac"],
            "layer_bound": r["layer"]["roofline_bound"],
            "layer_GBps": r["layer"]["achieved_GBps"],
            "layer_TFLOPs": r["layer"]["achieved_TFLOPs"],
            "gate_up": {"us": r["phases_us"]["gate_up"], "bound": roof["bound"],
                        "achieved": roof["achieved"], "unit": roof["unit"], "frac": roof["frac"]},
            "down_us": r["phases_us"]["down"],
            "e2e_tokens_per_s": r["e2e"]["value"], "steps": r["steps"],
            "experts_hit": r["n_hit"], "clocks": r["clocks"]}


def main():
    args = parse_args()
    rank = int(os.environ.get("RANK", "0"))
    world = int(os.environ.get("WORLD_SIZE", "1"))
    cfg = load_config(args.config, args.T, args.E)
    if args.impl == "reference":
        run_reference(args, cfg, rank)
        return
    if args.gpus != 1 or world != 1:
        sys.stderr.write("bench.py: this library runs on one GPU; run it with --gpus 1 "
                         "(no torchrun)\n")
        sys.exit(2)

    import torch

    import routed_expert_ffn_moe_gb300 as moe
    from routed_expert_ffn_moe_gb300 import build as moe_build

    torch.cuda.set_device(0)
    moe_build.build()
    moe.load()

    want_cpu = not args.no_cpu_baseline
    r = measure(cfg, args.steps, args.warmup, graph=not args.no_graph, e2e_steps=args.e2e_steps,
                keep_inputs=want_cpu, passes=args.graph_passes)
    roof = dict(r["roofline"])
    roof["traffic"] = ncu_traffic(cfg.name)
    out = {
        "metric": METRIC, "value": cfg.T / (r["ms"] * 1e-3), "unit": "tokens/s", "n_gpus": 1,
        "steps": r["steps"], "warmup": args.warmup, "ms_per_step": r["ms"],
        "higher_is_better": True, "scaling": "weak", "vs_baseline": None,
        "dtype": dtype_of(cfg), "data": "synthetic",
        "config": config_record(
            cfg,
            launch=(f"CUDA graph replay of {r['graph_passes']} moe_forward call(s) back to back"
                    if r["graph"] else "eager"),
            l2="inputs larger than L2 (expert weights "
               f"{(cfg.E + cfg.n_shared) * moe_roofline_expert_bytes(cfg) / 1e9:.1f} GB), no flush",
            experts_hit=r["n_hit"], layer=r["layer"], phases_us=r["phases_us"]),
        "roofline": roof,
        "e2e": r["e2e"],
        "gpu_launches": r["launches_per_step"] * r["steps"],
        "clocks": r["clocks"],
    }
    if want_cpu:
        out["cpu_baseline"] = cpu_baseline_full_layer(cfg, r["dev"])
    r = None
    torch.cuda.empty_cache()
    sweep = []
    for name in SWEEPS[args.sweep]:
        sc = load_config(name)
        sweep.append(sweep_point(measure(sc, args.steps, args.warmup, graph=not args.no_graph,
                                         min_ms=args.sweep_min_ms, passes=args.graph_passes)))
    out["sweep"] = sweep
    print(json.dumps(out), flush=True)


def moe_roofline_expert_bytes(cfg) -> int:
    from routed_expert_ffn_moe_gb300 import roofline as R
    return R.expert_bytes(cfg.d, cfg.f, cfg.wdtype)


if __name__ == "__main__":
    main()
