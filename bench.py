#!/usr/bin/env python
"""Benchmark of the routed-expert MoE FFN layer (router, permute, expert SwiGLU FFN, combine +
shared expert) on GB300, through the library's C ABI.

One step = one pass of the whole layer over one batch of T tokens, inputs already in HBM.
Prints one JSON line (rank 0). Default workload: the DeepSeek-V3-shaped decode layer (T=256,
d=7168, 256 routed + 1 shared experts, top-8, f=2048, bf16 weights).

  python bench.py [--gpus N] [--steps K] [--warmup W] [--config NAME] [--impl ours|reference]

N > 1 runs N independent replicas (one per GPU, launched by torchrun): the layer does not
shard on one node without an exchange this build does not implement, so per-GPU work is fixed
("weak" scaling) and the value is the sum over GPUs.
--impl reference times the CPU oracle on the host cores instead (rank 0 only).
"""
from __future__ import annotations

import argparse
import hashlib
import json
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


def parse_args(argv=None):
    p = argparse.ArgumentParser()
    p.add_argument("--gpus", type=int, default=1)
    p.add_argument("--steps", type=int, default=200)
    p.add_argument("--warmup", type=int, default=10)
    p.add_argument("--config", default="v3_decode")
    p.add_argument("--impl", choices=("ours", "reference"), default="ours")
    p.add_argument("--no-cpu-baseline", action="store_true")
    p.add_argument("--no-graph", action="store_true",
                   help="launch the four calls eagerly each step instead of replaying a CUDA graph")
    p.add_argument("--e2e-steps", type=int, default=None)
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


def measured_peaks():
    path = os.path.join(ROOT, "MEASURED_PEAKS.json")
    try:
        with open(path) as fh:
            return json.load(fh), "measured"
    except (OSError, ValueError):
        return {"hbm_gbs": FALLBACK_HBM_GBS, "bf16_tflops": FALLBACK_BF16_TFLOPS,
                "bf16_tflops_sustained": 1700.0}, "fallback"


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
    """nvidia-smi clocks/throttle reasons sampled every 100 ms during the timed region."""
    Q = ("index,clocks.sm,clocks.max.sm,power.draw,clocks_event_reasons.active,"
         "clocks_event_reasons.hw_slowdown,clocks_event_reasons.hw_thermal_slowdown,"
         "clocks_event_reasons.sw_thermal_slowdown,clocks_event_reasons.sw_power_cap")

    def __init__(self, dev_index: int):
        self.proc = None
        self.dev = dev_index

    def __enter__(self):
        try:
            import torch
            uuid = str(torch.cuda.get_device_properties(self.dev).uuid)
            sel = ["-i", uuid if uuid.startswith("GPU-") else "GPU-" + uuid]
        except Exception:
            sel = []
        try:
            self.proc = subprocess.Popen(["nvidia-smi", "--query-gpu=" + self.Q,
                                          "--format=csv,noheader,nounits", "-lms", "100"] + sel,
                                         stdout=subprocess.PIPE, stderr=subprocess.DEVNULL, text=True)
        except OSError:
            self.proc = None
        return self

    def __exit__(self, *exc):
        self.lines = []
        if self.proc is not None:
            time.sleep(0.15)
            self.proc.terminate()
            try:
                out, _ = self.proc.communicate(timeout=5)
            except subprocess.TimeoutExpired:
                self.proc.kill()
                out, _ = self.proc.communicate()
            self.lines = [ln for ln in out.splitlines() if ln.strip()]
        return False

    def summary(self):
        sm, mx, reasons = [], [], set()
        names = ["hw_slowdown", "hw_thermal_slowdown", "sw_thermal_slowdown", "sw_power_cap"]
        for ln in getattr(self, "lines", []):
            parts = [p.strip() for p in ln.split(",")]
            if len(parts) < 9:
                continue
            try:
                sm.append(float(parts[1]))
                mx.append(float(parts[2]))
            except ValueError:
                continue
            for nm, v in zip(names, parts[5:9]):
                if v.lower() == "active":
                    reasons.add(nm)
        if not sm:
            return {"sm_mhz": None, "sm_max_mhz": None, "reasons": [], "samples": 0}
        return {"sm_mhz": statistics.median(sm), "sm_max_mhz": max(mx), "reasons": sorted(reasons),
                "samples": len(sm)}


# ---------------------------------------------------------------------------------------------
# CPU oracle (baseline leg and --impl reference)
# ---------------------------------------------------------------------------------------------

_ORACLE_INPUTS = {}


def _oracle_inputs(cfg):
    """Router weight, bias and the shared expert's weights on the host (drawn once)."""
    if cfg.name not in _ORACLE_INPUTS:
        import synth
        _ORACLE_INPUTS[cfg.name] = (synth.host_wg(cfg), synth.host_bias(cfg),
                                    synth.host_expert(cfg, cfg.E if cfg.n_shared else 0))
    return _ORACLE_INPUTS[cfg.name]


def oracle_sample_rate(cfg, budget_s: float):
    """Tokens/s of the CPU oracle on this workload, from a bounded sample: n tokens through the
    router and through the shared expert's SwiGLU FFN (every expert has the same size, so one
    token of the layer costs the router plus k+1 expert FFNs). Returns (tokens/s, sample, cores,
    seconds spent)."""
    os.environ.setdefault("OMP_NUM_THREADS", str(os.cpu_count() or 1))
    import oracle
    import synth
    cores = int(os.environ["OMP_NUM_THREADS"])
    wg, bias, ew = _oracle_inputs(cfg)

    def run(n):
        x = synth.host_x(cfg, tokens=range(n))
        t0 = time.perf_counter()
        logits = oracle.router_logits(x, wg, bias)
        oracle.route(logits, cfg.k)
        t1 = time.perf_counter()
        oracle.expert_rows(x, ew.w13, ew.w2, cfg.wdtype, ew.s13, ew.s2)
        t2 = time.perf_counter()
        return t1 - t0, t2 - t1

    r1, f1 = run(1)
    n = int(max(1, min(cfg.T, budget_s / max(r1 + f1, 1e-9))))
    tr, tf = run(n)
    secs = tr + (cfg.k + cfg.n_shared) * tf
    sample = (f"first {n} of {cfg.T} tokens: fp32 router + top-k over all {cfg.E} experts, and one "
              f"fp64 SwiGLU expert FFN per token timed and scaled by the k+{cfg.n_shared}="
              f"{cfg.k + cfg.n_shared} equal-size experts each token runs")
    return n / secs, sample, cores, tr + tf


def run_reference(args, cfg, rank):
    if rank != 0:
        return
    per_step_budget = max(0.3, min(3.0, 150.0 / max(1, args.steps + args.warmup)))
    rates = []
    t_all = []
    sample = cores = None
    for i in range(args.warmup + args.steps):
        rate, sample, cores, secs = oracle_sample_rate(cfg, per_step_budget)
        if i >= args.warmup:
            rates.append(rate)
            t_all.append(cfg.T / rate * 1e3)
    value = statistics.median(rates)
    out = {"impl": "reference", "metric": METRIC, "value": value, "unit": "tokens/s",
           "n_gpus": args.gpus, "steps": args.steps, "warmup": args.warmup,
           "ms_per_step": statistics.median(t_all), "higher_is_better": True, "scaling": "weak",
           "vs_baseline": None, "dtype": "f64", "data": "synthetic",
           "config": {"workload": workload_desc(cfg)},
           "cpu_baseline": {"value": value, "unit": "tokens/s", "cores": cores, "kind": "oracle",
                            "sample": sample},
           "e2e": {"value": value, "unit": "tokens/s", "h2d_bytes_per_step": 0,
                   "d2h_bytes_per_step": 0}}
    print(json.dumps(out), flush=True)


# ---------------------------------------------------------------------------------------------
# replicas: every rank times its own layer; the job's time is the slowest rank's
# ---------------------------------------------------------------------------------------------

def max_over_ranks(values, dist, device):
    """Element-wise maximum of `values` (floats) over all ranks of the process group."""
    import torch
    t = torch.tensor([float(v) for v in values], dtype=torch.float64, device=device)
    dist.all_reduce(t, op=dist.ReduceOp.MAX)
    return [float(v) for v in t.tolist()]


def job_tokens_per_s(tokens_per_rank: int, world: int, ms: float) -> float:
    """Whole-job throughput: every rank processes its own batch in (at most) `ms`."""
    return world * tokens_per_rank / (ms * 1e-3)


# ---------------------------------------------------------------------------------------------
# GPU arm
# ---------------------------------------------------------------------------------------------

def main():
    args = parse_args()
    rank = int(os.environ.get("RANK", "0"))
    world = int(os.environ.get("WORLD_SIZE", "1"))
    local_rank = int(os.environ.get("LOCAL_RANK", "0"))
    import synth
    over = {k: v for k, v in (("T", args.T), ("E", args.E)) if v is not None}
    cfg = synth.get_config(args.config, **over)
    if over:
        import dataclasses
        cfg = dataclasses.replace(cfg, name=cfg.name + "".join(f"_{k}{v}" for k, v in over.items()))
    if args.impl == "reference":
        run_reference(args, cfg, rank)
        return

    import torch
    import torch.distributed as dist

    import routed_expert_ffn_moe_gb300 as moe
    from routed_expert_ffn_moe_gb300 import build as moe_build
    from routed_expert_ffn_moe_gb300 import roofline as R

    torch.cuda.set_device(local_rank)
    if world > 1:
        dist.init_process_group("nccl", device_id=torch.device("cuda", local_rank))
    moe_build.build()
    moe.load()

    dev = synth.device_inputs(cfg)
    w = {k: dev[k] for k in ("wg", "bias", "w13", "w2", "s13", "s2")}
    x = dev["x"]                       # the layer's input buffer (also the e2e copy target)
    layer = moe.MoeLayer(cfg.T, cfg.d, cfg.E, cfg.k, cfg.f, cfg.n_shared, cfg.wdtype, w)
    stream = torch.cuda.current_stream()

    for _ in range(args.warmup):
        layer.forward(x)
    torch.cuda.synchronize()
    moe.moe_check_device_status(layer.ws)

    def barrier():
        if world > 1:
            dist.barrier()
        torch.cuda.synchronize()

    # One step = one layer pass (one moe_forward call). By default it is captured once into a CUDA graph
    # (the library enqueues no synchronisation or allocation) and the graph is replayed; the
    # library's phase events are captured with it and re-recorded by every replay.
    graph = None
    if not args.no_graph:
        moe.moe_profile_enable(True)
        graph = torch.cuda.CUDAGraph()
        with torch.cuda.graph(graph):
            layer.forward(x)
        for _ in range(2):
            graph.replay()
        torch.cuda.synchronize()
        launches_per_step = moe.moe_profile_read()["kernel_launches"]  # counted at capture

    def step():
        if graph is not None:
            graph.replay()
        else:
            layer.forward(x)

    # ---- timed region: K steps on device-resident inputs --------------------------------
    start, end = torch.cuda.Event(enable_timing=True), torch.cuda.Event(enable_timing=True)
    barrier()
    with ClockSampler(local_rank) as clocks:
        if graph is None:
            moe.moe_profile_enable(True)
        start.record(stream)
        for _ in range(args.steps):
            step()
        end.record(stream)
        torch.cuda.synchronize()
        moe.moe_profile_enable(False)
    barrier()
    ms = start.elapsed_time(end) / args.steps
    prof = moe.moe_profile_read()
    if graph is not None:  # phase events hold the last replay; launches counted at capture
        prof["kernel_launches"] = launches_per_step * args.steps
    moe.moe_check_device_status(layer.ws)

    # ---- end to end: pinned host x -> device, the layer, y -> pinned host ----------------
    e2e_steps = args.e2e_steps or max(3, args.steps // 4)
    x_host = torch.empty(x.shape, dtype=x.dtype, pin_memory=True)
    x_host.copy_(x)
    y_host = torch.empty(layer.y.shape, dtype=layer.y.dtype, pin_memory=True)
    barrier()
    e0, e1 = torch.cuda.Event(enable_timing=True), torch.cuda.Event(enable_timing=True)
    e0.record(stream)
    for _ in range(e2e_steps):
        x.copy_(x_host, non_blocking=True)
        step()
        y_host.copy_(layer.y, non_blocking=True)
    e1.record(stream)
    torch.cuda.synchronize()
    barrier()
    ms_e2e = e0.elapsed_time(e1) / e2e_steps

    if world > 1:
        ms, ms_e2e = max_over_ranks([ms, ms_e2e], dist, "cuda")

    # ---- roofline of the dominant kernel (expert gate/up) and of the layer ---------------
    off = layer.expert_offsets.cpu().tolist()
    counts = [off[e + 1] - off[e] for e in range(cfg.E)]
    n_hit = sum(1 for c in counts if c > 0)
    n_run = n_hit + cfg.n_shared
    peaks, peak_src = measured_peaks()
    hbm = float(peaks["hbm_gbs"])
    calls = max(1, prof["ffn_calls"])
    ms_up = prof["ms_gate_up"] / calls
    ms_dn = prof["ms_down"] / calls
    up_bytes = R.gate_up_bytes(cfg.d, cfg.f, cfg.wdtype, n_run)
    dn_bytes = R.down_bytes(cfg.d, cfg.f, cfg.wdtype, n_run)
    achieved = up_bytes / (ms_up * 1e-3) / 1e9
    traffic = ncu_traffic(cfg.name)
    layer_bytes = R.layer_bytes(cfg.T, cfg.d, cfg.E, cfg.f, cfg.n_shared, cfg.wdtype, n_hit)
    layer_flops = R.layer_flops(cfg.T, cfg.d, cfg.E, cfg.k, cfg.f, cfg.n_shared)
    tc_peak = float(peaks.get("bf16_tflops_sustained", FALLBACK_BF16_TFLOPS)) * 1e12
    t_floor = R.roofline_time(layer_flops, layer_bytes, tc_peak, hbm * 1e9)

    value = job_tokens_per_s(cfg.T, world, ms)
    # The dominant kernel is the gate/up pass. Where the layer is HBM-bound it is rated by its
    # algorithmic bytes against the measured copy bandwidth; where the layer is tensor-bound, by
    # its FLOPs (2 * slots * 2f * d) against the sustained bf16 tensor peak (the FP8 weights are
    # dequantised on chip, so the MMAs run in bf16 or f16).
    if layer_bytes / (hbm * 1e9) >= layer_flops / tc_peak:
        roof = {"bound": "hbm", "kernel": "expert gate/up (SiLU x up fused)",
                "achieved": achieved, "peak": hbm, "unit": "GB/s", "frac": achieved / hbm,
                "peak_source": peak_src, "traffic": traffic,
                "algorithmic_bytes_per_launch": up_bytes}
    else:
        up_flops = 2.0 * (cfg.T * cfg.k + cfg.n_shared * cfg.T) * 2 * cfg.f * cfg.d
        tflops = up_flops / (ms_up * 1e-3) / 1e12
        roof = {"bound": "tensor", "kernel": "expert gate/up (SiLU x up fused)",
                "achieved": tflops, "peak": tc_peak / 1e12, "unit": "TFLOP/s",
                "frac": tflops * 1e12 / tc_peak, "peak_source": peak_src + " (sustained bf16)",
                "traffic": traffic, "algorithmic_flops_per_launch": up_flops,
                "algorithmic_bytes_per_launch": up_bytes}
    out = {
        "metric": METRIC, "value": value, "unit": "tokens/s", "n_gpus": world,
        "steps": args.steps, "warmup": args.warmup, "ms_per_step": ms, "higher_is_better": True,
        "scaling": "weak", "vs_baseline": None,
        "dtype": {"bf16": "bf16", "fp8": "fp8_e4m3 weights, bf16 activations",
                  "mxfp4": "mxfp4 (e2m1 + e8m0) weights, bf16 activations as two e4m3 terms"}[cfg.wdtype],
        "data": "synthetic",
        "config": {"workload": workload_desc(cfg), "T": cfg.T, "parallelism": f"replicas x{world}",
                   "launch": "eager" if graph is None else "CUDA graph replay of one moe_forward call",
                   "l2": "inputs larger than L2 (expert weights "
                         f"{(cfg.E + cfg.n_shared) * R.expert_bytes(cfg.d, cfg.f, cfg.wdtype) / 1e9:.1f} GB), no flush",
                   "experts_hit": n_hit,
                   "layer": {"us": ms * 1e3, "algorithmic_bytes": layer_bytes,
                             "flops": layer_flops,
                             "achieved_GBps": layer_bytes / (ms * 1e-3) / 1e9,
                             "achieved_TFLOPs": layer_flops / (ms * 1e-3) / 1e12,
                             "roofline_frac": t_floor / (ms * 1e-3),
                             "roofline_bound": "hbm" if layer_bytes / (hbm * 1e9) >= layer_flops / tc_peak else "tensor"},
                   "phases_us": {"gate_up": ms_up * 1e3, "down": ms_dn * 1e3}},
        "roofline": roof,
        "e2e": {"value": job_tokens_per_s(cfg.T, world, ms_e2e), "unit": "tokens/s",
                "h2d_bytes_per_step": x.numel() * x.element_size(),
                "d2h_bytes_per_step": layer.y.numel() * layer.y.element_size()},
        "gpu_launches": prof["kernel_launches"],
        "clocks": clocks.summary(),
    }
    if rank == 0 and world == 1 and not args.no_cpu_baseline:
        rate, sample, cores, _ = oracle_sample_rate(cfg, 12.0)
        out["cpu_baseline"] = {"value": rate, "unit": "tokens/s", "cores": cores, "kind": "oracle",
                               "sample": sample}
    if rank == 0:
        print(json.dumps(out), flush=True)
    if world > 1:
        dist.destroy_process_group()


if __name__ == "__main__":
    main()
