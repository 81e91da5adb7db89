"""bench.py's host-side logic on CPU: it refuses more than one GPU before touching one, the
reference arm (the CPU oracle) prints one line on rank 0 only, the clock sampler reads
nvidia-smi's lines and tells the samples inside the timed region from the rest, and the timed
graph's passes per replay keep the headline's pass count exact."""
import datetime
import json
import os
import subprocess
import sys

ROOT = os.path.dirname(os.path.dirname(os.path.abspath(__file__)))


def run_bench(args, env_extra=None, timeout=300):
    env = dict(os.environ, **(env_extra or {}))
    return subprocess.run([sys.executable, os.path.join(ROOT, "bench.py")] + args, cwd=ROOT,
                          env=env, capture_output=True, text=True, timeout=timeout)


def test_more_than_one_gpu_is_refused_before_any_gpu_work():
    r = run_bench(["--gpus", "2"])
    assert r.returncode == 2 and "one GPU" in r.stderr and r.stdout == ""
    r = run_bench(["--gpus", "1"], {"WORLD_SIZE": "2", "RANK": "0"})
    assert r.returncode == 2 and "one GPU" in r.stderr


def test_reference_arm_prints_one_line_on_rank_0_only():
    args = ["--impl", "reference", "--config", "tiny", "--steps", "2", "--warmup", "1"]
    r = run_bench(args)
    assert r.returncode == 0, r.stderr
    lines = [ln for ln in r.stdout.splitlines() if ln.strip()]
    assert len(lines) == 1
    out = json.loads(lines[0])
    assert out["impl"] == "reference" and out["value"] > 0 and out["steps"] == 2
    assert out["unit"] == "tokens/s" and out["cpu_baseline"]["kind"] == "oracle"
    assert out["e2e"]["h2d_bytes_per_step"] == 0
    assert out["config"]["T"] == 16 and out["config"]["sample_tokens_per_step"] >= 1
    # one step is one whole oracle layer on the sample: tokens / step time
    n = out["config"]["sample_tokens_per_step"]
    assert abs(out["value"] - n / (out["ms_per_step"] * 1e-3)) <= 1e-6 * out["value"]
    r1 = run_bench(args, {"RANK": "1", "WORLD_SIZE": "2"})
    assert r1.returncode == 0 and r1.stdout.strip() == ""


def test_clock_summary_separates_the_timed_region():
    sys.path.insert(0, ROOT)
    import bench
    base = datetime.datetime(2026, 1, 2, 3, 4, 5)

    def line(sec, mhz, power_cap=False, thermal=False):
        ts = (base + datetime.timedelta(seconds=sec)).strftime("%Y/%m/%d %H:%M:%S.%f")[:-3]
        act = "Active" if power_cap else "Not Active"
        th = "Active" if thermal else "Not Active"
        return f"{ts}, 0, {mhz}, 2070, 900.0, 0x0, Not Active, {th}, Not Active, {act}"

    cs = bench.ClockSampler(0)
    cs.lines = [line(0.0, 1000), line(1.0, 2070), line(1.1, 2055, power_cap=True),
                line(2.0, 1500, thermal=True), "garbage"]
    t0 = (base + datetime.timedelta(seconds=0.95)).timestamp()
    cs.mark_timed(t0, t0 + 0.2)
    s = cs.summary()
    assert s["samples"] == 4 and s["samples_in_timed_region"] == 2
    assert s["timed_region"]["sm_mhz"] == (2070 + 2055) / 2
    assert s["timed_region"]["reasons"] == ["sw_power_cap"]
    assert s["reasons"] == ["hw_thermal_slowdown", "sw_power_cap"] and s["sm_max_mhz"] == 2070


def test_graph_passes_keep_the_timed_pass_count_exact():
    sys.path.insert(0, ROOT)
    import bench
    assert bench.graph_passes(200, 8) == 8
    assert bench.graph_passes(20, 8) == 5        # 4 replays of 5 passes
    assert bench.graph_passes(7, 8) == 7
    assert bench.graph_passes(13, 8) == 1        # a prime above 8: one pass a replay
    assert bench.graph_passes(12, 8, graph=False) == 1
    assert bench.graph_passes(13, 8, exact=False) == 8   # sweep points round up instead
    for k in range(1, 60):
        p = bench.graph_passes(k, 8)
        assert 1 <= p <= 8 and k % p == 0
