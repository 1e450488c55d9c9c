#!/usr/bin/env python3
"""Benchmark of one cascade beam decode step: paged KV append + shared-prefix decode attention.

A step is one layer over the whole batch: bsp_append_kv then bsp_decode_attn (prompt kernel on tensor
cores, which also finishes the requests whose tails it gathers; the tail + log-sum-exp merge kernel for
the others). Default workload: the wide-beam shape (batch 128, beam 96, 16/8 heads, head_dim 128, bf16,
page 32, prompt U{2800..3200}, tail U{0..3}); the line also carries the other decode workloads
(config.configs: steps/s and per-kernel times of each) unless --no-configs.

  python bench.py [--gpus N] [--steps K] [--warmup W] [--impl native|reference]

Prints one JSON line (rank 0). Under torchrun each rank runs its own independent batch (requests
shard across GPUs; nothing is exchanged on the data path) and the time is the max over ranks.
"""
from __future__ import annotations

import argparse
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

import numpy as np  # noqa: E402
import torch  # noqa: E402

METRIC = "beam decode-attn steps/s"
DEFAULT_WORKLOAD = "wide_beam_b128_w96"
PROFILE_TRAFFIC = os.path.join(ROOT, "profiles", "prefix_traffic.json")


def parse():
    ap = argparse.ArgumentParser()
    ap.add_argument("--gpus", type=int, default=1)
    ap.add_argument("--steps", type=int, default=2000)
    ap.add_argument("--warmup", type=int, default=20)
    ap.add_argument("--impl", default="native", choices=["native", "reference"])
    ap.add_argument("--workload", default=DEFAULT_WORKLOAD)
    ap.add_argument("--sets", type=int, default=3, help="rotated input sets (each larger than L2)")
    ap.add_argument("--cpu-seconds", type=float, default=12.0, help="budget of the CPU-oracle sample")
    ap.add_argument("--no-cpu-baseline", action="store_true")
    ap.add_argument("--e2e-steps", type=int, default=50)
    ap.add_argument("--repeats", type=int, default=10, help="timed replays of the K steps (at least 10)")
    ap.add_argument("--no-configs", action="store_true", help="skip the other workloads of the line")
    return ap.parse_args()


# ---------------------------------------------------------------- distributed plumbing (host only)
def dist_init(args):
    world = int(os.environ.get("WORLD_SIZE", "1"))
    rank = int(os.environ.get("RANK", "0"))
    local = int(os.environ.get("LOCAL_RANK", "0"))
    if world > 1:
        import torch.distributed as dist
        backend = "nccl" if torch.cuda.is_available() else "gloo"
        if torch.cuda.is_available():
            torch.cuda.set_device(local)
        dist.init_process_group(backend=backend)
    elif torch.cuda.is_available():
        torch.cuda.set_device(0)
    return rank, world, local


def barrier(world):
    if world > 1:
        import torch.distributed as dist
        dist.barrier()


def reduce_max(x: float, world: int) -> float:
    if world == 1:
        return x
    import torch.distributed as dist
    t = torch.tensor([x], dtype=torch.float64, device="cuda" if torch.cuda.is_available() else "cpu")
    dist.all_reduce(t, op=dist.ReduceOp.MAX)
    return float(t.item())


# ---------------------------------------------------------------- clocks
class ClockSampler:
    FIELDS = ("index,clocks.sm,clocks.max.sm,power.draw,clocks_event_reasons.active,"
              "clocks_event_reasons.hw_slowdown,clocks_event_reasons.hw_thermal_slowdown,"
              "clocks_event_reasons.sw_thermal_slowdown,clocks_event_reasons.sw_power_cap")

    def __init__(self, gpu_index: int):
        self.gpu = gpu_index
        self.proc = None

    def __enter__(self):
        try:
            self.proc = subprocess.Popen(
                ["nvidia-smi", f"--id={self.gpu}", f"--query-gpu={self.FIELDS}", "--format=csv,noheader,nounits",
                 "-lms", "100"], stdout=subprocess.PIPE, stderr=subprocess.DEVNULL, text=True)
        except (OSError, ValueError):
            self.proc = None
        time.sleep(0.3)
        return self

    def __exit__(self, *exc):
        self.result = {"sm_mhz": None, "sm_max_mhz": None, "reasons": [], "samples": 0}
        if self.proc is None:
            return False
        time.sleep(0.25)
        self.proc.terminate()
        try:
            out, _ = self.proc.communicate(timeout=5)
        except subprocess.TimeoutExpired:
            self.proc.kill()
            out, _ = self.proc.communicate()
        sm, smax, reasons = [], [], set()
        names = ["hw_slowdown", "hw_thermal_slowdown", "sw_thermal_slowdown", "sw_power_cap"]
        for line in out.splitlines():
            parts = [p.strip() for p in line.split(",")]
            if len(parts) < 9:
                continue
            try:
                sm.append(float(parts[1]))
                smax.append(float(parts[2]))
            except ValueError:
                continue
            for name, val in zip(names, parts[5:9]):
                if val.lower() == "active":
                    reasons.add(name)
        if sm:
            self.result = {"sm_mhz": statistics.median(sm), "sm_max_mhz": max(smax), "reasons": sorted(reasons),
                           "samples": len(sm)}
        return False


# ---------------------------------------------------------------- peaks / traffic
def measured_peaks():
    path = os.path.join(ROOT, "MEASURED_PEAKS.json")
    if os.path.exists(path):
        with open(path) as f:
            d = json.load(f)
        return float(d["hbm_gbs"]), float(d["bf16_tflops"]), "measured"
    return 6800.0, 1900.0, "fallback"


def kernel_source_hash(kernel_file: str):
    """Hash of the sources a prompt kernel is built from (its own file and the shared device headers)."""
    h = hashlib.sha256()
    for name in (kernel_file, "bsp_ptx.cuh", "bsp_internal.h", "bsp_prompt.cuh"):
        with open(os.path.join(ROOT, "beam_search_shared_gb300", "csrc", name), "rb") as f:
            h.update(f.read())
    return h.hexdigest()[:16]


def profiled_traffic(workload: str, kernel: str, kernel_file: str):
    """DRAM bytes per prompt-kernel launch from the committed ncu record of this workload, if the kernel's
    sources are unchanged since the capture."""
    if not os.path.exists(PROFILE_TRAFFIC):
        return None
    with open(PROFILE_TRAFFIC) as f:
        d = json.load(f)
    for r in d.get("records", []):
        if (r.get("workload") == workload and r.get("kernel", "").startswith(kernel) and
                r.get("kernel_source_sha") == kernel_source_hash(kernel_file)):
            return r.get("dram_bytes_per_launch")
    return None


# ---------------------------------------------------------------- oracle timing (CPU)
class OracleTimer:
    """The fp64 oracle (append scatter + unsplit attention) timed on bounded row samples of one step."""

    def __init__(self, case):
        import oracle
        from beam_search_shared_gb300 import synth
        self.oracle = oracle
        self.case = case
        wl = case.workload
        self.R = wl.batch * wl.beam_width
        self.kp, self.vp = synth.bits(case.k_pool).copy(), synth.bits(case.v_pool).copy()
        self.kn, self.vn = synth.bits(case.k_new), synth.bits(case.v_new)
        self.kw = dict(dtype=wl.dtype, B=wl.batch, W=wl.beam_width, Hq=wl.num_q_heads, Hkv=wl.num_kv_heads,
                       D=wl.head_dim, ps=wl.page_size, num_pages=case.num_pages, prefix_len=case.prefix_len,
                       tail_len=case.tail_len, prefix_pages=case.prefix_pages, beam_pages=case.beam_pages,
                       cache_indirection=case.cache_indirection, q_bits=synth.bits(case.q), k_pool_bits=self.kp,
                       v_pool_bits=self.vp, scale=1 / math.sqrt(wl.head_dim))
        self.rng = np.random.default_rng(0)
        oracle.build()
        cores = len(os.sched_getaffinity(0))
        self.cores = min(cores, int(os.environ.get("OMP_NUM_THREADS", cores)))
        t0 = time.perf_counter()
        self.sample(min(self.R, 8))
        self.per_row = (time.perf_counter() - t0) / min(self.R, 8)

    def rows_for(self, seconds):
        return int(max(1, min(self.R, seconds / max(self.per_row, 1e-9))))

    def sample(self, n):
        rows = np.sort(self.rng.choice(self.R, n, replace=False)).astype(np.int32)
        self.oracle.decode_attn(rows=rows, **self.kw)

    def step_seconds(self, n):
        """One step's time: the append in full plus n of R rows of attention, scaled to all rows."""
        wl = self.case.workload
        t0 = time.perf_counter()
        self.oracle.append_kv(Hkv=wl.num_kv_heads, D=wl.head_dim, ps=wl.page_size, num_pages=self.case.num_pages,
                              out_cache_loc=self.case.out_cache_loc, k_new_bits=self.kn, v_new_bits=self.vn,
                              k_pool_bits=self.kp, v_pool_bits=self.vp)
        t_app = time.perf_counter() - t0
        t0 = time.perf_counter()
        self.sample(n)
        t_attn = time.perf_counter() - t0
        return t_app + t_attn * self.R / n, t_app + t_attn


def cpu_model():
    try:
        out = subprocess.run(["lscpu"], capture_output=True, text=True, timeout=5).stdout
        for line in out.splitlines():
            if line.startswith("Model name"):
                return line.split(":", 1)[1].strip()
    except (OSError, subprocess.TimeoutExpired):
        pass
    return "unknown"


# ---------------------------------------------------------------- main
# prompt kernel of each plan layout, and the sources it is built from (for the traffic record's key)
LAYOUT_KERNEL = {0: ("prefix_attn_kernel", "bsp_prefix.cu"), 1: ("prefix_alt_kernel", "bsp_alt.cu"),
                 2: ("prefix_wide_kernel", "bsp_wide.cu")}
# the other decode workloads reported beside the headline, in the same line
OTHER_CONFIGS = ["qwen3_0p6b_b64_w30", "qwen3_4b_fp16_d128", "qwen3_4b_fp16_d64", "qwen3_4b_fp16_d256"]


def graph_of(fn, n):
    """A CUDA graph of the calls fn(0) .. fn(n - 1)."""
    g = torch.cuda.CUDAGraph()
    with torch.cuda.graph(g):
        for j in range(n):
            fn(j)
    return g


def time_graph(g, reps, stream):
    """Device time (ms) of each of `reps` replays of graph g, one event pair around each replay (after
    one untimed replay)."""
    g.replay()
    torch.cuda.synchronize()
    out = []
    for _ in range(reps):
        e0, e1 = torch.cuda.Event(enable_timing=True), torch.cuda.Event(enable_timing=True)
        e0.record(stream)
        g.replay()
        e1.record(stream)
        torch.cuda.synchronize()
        out.append(e0.elapsed_time(e1))
    return out


class DecodeBench:
    """Rotated input sets of one decode workload (each its own workspace and plan) and the timings of
    a step (append + attention) and of its kernels."""

    def __init__(self, wl, nsets, seed0, dev, **case_kw):
        from beam_search_shared_gb300 import synth
        from beam_search_shared_gb300.step import DeviceStep, algorithmic_bytes
        self.wl = wl
        self.sets = []
        for i in range(nsets):
            case = synth.make_case(wl, seed0 + i, full_step=True, device=dev, **case_kw)
            st = DeviceStep(case, device=dev)
            st.make_plan()
            self.sets.append(st)
        torch.cuda.synchronize()
        self.ab = [algorithmic_bytes(s.case, s.fused_requests()) for s in self.sets]
        self.tail_launch = [s.plan.tail_requests > 0 for s in self.sets]
        self.layout = int(self.sets[0].plan.layout)
        self.stream = torch.cuda.current_stream()

    def set_of(self, j):
        return self.sets[j % len(self.sets)]

    def step(self, j):
        s = self.set_of(j)
        s.append()
        s.attend()

    def warm(self, n):
        from beam_search_shared_gb300 import bsp
        for j in range(n):
            self.step(j)
        torch.cuda.synchronize()
        for s in self.sets:
            assert bsp.read_device_status(s.plan) == (0, 0)

    def launches(self, K):
        return sum(1 + (s.plan.num_units > 0) + (s.plan.tail_requests > 0) for s in (self.set_of(j) for j in range(K)))

    def kernel_times(self, Kt, reps):
        """Per-kernel times (us): the append and the attention each as Kt launches back to back in one
        graph (one event pair around each replay: launch gaps included, no event node between launches),
        medians over `reps` replays; when a set needs the tail kernel, the attention time is the prompt
        and tail kernels together, and their split comes from a replay with an event pair around each
        kernel (an event node delays the next launch: upper bounds)."""
        from beam_search_shared_gb300 import bsp
        out = {}
        g = graph_of(lambda j: self.set_of(j).append(), Kt)
        out["us_append"] = 1e3 * statistics.median(time_graph(g, reps, self.stream)) / Kt
        g = graph_of(lambda j: self.set_of(j).attend(), Kt)
        out["us_attention"] = 1e3 * statistics.median(time_graph(g, reps, self.stream)) / Kt
        del g
        if any(self.tail_launch):
            mk = lambda: torch.cuda.Event(enable_timing=True, external=True)
            ev = [[mk() for _ in range(3)] for _ in range(Kt)]
            for e in [e for tri in ev for e in tri]:
                e.record()
            torch.cuda.synchronize()
            g = graph_of(lambda j: self.set_of(j).attend(events=ev[j]), Kt)
            g.replay()
            torch.cuda.synchronize()
            g.replay()
            torch.cuda.synchronize()
            t_pre = [ev[i][0].elapsed_time(ev[i][1]) for i in range(Kt)]
            t_tail = [ev[i][1].elapsed_time(ev[i][2]) for i in range(Kt) if self.tail_launch[i % len(self.sets)]]
            out["us_prefix_event_pair"] = 1e3 * statistics.mean(t_pre)
            out["us_tail_event_pair"] = 1e3 * statistics.mean(t_tail)
            # the prompt kernel alone: the back-to-back attention time less the tail kernel's share
            out["us_prefix"] = out["us_attention"] * statistics.mean(t_pre) / (statistics.mean(t_pre) +
                                                                                statistics.mean(t_tail))
            out["us_tail_merge"] = out["us_attention"] - out["us_prefix"]
            del g
        else:
            out["us_prefix"] = out["us_attention"]
            out["us_tail_merge"] = None
        for s in self.sets:
            assert bsp.read_device_status(s.plan) == (0, 0)
        return out

    def fractions(self, kt, hbm_gbs):
        """Algorithmic bytes per kernel launch and the achieved fractions of HBM bandwidth."""
        ab = self.ab
        pre = statistics.mean(a["prefix"] for a in ab)
        app = statistics.mean(a["append"] for a in ab)
        tl = [a["tail"] for a, t in zip(ab, self.tail_launch) if t]
        out = {"prefix_bytes": pre, "append_bytes": app,
               "prefix_gbs": pre / (kt["us_prefix"] / 1e6) / 1e9,
               "append_gbs": app / (kt["us_append"] / 1e6) / 1e9,
               "prefix_tflops": statistics.mean(a["prefix_flops"] for a in ab) / (kt["us_prefix"] / 1e6) / 1e12}
        out["prefix_frac"] = out["prefix_gbs"] / hbm_gbs
        out["append_frac"] = out["append_gbs"] / hbm_gbs
        if tl and kt["us_tail_merge"]:
            out["tail_bytes"] = statistics.mean(tl)
            out["tail_gbs"] = out["tail_bytes"] / (kt["us_tail_merge"] / 1e6) / 1e9
            out["tail_frac"] = out["tail_gbs"] / hbm_gbs
        return out

    def step_graphs(self, K):
        chunk = min(K, 2000)
        sizes = [chunk] * (K // chunk) + ([K % chunk] if K % chunk else [])
        graphs, done = [], 0
        for n in sizes:
            graphs.append(graph_of(lambda j, d=done: self.step(d + j), n))
            done += n
        for g in graphs:  # untimed warm replay
            g.replay()
        torch.cuda.synchronize()
        return graphs

    def time_steps(self, graphs, reps, world):
        """ms of each of `reps` timed replays of all K steps (barrier + synchronize on both sides of each),
        max over ranks."""
        out = []
        for _ in range(reps):
            e0, e1 = torch.cuda.Event(enable_timing=True), torch.cuda.Event(enable_timing=True)
            barrier(world)
            torch.cuda.synchronize()
            e0.record(self.stream)
            for g in graphs:
                g.replay()
            e1.record(self.stream)
            torch.cuda.synchronize()
            barrier(world)
            out.append(reduce_max(e0.elapsed_time(e1), world))
        return out

    def release(self):
        self.sets = []
        torch.cuda.synchronize()
        torch.cuda.empty_cache()


def config_summary(wl, args, dev, hbm_gbs, reps=5, **case_kw):
    """Steps/s and per-kernel times of one more decode workload (two rotated input sets)."""
    b = DecodeBench(wl, 2, 3000, dev, **case_kw)
    b.warm(max(3, args.warmup))
    K = min(args.steps, 200)
    kt = b.kernel_times(min(K, 20), reps)
    fr = b.fractions(kt, hbm_gbs)
    graphs = b.step_graphs(K)
    ms = b.time_steps(graphs, reps, 1)
    med = statistics.median(ms) / K
    del graphs
    e2e = run_e2e(b.sets[0], args.e2e_steps, 1)
    R = wl.batch * wl.beam_width
    s0 = b.sets[0].plan
    out = {"steps_per_s": 1e3 / med, "beam_steps_per_s": R * 1e3 / med, "us_per_step": 1e3 * med,
           "us_per_step_spread": [1e3 * min(ms) / K, 1e3 * max(ms) / K], "layout": int(s0.layout),
           "prompt_kernel": LAYOUT_KERNEL[int(s0.layout)][0], "tail_requests": int(s0.tail_requests),
           "us_prefix": kt["us_prefix"], "us_tail_merge": kt["us_tail_merge"], "us_append": kt["us_append"],
           "prefix_frac_of_hbm": fr["prefix_frac"], "append_frac_of_hbm": fr["append_frac"],
           "tail_frac_of_hbm": fr.get("tail_frac"), "prefix_tflops": fr["prefix_tflops"],
           "e2e_steps_per_s": e2e["value"], "us_plan_host": e2e["us_plan_host"],
           "us_plan_full_host": e2e["us_plan_full_host"]}
    b.release()
    return out


def bucketed_summary(args, dev, reps=5):
    """The single-allocation decode (one request, one beam, 32/8 heads, fp16, 10368-row allocation, T = 1):
    a step over the valid prefix against a step that attends every row of the allocation."""
    from beam_search_shared_gb300 import synth
    out = {}
    for P in (10000, 2047):
        wl = synth.WORKLOADS[f"bucketed_prefix_p{P}"]
        us = {}
        for name, kw in (("bound", {}), ("full_allocation", {"prompt_lengths": [10367]})):
            b = DecodeBench(wl, 2, 4000, dev, **kw)
            b.warm(max(3, args.warmup))
            K = 200
            graphs = b.step_graphs(K)
            us[name] = 1e3 * statistics.median(b.time_steps(graphs, reps, 1)) / K
            del graphs
            b.release()
        out[f"p{P}"] = {"us_per_step_bound": us["bound"], "us_per_step_full_allocation": us["full_allocation"],
                        "full_over_bound": us["full_allocation"] / us["bound"]}
    return out


def main():
    args = parse()
    rank, world, local = dist_init(args)
    from beam_search_shared_gb300 import synth
    if args.workload in synth.PREFILL_WORKLOADS:
        return run_prefill(args, rank, world, local)
    wl = synth.WORKLOADS[args.workload]
    R = wl.batch * wl.beam_width

    if args.impl == "reference":
        if rank != 0:
            return
        timer = OracleTimer(synth.make_case(wl, 1000, full_step=True, device="cpu"))
        for _ in range(max(3, args.warmup)):
            timer.step_seconds(1)
        n = timer.rows_for(args.cpu_seconds / max(1, args.steps))
        per_step, spent = [], 0.0
        for _ in range(args.steps):
            s, w = timer.step_seconds(n)
            per_step.append(s)
            spent += w
        v = 1.0 / statistics.mean(per_step)
        line = {"impl": "reference", "metric": METRIC, "value": v, "unit": "steps/s", "n_gpus": args.gpus,
                "steps": args.steps, "warmup": max(3, args.warmup), "ms_per_step": 1e3 / v,
                "higher_is_better": True, "scaling": "weak", "vs_baseline": None, "dtype": "f64",
                "data": "synthetic", "config": {"workload": wl.name, "batch": wl.batch, "beam_width": wl.beam_width},
                "cpu_baseline": {"value": v, "unit": "steps/s", "cores": timer.cores, "kind": "oracle",
                                 "sample": f"{n} of {timer.R} beam rows per step ({spent:.1f} s in total), "
                                           f"scaled linearly; append scatter in full; {cpu_model()}"},
                "e2e": {"value": v, "unit": "steps/s", "h2d_bytes_per_step": 0, "d2h_bytes_per_step": 0}}
        print(json.dumps(line), flush=True)
        return

    from beam_search_shared_gb300 import bsp
    bsp.load(build_if_missing=True)
    dev = torch.device("cuda", local if world > 1 else 0)
    torch.cuda.set_device(dev)
    hbm_gbs, bf16_tflops, peak_kind = measured_peaks()

    # ---- the headline workload: rotated input sets, each its own workspace and plan
    hb = DecodeBench(wl, args.sets, 1000 + 97 * rank, dev)
    hb.warm(max(3, args.warmup))
    K = args.steps
    Kt = min(K, 50)
    kt = hb.kernel_times(Kt, 5)
    fr = hb.fractions(kt, hbm_gbs)

    # ---- timed region: exactly K steps replayed from CUDA graphs without timing nodes, repeated; the
    # value is the median repeat
    graphs = hb.step_graphs(K)
    reps = max(10, args.repeats)
    with ClockSampler(torch.cuda.current_device()) as clk:
        rep_ms = hb.time_steps(graphs, reps, world)
    del graphs
    med_ms = statistics.median(rep_ms)
    ms_per_step = med_ms / K
    value = world * K / (med_ms / 1e3)
    for s in hb.sets:
        assert bsp.read_device_status(s.plan) == (0, 0)

    layout = hb.layout
    kname, ksrc = LAYOUT_KERNEL[layout]
    traffic = profiled_traffic(wl.name, kname, ksrc)
    achieved = fr["prefix_gbs"]

    # ---- e2e: host buffers through the C ABI (plan from host arrays, H2D inputs, D2H outputs)
    e2e = run_e2e(hb.sets[0], args.e2e_steps, world)
    # ---- RoPE and E4M3 appends, timed on their own after the step timing (they rewrite the new tokens' rows)
    rope_append = measure_rope_append(hb.sets, Kt, hbm_gbs)
    fp8_append = measure_fp8_append(hb.sets, Kt, hbm_gbs)
    fp8_attention = measure_fp8_attention(hb.sets[0], Kt, hbm_gbs)
    launches = hb.launches(K)
    step_bytes = fr["prefix_bytes"] + statistics.mean(a["tail"] for a in hb.ab)
    prefix_units = int(hb.sets[0].plan.num_units)
    hb.release()

    line = {
        "metric": METRIC, "value": value, "unit": "steps/s", "n_gpus": world, "steps": K,
        "warmup": max(3, args.warmup), "ms_per_step": ms_per_step, "higher_is_better": True, "scaling": "weak",
        "vs_baseline": None, "dtype": wl.dtype, "data": "synthetic",
        "config": {"workload": wl.name, "batch": wl.batch, "beam_width": wl.beam_width,
                   "q_heads": wl.num_q_heads, "kv_heads": wl.num_kv_heads, "head_dim": wl.head_dim,
                   "page_size": wl.page_size, "prompt": f"U{{{wl.prompt[0]}..{wl.prompt[1]}}}",
                   "tail": f"U{{{wl.tail[0]}..{wl.tail[1]}}}", "parallelism": f"dp{world} (independent batches)",
                   "beam_steps_per_s": value * R,
                   "l2": f"inputs larger than L2: {len(hb.ab)} rotated input sets, each step moving "
                         f"{step_bytes / 1e6:.0f} MB",
                   "repeats": reps, "ms_per_step_spread": [min(rep_ms) / K, max(rep_ms) / K],
                   "prompt_kernel": kname, "layout": layout,
                   "us_append": kt["us_append"], "us_prefix": kt["us_prefix"], "us_attention": kt["us_attention"],
                   "us_prefix_event_pair": kt.get("us_prefix_event_pair"), "us_tail_merge": kt["us_tail_merge"],
                   "gbs_append": fr["append_gbs"], "append_frac_of_hbm": fr["append_frac"],
                   "gbs_tail_merge": fr.get("tail_gbs"), "tail_frac_of_hbm": fr.get("tail_frac"),
                   "prefix_tflops": fr["prefix_tflops"], "prefix_units": prefix_units},
        "roofline": {"bound": "hbm", "achieved": achieved, "peak": hbm_gbs, "unit": "GB/s",
                     "frac": achieved / hbm_gbs, "traffic": traffic,
                     "kernel": kname, "peak_kind": peak_kind,
                     "algorithmic_bytes_per_launch": fr["prefix_bytes"]},
        "e2e": e2e,
        "rope_append": rope_append,
        "fp8_append": fp8_append,
        "fp8_attention": fp8_attention,
        "gpu_launches": launches * reps,
        "timing": f"value: median of {reps} repeats of a CUDA-graph replay of exactly K steps without timing "
                  f"nodes (spread in config.ms_per_step_spread); us_prefix (and the roofline), us_append: one event "
                  f"pair around a graph of {Kt} back-to-back launches (launch gaps included), median of 5 replays; "
                  "a tail-kernel share, when present, from a replay with an event pair around each kernel",
        "clocks": clk.result,
    }
    if rank == 0 and world == 1 and not args.no_configs:
        others = {}
        for name in OTHER_CONFIGS:
            others[name] = config_summary(synth.WORKLOADS[name], args, dev, hbm_gbs)
        others["bucketed_prefix"] = bucketed_summary(args, dev)
        line["configs"] = others
    if rank == 0 and world == 1 and not args.no_cpu_baseline:
        timer = OracleTimer(synth.make_case(wl, 1000, full_step=True, device="cpu"))
        n = timer.rows_for(args.cpu_seconds)
        s, w = timer.step_seconds(n)
        line["cpu_baseline"] = {"value": 1.0 / s, "unit": "steps/s", "cores": timer.cores, "kind": "oracle",
                                "sample": f"{n} of {timer.R} beam rows of one step ({w:.1f} s), scaled "
                                          f"linearly; append scatter in full; {cpu_model()}"}
    if rank == 0:
        print(json.dumps(line), flush=True)
    if world > 1:
        import torch.distributed as dist
        dist.destroy_process_group()


def measure_rope_append(sets, Kt, hbm_gbs):
    """bsp_rope_append_kv over each set's new tokens (rotate-half over the whole head, base 1e6, a
    40960-position table; the new tokens' q rows rotated in place): Kt launches back to back in one
    graph, one event pair around its replay. Algorithmic bytes: K and V rows read and written to the
    pools, q rows read and written, slots and positions, the table rows of the distinct positions."""
    from beam_search_shared_gb300 import bsp, synth
    wl = sets[0].case.workload
    rope = bsp.Rope(40960, wl.head_dim, 1e6)
    items, nbytes = [], []
    for s in sets:
        c = s.case
        n = int(c.out_cache_loc.size)
        pos_h = synth.token_positions(c)
        pos = torch.from_numpy(pos_h).to(s.q.device)
        qn = s.q[torch.from_numpy(c.new_rows).long().to(s.q.device)].reshape(n, -1).contiguous()
        items.append((s, pos, qn))
        e = 2
        nbytes.append(n * (4 * wl.num_kv_heads * wl.head_dim * e + 2 * wl.num_q_heads * wl.head_dim * e + 8) +
                      len(np.unique(pos_h)) * wl.head_dim * 4)

    def launch(j):
        s, pos, qn = items[j % len(items)]
        bsp.rope_append_kv(s.plan, rope, pos, qn, s.k_new, s.v_new, s.out_cache_loc, s.k_pool, s.v_pool)

    for j in range(3):
        launch(j)
    torch.cuda.synchronize()
    g = torch.cuda.CUDAGraph()
    with torch.cuda.graph(g):
        for j in range(Kt):
            launch(j)
    g.replay()
    torch.cuda.synchronize()
    stream = torch.cuda.current_stream()
    e0, e1 = torch.cuda.Event(enable_timing=True), torch.cuda.Event(enable_timing=True)
    e0.record(stream)
    g.replay()
    e1.record(stream)
    torch.cuda.synchronize()
    for s, _, _ in items:
        assert bsp.read_device_status(s.plan) == (0, 0)
    us = 1e3 * e0.elapsed_time(e1) / Kt
    b = statistics.mean(nbytes)
    gbs = b / (us / 1e6) / 1e9
    return {"kernel": "rope_append_kernel", "us": us, "gbs": gbs, "frac_of_hbm": gbs / hbm_gbs,
            "algorithmic_bytes_per_launch": b, "rotary_dim": wl.head_dim, "layout": "rotate-half",
            "timing": f"one event pair around {Kt} back-to-back launches (launch gaps included)"}


def measure_fp8_attention(st, Kt, hbm_gbs):
    """bsp_decode_attn_fp8 over E4M3 pools of the same shape as the set's 16-bit pools (random E4M3 codes,
    k_scale = v_scale = 0.5): Kt launches back to back in one graph, one event pair around each of 5
    replays (median). The pools (one byte per element) are larger than L2. Algorithmic bytes: the 16-bit
    step's with the K/V rows at one byte per element."""
    from beam_search_shared_gb300 import bsp, synth
    from beam_search_shared_gb300.step import algorithmic_bytes
    c = st.case
    wl = c.workload
    g = torch.Generator(device=st.q.device).manual_seed(4242)
    k8 = synth.e4m3_codes(tuple(c.k_pool.shape), g, device=st.q.device)
    v8 = synth.e4m3_codes(tuple(c.v_pool.shape), g, device=st.q.device)
    geo = bsp.geometry(wl.num_q_heads, wl.num_kv_heads, wl.head_dim, wl.page_size, c.num_pages, wl.dtype,
                       kv_dtype=bsp.KV_DTYPE_E4M3)
    ws = bsp.Workspace(geo, wl.batch, wl.beam_width, c.prefix_pages.shape[1], device=st.q.device)
    plan = ws.plan(geo, wl.batch, wl.beam_width, c.prefix_len, c.tail_len, c.prefix_pages, st.max_tail)

    def launch(j):
        bsp.decode_attn_fp8(plan, st.q, k8, v8, st.beam_pages, st.cache_indirection, st.scale, 0.5, 0.5, st.o,
                            st.lse)

    for j in range(3):
        launch(j)
    torch.cuda.synchronize()
    assert bsp.read_device_status(plan) == (0, 0)
    fused = bsp.plan_requests(*bsp.plan_build(geo, wl.batch, wl.beam_width, c.prefix_len, c.tail_len,
                                              c.prefix_pages, st.max_tail, plan.num_sms))[:, 5] != 0
    ab16 = algorithmic_bytes(c, fused)
    # the 16-bit step's prompt-kernel bytes less half of every K/V row it reads
    T = c.tail_len.astype(np.int64)
    kv16 = ab16["prefix_kv"] + int(np.sum(T[fused])) * wl.beam_width * wl.num_kv_heads * wl.head_dim * 4
    b = ab16["prefix"] - kv16 // 2
    g_ = graph_of(launch, Kt)
    us = 1e3 * statistics.median(time_graph(g_, 5, torch.cuda.current_stream())) / Kt
    del g_
    assert bsp.read_device_status(plan) == (0, 0)
    gbs = b / (us / 1e6) / 1e9
    kname = LAYOUT_KERNEL[int(plan.layout)][0]
    out = {"kernel": f"{kname} (E4M3 pools)", "us": us, "gbs": gbs, "frac_of_hbm": gbs / hbm_gbs,
           "algorithmic_bytes_per_launch": b, "tail_requests": int(plan.tail_requests),
           "timing": f"one event pair around {Kt} back-to-back launches (launch gaps included), median of 5 replays"}
    del k8, v8, ws
    torch.cuda.empty_cache()
    return out


def measure_fp8_append(sets, Kt, hbm_gbs):
    """bsp_append_kv_fp8 of each set's new tokens into E4M3 pools of the same geometry (multipliers 1):
    Kt launches back to back in one graph, one event pair. Algorithmic bytes: the 16-bit K and V rows
    read, the 8-bit rows written, the slots."""
    from beam_search_shared_gb300 import bsp
    wl = sets[0].case.workload
    items, nbytes = [], []
    for s in sets:
        c = s.case
        shape = (c.num_pages, wl.num_kv_heads, wl.page_size, wl.head_dim)
        k8 = torch.zeros(shape, dtype=torch.uint8, device=s.q.device)
        v8 = torch.zeros(shape, dtype=torch.uint8, device=s.q.device)
        items.append((s, k8, v8))
        n = int(c.out_cache_loc.size)
        nbytes.append(n * (2 * wl.num_kv_heads * wl.head_dim * (2 + 1) + 4))

    def launch(j):
        s, k8, v8 = items[j % len(items)]
        bsp.append_kv_fp8(s.plan, s.k_new, s.v_new, s.out_cache_loc, k8, v8)

    for j in range(3):
        launch(j)
    torch.cuda.synchronize()
    g = torch.cuda.CUDAGraph()
    with torch.cuda.graph(g):
        for j in range(Kt):
            launch(j)
    g.replay()
    torch.cuda.synchronize()
    stream = torch.cuda.current_stream()
    e0, e1 = torch.cuda.Event(enable_timing=True), torch.cuda.Event(enable_timing=True)
    e0.record(stream)
    g.replay()
    e1.record(stream)
    torch.cuda.synchronize()
    for s, _, _ in items:
        assert bsp.read_device_status(s.plan) == (0, 0)
    us = 1e3 * e0.elapsed_time(e1) / Kt
    b = statistics.mean(nbytes)
    gbs = b / (us / 1e6) / 1e9
    return {"kernel": "append_kv_fp8_kernel", "us": us, "gbs": gbs, "frac_of_hbm": gbs / hbm_gbs,
            "algorithmic_bytes_per_launch": b, "source": wl.dtype, "cache": "e4m3",
            "timing": f"one event pair around {Kt} back-to-back launches (launch gaps included)"}


def host_us(fn, n=200):
    """Median host time (us) of fn() over n calls, the stream drained between calls."""
    ts = []
    for _ in range(n):
        torch.cuda.synchronize()
        t0 = time.perf_counter()
        fn()
        ts.append(time.perf_counter() - t0)
    torch.cuda.synchronize()
    return 1e6 * statistics.median(ts)


def run_e2e(st, steps, world):
    """Steps through the public API from pinned host buffers: per-step plan update (the batch's plan is
    dealt once, before the loop) + H2D inputs + append + attention + D2H outputs. Also the host time of
    a per-step plan update and of a full plan."""
    from beam_search_shared_gb300 import bsp
    c = st.case
    wl = c.workload
    pin = lambda t: t.detach().cpu().contiguous().pin_memory()
    h_q, h_kn, h_vn = pin(c.q), pin(st.k_new), pin(st.v_new)
    h_loc = pin(torch.from_numpy(c.out_cache_loc))
    h_bp = pin(torch.from_numpy(c.beam_pages))
    h_ci = pin(torch.from_numpy(c.cache_indirection))
    h_o = torch.empty(st.o.shape, dtype=st.o.dtype).pin_memory()
    h_lse = torch.empty(st.lse.shape, dtype=torch.float32).pin_memory()
    d_q, d_kn, d_vn = torch.empty_like(st.q), torch.empty_like(st.k_new), torch.empty_like(st.v_new)
    d_loc, d_bp, d_ci = torch.empty_like(st.out_cache_loc), torch.empty_like(st.beam_pages), torch.empty_like(
        st.cache_indirection)
    tails = np.ascontiguousarray(c.tail_len, np.int32)
    full_plan = lambda: st.ws.plan(st.geo, wl.batch, wl.beam_width, c.prefix_len, c.tail_len, c.prefix_pages,
                                   st.max_tail)
    us_plan_full = host_us(full_plan)
    plan = full_plan()
    us_plan_host = host_us(lambda: bsp.plan_update_tails(plan, tails))
    h2d = sum(t.numel() * t.element_size() for t in (h_q, h_kn, h_vn, h_loc, h_bp, h_ci))
    h2d += 64 + 48 * wl.batch  # the update's image header and request records
    d2h = h_o.numel() * h_o.element_size() + h_lse.numel() * 4

    def one():
        bsp.plan_update_tails(plan, tails)
        for d, h in ((d_q, h_q), (d_kn, h_kn), (d_vn, h_vn), (d_loc, h_loc), (d_bp, h_bp), (d_ci, h_ci)):
            d.copy_(h, non_blocking=True)
        bsp.append_kv(plan, d_kn, d_vn, d_loc, st.k_pool, st.v_pool)
        bsp.decode_attn(plan, d_q, st.k_pool, st.v_pool, d_bp, d_ci, st.scale, st.o, st.lse)
        h_o.copy_(st.o, non_blocking=True)
        h_lse.copy_(st.lse, non_blocking=True)

    for _ in range(3):
        one()
    torch.cuda.synchronize()
    assert bsp.read_device_status(plan) == (0, 0)
    barrier(world)
    t0 = time.perf_counter()
    for _ in range(steps):
        one()
    torch.cuda.synchronize()
    dt = reduce_max(time.perf_counter() - t0, world)
    assert bsp.read_device_status(plan) == (0, 0)
    st.make_plan()  # leave the set's own plan current
    torch.cuda.synchronize()
    return {"value": world * steps / dt, "unit": "steps/s", "h2d_bytes_per_step": int(h2d),
            "d2h_bytes_per_step": int(d2h), "steps": steps, "us_plan_host": us_plan_host,
            "us_plan_full_host": us_plan_full,
            "plan": "dealt once for the batch's prompts before the loop; bsp_plan_update_tails every step"}


# ---------------------------------------------------------------- prefill over the cached prefix
PREFILL_METRIC = "prefill tokens/s"


def run_prefill(args, rank, world, local):
    """Prefill over the cached prefix: a step = bsp_append_kv of the prompt tokens' K/V + bsp_prefill_attn.
    `value` is prompt tokens per second over all ranks; the roofline is the prompt kernel's tensor
    throughput (flops of the kept (row, key) pairs only) against the measured dense 16-bit peak."""
    from beam_search_shared_gb300 import bsp, synth
    from beam_search_shared_gb300.step import PrefillStep, prefill_work
    wl = synth.PREFILL_WORKLOADS[args.workload]
    if args.impl == "reference":
        if rank == 0:
            v, cores, sample = prefill_oracle_rate(wl, args.cpu_seconds)
            print(json.dumps({"impl": "reference", "metric": PREFILL_METRIC, "value": v, "unit": "tokens/s",
                              "n_gpus": args.gpus, "steps": args.steps, "warmup": max(3, args.warmup),
                              "higher_is_better": True, "scaling": "weak", "vs_baseline": None, "dtype": "f64",
                              "data": "synthetic", "config": {"workload": wl.name},
                              "cpu_baseline": {"value": v, "unit": "tokens/s", "cores": cores, "kind": "oracle",
                                               "sample": sample},
                              "e2e": {"value": v, "unit": "tokens/s", "h2d_bytes_per_step": 0,
                                      "d2h_bytes_per_step": 0}}), flush=True)
        return
    bsp.load(build_if_missing=True)
    dev = torch.device("cuda", local if world > 1 else 0)
    torch.cuda.set_device(dev)
    sets = []
    for i in range(args.sets):
        st = PrefillStep(synth.make_prefill_case(wl, 2000 + 97 * rank + i, device=dev), device=dev)
        st.make_plan()
        sets.append(st)
    torch.cuda.synchronize()
    work = [prefill_work(s.case) for s in sets]
    tokens = [s.case.rows for s in sets]
    for i in range(max(3, args.warmup)):
        s = sets[i % len(sets)]
        s.append()
        s.attend()
    torch.cuda.synchronize()
    for s in sets:
        assert bsp.read_device_status(s.plan) == (0, 0)
    K = args.steps
    stream = torch.cuda.current_stream()
    # the prompt kernel alone, back to back, one event pair around the graph
    Kt = min(K, 50)
    g_p = torch.cuda.CUDAGraph()
    with torch.cuda.graph(g_p):
        for j in range(Kt):
            sets[j % len(sets)].attend()
    g_p.replay()
    torch.cuda.synchronize()
    e0, e1 = torch.cuda.Event(enable_timing=True), torch.cuda.Event(enable_timing=True)
    e0.record(stream)
    g_p.replay()
    e1.record(stream)
    torch.cuda.synchronize()
    attn_ms = e0.elapsed_time(e1) / Kt
    # timed region: K steps (append + attention) from graphs without timing nodes
    chunk = min(K, 500)
    sizes = [chunk] * (K // chunk) + ([K % chunk] if K % chunk else [])
    graphs, done = [], 0
    for n in sizes:
        g = torch.cuda.CUDAGraph()
        with torch.cuda.graph(g):
            for j in range(n):
                s = sets[(done + j) % len(sets)]
                s.append()
                s.attend()
        graphs.append(g)
        done += n
    for g in graphs:
        g.replay()
    torch.cuda.synchronize()
    ev0, ev1 = torch.cuda.Event(enable_timing=True), torch.cuda.Event(enable_timing=True)
    with ClockSampler(torch.cuda.current_device()) as clk:
        barrier(world)
        torch.cuda.synchronize()
        ev0.record(stream)
        for g in graphs:
            g.replay()
        ev1.record(stream)
        torch.cuda.synchronize()
        barrier(world)
    elapsed_ms = reduce_max(ev0.elapsed_time(ev1), world)
    tok_per_step = statistics.mean(tokens[j % len(sets)] for j in range(K))
    value = world * K * tok_per_step / (elapsed_ms / 1e3)
    for s in sets:
        assert bsp.read_device_status(s.plan) == (0, 0)
    hbm_gbs, bf16_tflops, peak_kind = measured_peaks()
    flops = statistics.mean(w["flops"] for w in work)
    achieved = flops / (attn_ms / 1e3) / 1e12
    e2e = run_prefill_e2e(sets[0], args.e2e_steps, world)
    line = {
        "metric": PREFILL_METRIC, "value": value, "unit": "tokens/s", "n_gpus": world, "steps": K,
        "warmup": max(3, args.warmup), "ms_per_step": elapsed_ms / K, "higher_is_better": True, "scaling": "weak",
        "vs_baseline": None, "dtype": wl.dtype, "data": "synthetic",
        "config": {"workload": wl.name, "batch": wl.batch, "q_heads": wl.num_q_heads, "kv_heads": wl.num_kv_heads,
                   "head_dim": wl.head_dim, "page_size": wl.page_size, "cached": f"U{{{wl.cached[0]}..{wl.cached[1]}}}",
                   "prompt": f"U{{{wl.prompt[0]}..{wl.prompt[1]}}}", "causal": wl.causal,
                   "alloc_rows": wl.alloc_rows, "parallelism": f"dp{world} (independent batches)",
                   "l2": f"{len(sets)} rotated input sets, pools of "
                         f"{sum(s.k_pool.numel() * 4 for s in sets) / 1e6:.0f} MB in all",
                   "us_prefill_attn": 1e3 * attn_ms, "prefill_attn_gbs": statistics.mean(w["bytes"] for w in work)
                   / (attn_ms / 1e3) / 1e9},
        "roofline": {"bound": "tensor", "achieved": achieved, "peak": bf16_tflops, "unit": "TFLOP/s",
                     "frac": achieved / bf16_tflops, "traffic": None,
                     "kernel": LAYOUT_KERNEL[int(sets[0].plan.layout)][0],
                     "peak_kind": peak_kind + " (16-bit dense; fp16 runs at the bf16 rate)",
                     "algorithmic_flops_per_launch": flops},
        "e2e": e2e,
        "gpu_launches": K * 2,
        "timing": f"value: CUDA-graph replay of exactly K steps (append + attention) without timing nodes; "
                  f"us_prefill_attn: one event pair around {Kt} back-to-back attention launches",
        "clocks": clk.result,
    }
    if rank == 0 and world == 1 and not args.no_cpu_baseline:
        v, cores, sample = prefill_oracle_rate(wl, args.cpu_seconds)
        line["cpu_baseline"] = {"value": v, "unit": "tokens/s", "cores": cores, "kind": "oracle", "sample": sample}
    if rank == 0:
        print(json.dumps(line), flush=True)
    if world > 1:
        import torch.distributed as dist
        dist.destroy_process_group()


def prefill_oracle_rate(wl, seconds):
    """The fp64 oracle's prefill rate on the host cores: one request of the workload's shape with fewer
    prompt tokens (sized from a short probe to take about `seconds`), scaled by the kept (row, key) pairs
    to the workload's own mix."""
    import oracle
    from beam_search_shared_gb300 import synth
    from beam_search_shared_gb300.step import prefill_work
    oracle.build()
    full = synth.make_prefill_case(wl, 2000)
    C0 = int(full.cached_len[0])

    def timed(S):
        sub = wl.with_(batch=1, alloc_rows=0)
        case = synth.make_prefill_case(sub, 2001, cached_lengths=[C0], prompt_lengths=[S])
        t0 = time.perf_counter()
        oracle.prefill_attn(dtype=sub.dtype, B=1, Hq=sub.num_q_heads, Hkv=sub.num_kv_heads, D=sub.head_dim,
                            ps=sub.page_size, num_pages=case.num_pages, cached_len=case.cached_len,
                            prompt_len=case.prompt_len, pages=case.pages, causal=sub.causal,
                            q_bits=synth.bits(case.q), k_pool_bits=synth.bits(case.k_pool),
                            v_pool_bits=synth.bits(case.v_pool), scale=1 / math.sqrt(sub.head_dim))
        return time.perf_counter() - t0, case

    S_max = int(max(1, full.prompt_len.max()))
    S = min(S_max, 16)
    t, case = timed(S)
    per_pair = t / max(1, prefill_work(case)["pairs"])
    while S < S_max:
        # the largest prompt whose pairs fit the budget at the probed rate
        nxt = S
        while nxt < S_max:
            c_try = nxt * 2 if nxt * 2 <= S_max else S_max
            pairs = C0 * c_try + c_try * (c_try + 1) // 2 if wl.causal else c_try * (C0 + c_try)
            if pairs * per_pair > seconds:
                break
            nxt = c_try
        if nxt == S:
            break
        S = nxt
        t, case = timed(S)
        per_pair = t / max(1, prefill_work(case)["pairs"])
    pf, ps_ = prefill_work(full), prefill_work(case)
    full_seconds = t * pf["pairs"] / max(1, ps_["pairs"])
    cores = len(os.sched_getaffinity(0))
    cores = min(cores, int(os.environ.get("OMP_NUM_THREADS", cores)))   # the oracle's OpenMP threads
    sample = (f"1 request of {S} prompt tokens after {C0} cached rows ({t:.1f} s), scaled by kept (row, key) "
              f"pairs to the {full.rows} prompt tokens of the workload; attention only; {cpu_model()}")
    return full.rows / full_seconds, cores, sample


def run_prefill_e2e(st, steps, world):
    """Prefill steps from pinned host buffers through the public API: plan from host arrays, H2D of q,
    the prompt K/V and its slots, append + attention, D2H of O and LSE; timed on the host."""
    from beam_search_shared_gb300 import bsp
    c = st.case
    h_q = st.q.cpu().pin_memory()
    h_kn, h_vn = st.k_new.cpu().pin_memory(), st.v_new.cpu().pin_memory()
    h_loc = torch.from_numpy(c.out_cache_loc).pin_memory()
    h_o = torch.empty(st.o.shape, dtype=st.o.dtype).pin_memory()
    h_lse = torch.empty(st.lse.shape, dtype=torch.float32).pin_memory()
    d_q, d_kn, d_vn = torch.empty_like(st.q), torch.empty_like(st.k_new), torch.empty_like(st.v_new)
    d_loc = torch.empty_like(st.out_cache_loc)
    h2d = sum(t.numel() * t.element_size() for t in (h_q, h_kn, h_vn, h_loc)) + int(st.plan.image_bytes)
    d2h = h_o.numel() * h_o.element_size() + h_lse.numel() * 4

    def one():
        plan = bsp.plan_prefill(st.geo, c.workload.batch, c.cached_len, c.prompt_len, c.pages, c.workload.causal,
                                st.ws)
        d_q.copy_(h_q, non_blocking=True)
        d_kn.copy_(h_kn, non_blocking=True)
        d_vn.copy_(h_vn, non_blocking=True)
        d_loc.copy_(h_loc, non_blocking=True)
        bsp.append_kv(plan, d_kn, d_vn, d_loc, st.k_pool, st.v_pool)
        bsp.prefill_attn(plan, d_q, st.k_pool, st.v_pool, st.scale, st.o, st.lse)
        h_o.copy_(st.o, non_blocking=True)
        h_lse.copy_(st.lse, non_blocking=True)

    for _ in range(3):
        one()
    torch.cuda.synchronize()
    barrier(world)
    t0 = time.perf_counter()
    for _ in range(steps):
        one()
    torch.cuda.synchronize()
    dt = reduce_max(time.perf_counter() - t0, world)
    st.make_plan()  # leave the set's own plan current
    torch.cuda.synchronize()
    return {"value": world * steps * c.rows / dt, "unit": "tokens/s", "h2d_bytes_per_step": int(h2d),
            "d2h_bytes_per_step": int(d2h), "steps": steps}


if __name__ == "__main__":
    main()
