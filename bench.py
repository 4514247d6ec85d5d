#!/usr/bin/env python3
"""Whole-job throughput of the budgeted-KV decode path on GB300.

One bench step is one pass of the whole hot path over one batch of synthetic
input shaped like an OPT-6.7B attention layer (8 x 32 heads, head_dim 128,
prompt 2048, 256 decode steps, budget 410 = 205 heavy + 205 recent, bf16):

  for each of L layer caches: H2O prompt phase (scores, top-k, gather) and
  HashEvict prompt phase (codes, replay, gather) on the same prompt;
  then 256 H2O decode steps and 256 HashEvict decode steps, token-major over
  the L layers, as a model decodes.

L layers (default 8, ~890 MB of caches plus 3.2 GB of prompts) keep every
cache out of L2 between its uses.  The device-timed value replays the step
from CUDA graphs with inputs already in HBM; the e2e value drives the same
job through the public API with pinned host inputs copied in and outputs
copied out inside the timed region.  The CPU oracle is timed on a bounded
sample of the same job.

    python bench.py [--gpus N] [--steps K] [--warmup W] [--impl reference]

With --gqa the job is H2O alone on a grouped-query layer (8 x 8 key/value
heads, each cache shared by 4 query heads; the same prompt, budget and decode
steps): one decode step there advances all 64 cache units (256 query heads)
of one layer cache by one token.  With --sh it is the persistence-of-importance
rule alone on the OPT-6.7B-shaped layer.
"""
import argparse
import hashlib
import json
import os
import statistics
import subprocess
import sys
import time

ROOT = os.path.dirname(os.path.abspath(__file__))
if ROOT not in sys.path:
    sys.path.insert(0, ROOT)

METRIC = "H2O decode steps/s (batch×heads) at 1 GB300; achieved HBM GB/s vs peak"
UNIT = "steps/s"
WORKLOAD = "opt-6.7b"
TRAFFIC_FILE = os.path.join(ROOT, "profiles", "ncu_traffic.json")


def parse():
    p = argparse.ArgumentParser()
    p.add_argument("--gpus", type=int, default=1)
    p.add_argument("--steps", type=int, default=10)
    p.add_argument("--warmup", type=int, default=3)
    p.add_argument("--impl", default="ours", choices=["ours", "reference"])
    p.add_argument("--layers", type=int, default=8)
    p.add_argument("--decode-steps", type=int, default=None)
    p.add_argument("--split", type=int, default=0, help="CTAs per unit in decode (0 = automatic)")
    p.add_argument("--oracle-units", type=int, default=64)
    p.add_argument("--no-e2e", action="store_true")
    p.add_argument("--no-cpu", action="store_true")
    p.add_argument("--kv8", action="store_true",
                   help="int8 cache slots (one fp32 scale per row) for both variants")
    p.add_argument("--gqa", action="store_true",
                   help="H2O on the grouped-query layer (8 x 8 key/value heads x 4 query heads)")
    p.add_argument("--sh", action="store_true",
                   help="the persistence-of-importance rule alone on the OPT-6.7B-shaped layer")
    p.add_argument("--no-overlap", action="store_true",
                   help="skip the second timed region with the two eviction jobs on two streams")
    return p.parse_args()


# ------------------------------------------------------------------ helpers

def load_peaks():
    path = os.path.join(ROOT, "MEASURED_PEAKS.json")
    try:
        with open(path) as f:
            d = json.load(f)
        return float(d["hbm_gbs"]), float(d["bf16_tflops"]), float(d.get("bf16_tflops_sustained", d["bf16_tflops"])), "measured"
    except Exception:
        return 6800.0, 1900.0, 1700.0, "fallback"


def file_digest(*names):
    h = hashlib.sha256()
    for n in names:
        with open(os.path.join(ROOT, "kv_cache_eviction_h2o_gb300", "csrc", n), "rb") as f:
            h.update(f.read())
    return h.hexdigest()[:16]


def ncu_traffic(kernel):
    """Per-launch DRAM bytes from the committed ncu capture, if it was taken
    on the current kernel source; None otherwise."""
    try:
        with open(TRAFFIC_FILE) as f:
            d = json.load(f)
        e = d[kernel]
        if e["source_digest"] != file_digest(*e["sources"]):
            return None
        return float(e["bytes_per_launch"])
    except Exception:
        return None


class Clocks:
    """nvidia-smi sampler for the timed region."""
    Q = ("index,clocks.sm,clocks.max.sm,power.draw,clocks_event_reasons.active,"
         "clocks_event_reasons.hw_slowdown,clocks_event_reasons.hw_thermal_slowdown,"
         "clocks_event_reasons.sw_thermal_slowdown,clocks_event_reasons.sw_power_cap")

    def __init__(self, gpu):
        self.gpu = gpu
        self.proc = None

    def start(self):
        try:
            self.proc = subprocess.Popen(["nvidia-smi", "--query-gpu=" + self.Q, "--format=csv,noheader,nounits",
                                          "-lms", "200", "-i", str(self.gpu)],
                                         stdout=subprocess.PIPE, stderr=subprocess.DEVNULL, text=True)
        except Exception:
            self.proc = None

    def stop(self):
        if self.proc is None:
            return None
        self.proc.terminate()
        try:
            out, _ = self.proc.communicate(timeout=5)
        except Exception:
            self.proc.kill()
            return None
        rows = []
        for line in out.strip().splitlines():
            f = [x.strip() for x in line.split(",")]
            if len(f) < 9:
                continue
            try:
                rows.append((float(f[1]), float(f[2]), float(f[3]), f[5:9]))
            except ValueError:
                continue
        if not rows:
            return None
        names = ["hw_slowdown", "hw_thermal_slowdown", "sw_thermal_slowdown", "sw_power_cap"]
        reasons = sorted({names[i] for r in rows for i, v in enumerate(r[3]) if v.lower() == "active"})
        loaded = [r for r in rows if r[2] > 0.25 * max(x[2] for x in rows)] or rows
        return {"sm_mhz": statistics.median(r[0] for r in loaded), "sm_max_mhz": max(r[1] for r in rows),
                "reasons": reasons, "samples": len(rows), "power_w_max": max(r[2] for r in rows)}


def max_over_ranks(x, world, device="cpu"):
    """Largest value of x over all ranks (the timing rule: the slowest rank
    sets the job time); x itself when world == 1."""
    if world <= 1:
        return float(x)
    import torch
    import torch.distributed as dist
    t = torch.tensor([float(x)], dtype=torch.float64, device=device)
    dist.all_reduce(t, op=dist.ReduceOp.MAX)
    return float(t.item())


def dist_setup(args):
    world = int(os.environ.get("WORLD_SIZE", "1"))
    rank = int(os.environ.get("RANK", "0"))
    local = int(os.environ.get("LOCAL_RANK", "0"))
    return world, rank, local


# ------------------------------------------------------------ algorithmic

def decode_bytes(U, B, d, eb, lsh, kv8=False):
    """Algorithmic HBM bytes of one full-cache decode launch over U units:
    per live slot K and V rows (int8 codes plus an 8-byte scale pair with
    kv8), plus score read+write (8-byte fp32 pair) and position read (H2O)
    or code and position read (HashEvict); per unit q, k, v in, fp32 out,
    one K/V row written (and its scale pair), victim score/code and
    position written, unit state read and written; plus the projection
    matrix once."""
    row = d * eb
    crow = d if kv8 else row
    sc = 8 if kv8 else 0
    if lsh:
        per_slot = 2 * crow + sc + 4 + 4
        fixed = 3 * row + 4 * d + 2 * crow + sc + 4 + 4 + 16
        return U * (B * per_slot + fixed) + d * 32 * 4
    per_slot = 2 * crow + sc + 8 + 8 + 4
    fixed = 3 * row + 4 * d + 2 * crow + sc + 8 + 4 + 16
    return U * (B * per_slot + fixed)


def decode_bytes_gqa(U, G, B, d, eb, kv8=False):
    """Algorithmic HBM bytes of one full-cache grouped-query H2O decode launch
    over U cache units of G query heads: per live slot K and V rows (int8
    codes plus an 8-byte scale pair with kv8), score read+write and position
    read, each once per unit (the heads share them); per query head q in and
    fp32 out; per unit k, v in, one K/V row written (and its scale pair),
    victim score and position written, unit state read and written."""
    row = d * eb
    crow = d if kv8 else row
    sc = 8 if kv8 else 0
    per_slot = 2 * crow + sc + 8 + 8 + 4
    fixed = G * (row + 4 * d) + 2 * row + 2 * crow + sc + 8 + 4 + 16
    return U * (B * per_slot + fixed)


def decode_bytes_sh(U, B, d, eb):
    """Algorithmic HBM bytes of one full-cache persistence-of-importance
    decode launch over U units: per live slot K and V rows, the 32-step
    history read and written and the position read; per unit q, k, v in,
    fp32 out, one K/V row, its history and position written, unit state
    read and written."""
    row = d * eb
    per_slot = 2 * row + 4 + 4 + 4
    fixed = 3 * row + 4 * d + 2 * row + 4 + 4 + 16
    return U * (B * per_slot + fixed)


def prefill_flops(U, T, d):
    """Both score passes of the H2O prompt phase: 2 x (2 d flops per causal
    (i, j) pair, T (T + 1) / 2 pairs per unit)."""
    return 2 * 2 * U * d * T * (T + 1) // 2


# ------------------------------------------------------------------ oracle

def oracle_job(w, wl_lsh, units, S, kv8=False):
    """The CPU oracle on a sample of units: H2O prompt + S steps and
    HashEvict prompt + S steps (int8 cache slots with kv8).  Returns
    (seconds, threads)."""
    import numpy as np

    import oracle
    from kv_cache_eviction_h2o_gb300 import workloads as wl
    g = wl.generate(w, units=units, steps=S)
    W = wl.lsh_matrix(wl_lsh)
    T = w.prompt
    t0 = time.perf_counter()
    st, _, _, _ = oracle.h2o_prefill(g["Q"], g["K"], g["V"], w.budget, w.heavy, w.recent, w.scale)
    if kv8:
        oracle.kv8(st)
    for t in range(S):
        oracle.h2o_decode_step(st, g["q"][t], g["k"][t], g["v"][t], T + t, w.recent, w.scale)
    ls = oracle.lsh_prefill(g["Q"], g["K"], g["V"], W, wl_lsh.budget, wl_lsh.recent)
    if kv8:
        oracle.kv8(ls)
    for t in range(S):
        oracle.lsh_decode_step(ls, g["q"][t], g["k"][t], g["v"][t], W, T + t, wl_lsh.recent, w.scale)
    return time.perf_counter() - t0, oracle.get_threads()


def oracle_job_gqa(w, units, S, kv8=False):
    """The CPU oracle on a sample of cache units of a grouped-query workload:
    H2O prompt + S steps.  Returns (seconds, threads)."""
    import oracle
    from kv_cache_eviction_h2o_gb300 import workloads as wl
    g = wl.generate(w, units=units, steps=S)
    T = w.prompt
    t0 = time.perf_counter()
    st, _, _, _, _ = oracle.h2o_prefill_gqa(g["Q"], g["K"], g["V"], w.budget, w.heavy, w.recent, w.scale)
    if kv8:
        oracle.kv8(st)
    for t in range(S):
        oracle.h2o_decode_step_gqa(st, g["q"][t], g["k"][t], g["v"][t], T + t, w.recent, w.scale)
    return time.perf_counter() - t0, oracle.get_threads()


def oracle_job_sh(w, units, S):
    """The CPU oracle on a sample of units: persistence-of-importance prompt
    + S steps.  Returns (seconds, threads)."""
    import oracle
    from kv_cache_eviction_h2o_gb300 import workloads as wl
    g = wl.generate(w, units=units, steps=S)
    T = w.prompt
    t0 = time.perf_counter()
    st, _, _, _ = oracle.sh_prefill(g["Q"], g["K"], g["V"], w.budget, w.heavy, w.recent, w.scale)
    for t in range(S):
        oracle.sh_decode_step(st, g["q"][t], g["k"][t], g["v"][t], T + t, w.recent, w.scale)
    return time.perf_counter() - t0, oracle.get_threads()


def oracle_rate(w, seconds, n_units, S):
    """Oracle time on n_units scaled to the metric: decode steps (all units of
    one layer cache advancing one token, both variants) per second."""
    per_layer_job = seconds * w.units / n_units
    return 2 * S / per_layer_job


# -------------------------------------------------------------- reference

def run_reference(args):
    world, rank, _ = dist_setup(args)
    if rank != 0:
        return
    if args.gqa or args.sh:
        return run_reference_single(args, world, "gqa" if args.gqa else "sh")
    from kv_cache_eviction_h2o_gb300 import workloads as wl
    w = wl.WORKLOADS[WORKLOAD]
    wl_lsh = wl.WORKLOADS["hashevict-" + WORKLOAD]
    S = args.decode_steps or w.steps
    n = max(1, args.oracle_units // 4)
    units = list(range(n))
    for _ in range(args.warmup):
        oracle_job(w, wl_lsh, units, S, args.kv8)
    times = []
    threads = 1
    for _ in range(args.steps):
        t, threads = oracle_job(w, wl_lsh, units, S, args.kv8)
        times.append(t)
    total = sum(times)
    value = oracle_rate(w, total / len(times), n, S)
    sample = "%d of %d units of one %s layer per step (prompt %d, %d decode steps, H2O + HashEvict)" % (
        n, w.units, WORKLOAD, w.prompt, S)
    line = {
        "impl": "reference", "metric": METRIC, "value": value, "unit": UNIT, "n_gpus": world,
        "steps": args.steps, "warmup": args.warmup,
        "ms_per_step": 1000.0 * total / len(times), "higher_is_better": True, "scaling": "weak",
        "vs_baseline": None, "dtype": "f64", "data": "synthetic",
        "config": {"workload": "%s-shaped layer: H2O + HashEvict, prompt %d -> %d decode steps, budget %d"
                               % (WORKLOAD, w.prompt, S, w.budget)},
        "cpu_baseline": {"value": value, "unit": UNIT, "cores": threads, "kind": "oracle", "sample": sample},
        "e2e": {"value": value, "unit": UNIT, "h2d_bytes_per_step": 0, "d2h_bytes_per_step": 0},
    }
    print(json.dumps(line))


def run_reference_single(args, world, variant):
    from kv_cache_eviction_h2o_gb300 import workloads as wl
    w = wl.WORKLOADS[GQA_WORKLOAD if variant == "gqa" else WORKLOAD]
    S = args.decode_steps or w.steps
    n = max(1, args.oracle_units // 16)
    units = list(range(n))
    job = (lambda: oracle_job_gqa(w, units, S, args.kv8)) if variant == "gqa" else (lambda: oracle_job_sh(w, units, S))
    for _ in range(args.warmup):
        job()
    times = []
    threads = 1
    for _ in range(args.steps):
        t, threads = job()
        times.append(t)
    total = sum(times)
    value = S / (total / len(times) * w.units / n)
    line = {
        "impl": "reference", "metric": METRIC, "value": value, "unit": UNIT, "n_gpus": world,
        "steps": args.steps, "warmup": args.warmup,
        "ms_per_step": 1000.0 * total / len(times), "higher_is_better": True, "scaling": "weak",
        "vs_baseline": None, "dtype": "f64", "data": "synthetic",
        "config": {"workload": gqa_config_name(w, S, 1, args.kv8) if variant == "gqa" else sh_config_name(w, S, 1)},
        "cpu_baseline": {"value": value, "unit": UNIT, "cores": threads, "kind": "oracle",
                         "sample": "%d of %d cache units of one %s layer per step (prompt %d, %d decode steps, %s)"
                                   % (n, w.units, w.name, w.prompt, S,
                                      "H2O" if variant == "gqa" else "persistence of importance")},
        "e2e": {"value": value, "unit": UNIT, "h2d_bytes_per_step": 0, "d2h_bytes_per_step": 0},
    }
    print(json.dumps(line))


GQA_WORKLOAD = "gqa-8x8x4"


def gqa_config_name(w, S, NL, kv8):
    return ("%s grouped-query layer x%d (%d x %d key/value heads x %d query heads): H2O, prompt %d -> %d decode "
            "steps, budget %d (%d heavy + %d recent)%s" % (GQA_WORKLOAD, NL, w.batch, w.heads, w.groups, w.prompt,
                                                          S, w.budget, w.heavy, w.recent,
                                                          ", int8 cache slots" if kv8 else ""))


def sh_config_name(w, S, NL):
    return ("%s-shaped layer x%d: persistence-of-importance rule (32-step pivotal histories), prompt %d -> %d "
            "decode steps, budget %d (%d heavy + %d recent)" % (w.name, NL, w.prompt, S, w.budget, w.heavy, w.recent))


# -------------------------------------------------------------------- ours

def run_ours(args):
    import torch
    import torch.distributed as dist

    from kv_cache_eviction_h2o_gb300 import binding as L
    from kv_cache_eviction_h2o_gb300 import build as lib_build
    from kv_cache_eviction_h2o_gb300 import workloads as wl

    world, rank, local = dist_setup(args)
    if world > 1:
        torch.cuda.set_device(local)
        dist.init_process_group("nccl", device_id=torch.device("cuda", local))
    else:
        torch.cuda.set_device(local)
    lib_build.build()
    L.lib()
    w = wl.WORKLOADS[WORKLOAD]
    wl_lsh = wl.WORKLOADS["hashevict-" + WORKLOAD]
    S = args.decode_steps or w.steps
    NL = args.layers
    U, T, d, B = w.units, w.prompt, w.head_dim, w.budget
    dt = L.H2O_BF16 | (L.H2O_KV8 if args.kv8 else 0)
    stream = torch.cuda.Stream()

    # ---- inputs resident in HBM, one set per layer cache
    layers = []
    with torch.cuda.stream(stream):
        for li in range(NL):
            g = wl.generate_device(w, seed_offset=li + 1000 * rank, steps=S)
            layers.append(g)
        W = torch.from_numpy(wl.lsh_matrix(wl_lsh)).cuda()
    torch.cuda.synchronize()
    h2o = [L.h2o_init(B, w.heavy, w.recent, w.batch, w.heads, d, dt, w.scale, stream) for _ in range(NL)]
    lsh = [L.lsh_init(B, wl_lsh.recent, w.batch, w.heads, d, dt, w.scale, W, stream) for _ in range(NL)]
    if args.split:
        for h in h2o + lsh:
            L.h2o_set_decode_split(h, args.split)
    out_h = [torch.empty((S, U, d), dtype=torch.float32, device="cuda") for _ in range(NL)]
    out_l = [torch.empty((S, U, d), dtype=torch.float32, device="cuda") for _ in range(NL)]
    vic_h = [torch.empty((S, U), dtype=torch.int32, device="cuda") for _ in range(NL)]
    vic_l = [torch.empty((S, U), dtype=torch.int32, device="cuda") for _ in range(NL)]

    def pre_h2o():
        for li in range(NL):
            g = layers[li]
            L.h2o_prefill(h2o[li], g["Q"], g["K"], g["V"], T)

    def pre_lsh():
        for li in range(NL):
            g = layers[li]
            L.lsh_prefill(lsh[li], g["Q"], g["K"], g["V"], T)

    def dec_h2o():
        for t in range(S):
            for li in range(NL):
                g = layers[li]
                L.h2o_decode_step(h2o[li], g["q"][t], g["k"][t], g["v"][t], out_h[li][t], vic_h[li][t])

    def dec_lsh():
        for t in range(S):
            for li in range(NL):
                g = layers[li]
                L.lsh_decode_step(lsh[li], g["q"][t], g["k"][t], g["v"][t], out_l[li][t], vic_l[li][t])

    phases = [("h2o_prefill", pre_h2o), ("lsh_prefill", pre_lsh), ("h2o_decode", dec_h2o), ("lsh_decode", dec_lsh)]
    # eager pass: allocates prompt scratch, sets kernel attributes, checks errors
    with torch.cuda.stream(stream):
        for _, f in phases:
            f()
    for h in h2o + lsh:
        L.h2o_sync(h)

    graphs = []
    with torch.cuda.stream(stream):
        for name, f in phases:
            gr = torch.cuda.CUDAGraph()
            gr.capture_begin()
            f()
            gr.capture_end()
            graphs.append((name, gr))
    torch.cuda.synchronize()

    def one_step(evs=None):
        with torch.cuda.stream(stream):
            for i, (name, gr) in enumerate(graphs):
                gr.replay()
                if evs is not None:
                    evs[i].record(stream)

    for _ in range(args.warmup):
        one_step()
    torch.cuda.synchronize()
    for h in h2o + lsh:
        L.h2o_sync(h)

    # ---- timed region
    clocks = Clocks(local)
    if world > 1:
        dist.barrier()
    torch.cuda.synchronize()
    clocks.start()
    time.sleep(0.3)
    start = torch.cuda.Event(enable_timing=True)
    end = torch.cuda.Event(enable_timing=True)
    step_events = [[torch.cuda.Event(enable_timing=True) for _ in graphs] for _ in range(args.steps)]
    start.record(stream)
    for i in range(args.steps):
        one_step(step_events[i])
    end.record(stream)
    torch.cuda.synchronize()
    if world > 1:
        dist.barrier()
    clk = clocks.stop()
    elapsed_ms = start.elapsed_time(end)
    phase_ms = {name: 0.0 for name, _ in graphs}
    for i in range(args.steps):
        prev = start if i == 0 else step_events[i - 1][-1]
        for j, (name, _) in enumerate(graphs):
            phase_ms[name] += prev.elapsed_time(step_events[i][j])
            prev = step_events[i][j]
    for h in h2o + lsh:
        L.h2o_sync(h)
    elapsed_ms = max_over_ranks(elapsed_ms, world, device="cuda")
    overlap = None if args.no_overlap else time_overlapped(args, torch, dist, graphs, stream, world,
                                                           2 * S * NL, h2o + lsh, L)

    K = args.steps
    ms_per_step = elapsed_ms / K
    decode_steps_per_bench_step = 2 * S * NL
    value = world * decode_steps_per_bench_step / (ms_per_step / 1000.0)
    hbm, tf_burst, tf_sus, peak_src = load_peaks()

    # ---- rooflines from the phase times (per-launch averages)
    eb = 2
    rl = []
    n_dec = S * NL * K
    for name, lsh_flag, src in (("h2o_decode", False, ["decode.cu", "common.cuh"]),
                                ("lsh_decode", True, ["decode.cu", "common.cuh"])):
        t_launch = phase_ms[name] / n_dec / 1000.0
        by = decode_bytes(U, B, d, eb, lsh_flag, args.kv8)
        ach = by / t_launch / 1e9
        rl.append({"kernel": name, "bound": "hbm", "achieved": ach, "peak": hbm, "unit": "GB/s",
                   "frac": ach / hbm, "traffic": ncu_traffic(name + ("_kv8" if args.kv8 else "")),
                   "algorithmic_bytes": by,
                   "launch_us": t_launch * 1e6, "peak_source": peak_src, "share": phase_ms[name] / elapsed_ms})
    t_pre = phase_ms["h2o_prefill"] / (NL * K) / 1000.0
    fl = prefill_flops(U, T, d)
    ach = fl / t_pre / 1e12
    rl.append({"kernel": "h2o_prefill", "bound": "tensor", "achieved": ach, "peak": tf_sus, "unit": "TFLOP/s",
               "frac": ach / tf_sus, "traffic": None, "algorithmic_flops": fl, "launch_us": t_pre * 1e6,
               "peak_source": peak_src, "share": phase_ms["h2o_prefill"] / elapsed_ms})
    t_lp = phase_ms["lsh_prefill"] / (NL * K) / 1000.0
    rl.append({"kernel": "lsh_prefill", "bound": "latency", "launch_us": t_lp * 1e6,
               "share": phase_ms["lsh_prefill"] / elapsed_ms})
    dominant = max(rl, key=lambda r: r["share"])
    main_rl = {k: dominant[k] for k in ("bound", "achieved", "peak", "unit", "frac", "traffic") if k in dominant}
    main_rl["kernel"] = dominant["kernel"]
    main_rl["peak_source"] = peak_src
    if "achieved" not in main_rl:
        main_rl = {k: rl[0][k] for k in ("bound", "achieved", "peak", "unit", "frac", "traffic")}
        main_rl["kernel"] = rl[0]["kernel"]

    # ---- end to end through the public API with pinned host buffers
    e2e = None
    if not args.no_e2e:
        e2e = run_e2e(args, L, torch, layers, h2o, lsh, out_h, out_l, vic_h, vic_l, W, S, NL, T, stream, world)

    # ---- CPU oracle on a bounded sample (rank 0, one GPU only)
    cpu = None
    if rank == 0 and world == 1 and not args.no_cpu:
        n = args.oracle_units
        secs, threads = oracle_job(w, wl_lsh, list(range(n)), S, args.kv8)
        cpu = {"value": oracle_rate(w, secs, n, S), "unit": UNIT, "cores": threads, "kind": "oracle",
               "sample": "%d of %d units of one layer (prompt %d, %d decode steps, H2O + HashEvict), %.1f s"
                         % (n, U, T, S, secs)}

    launches_per_step = NL * (4 + 3) + 2 * S * NL
    line = {
        "metric": METRIC, "value": value, "unit": UNIT, "n_gpus": world, "steps": K, "warmup": args.warmup,
        "ms_per_step": ms_per_step, "higher_is_better": True, "scaling": "weak", "vs_baseline": None,
        "dtype": "bf16", "data": "synthetic",
        "config": {"workload": "%s-shaped layer x%d: H2O + HashEvict, prompt %d -> %d decode steps, budget %d "
                               "(%d heavy + %d recent)%s" % (WORKLOAD, NL, T, S, B, w.heavy, w.recent,
                                                             ", int8 cache slots" if args.kv8 else ""),
                   "cache": "int8 codes + fp32 scale per row" if args.kv8 else "bf16",
                   "batch": w.batch, "heads": w.heads, "head_dim": d, "prompt": T, "decode_steps": S,
                   "budget": B, "layers": NL, "global_batch": w.batch * world,
                   "parallelism": "replicas" if world > 1 else "single",
                   "l2": "inputs larger than L2: %d layer caches (%.0f MB) + prompts (%.0f MB); a cache is reused "
                         "only after %d others" % (NL, 2 * NL * decode_bytes(U, B, d, eb, False, args.kv8) / 1e6,
                                                   NL * 3 * U * T * d * eb / 1e6, NL - 1),
                   "step": "one decode step = all %d (batch x head) units of one layer cache advance one token; "
                           "both eviction variants counted; prompt phases inside the timed step" % U},
        "roofline": main_rl,
        "rooflines": rl,
        "phases_ms_per_step": {k: v / K for k, v in phase_ms.items()},
        "head_steps_per_s": value * U,
        "cpu_baseline": cpu,
        "clocks": clk,
        "e2e": e2e,
        "gpu_launches": launches_per_step * K,
        "overlap": overlap,
    }
    for h in h2o + lsh:
        L.h2o_destroy(h)
    if rank == 0:
        print(json.dumps(line))
    if world > 1:
        dist.destroy_process_group()


def time_overlapped(args, torch, dist, graphs, stream, world, units_per_step, handles, L):
    """The same K steps with the two eviction jobs, independent of each
    other, on two streams: the H2O prompt and decode graphs on `stream`, the
    HashEvict ones on a second stream, joined at the end of every step, so a
    job's prompt phase and per-launch fixed costs run under the other job's
    HBM-bound decode.  Timed like the main region (barrier, device events,
    max over ranks); per-kernel rooflines come from the serial region."""
    gd = dict(graphs)
    side = torch.cuda.Stream()
    fork = [torch.cuda.Event() for _ in range(2)]
    join = [torch.cuda.Event() for _ in range(2)]

    def step(i):
        fork[i % 2].record(stream)
        side.wait_event(fork[i % 2])
        with torch.cuda.stream(side):
            gd["lsh_prefill"].replay()
            gd["lsh_decode"].replay()
            join[i % 2].record(side)
        with torch.cuda.stream(stream):
            gd["h2o_prefill"].replay()
            gd["h2o_decode"].replay()
            stream.wait_event(join[i % 2])

    for i in range(max(args.warmup, 3)):
        step(i)
    torch.cuda.synchronize()
    if world > 1:
        dist.barrier()
    torch.cuda.synchronize()
    start = torch.cuda.Event(enable_timing=True)
    end = torch.cuda.Event(enable_timing=True)
    start.record(stream)
    for i in range(args.steps):
        step(i)
    end.record(stream)
    torch.cuda.synchronize()
    if world > 1:
        dist.barrier()
    for h in handles:
        L.h2o_sync(h)
    ms = max_over_ranks(start.elapsed_time(end), world, device="cuda") / args.steps
    return {"value": world * units_per_step / (ms / 1000.0), "unit": UNIT, "ms_per_step": ms, "steps": args.steps,
            "schedule": "H2O job and HashEvict job on two streams, joined every step"}


def run_e2e(args, L, torch, layers, h2o, lsh, out_h, out_l, vic_h, vic_l, W, S, NL, T, stream, world):
    """Same job through the public API, eager, with every input copied in from
    pinned host memory and every output copied out inside the timed region."""
    host_in = []
    for g in layers:
        host_in.append({k: g[k].cpu().pin_memory() for k in ("Q", "K", "V", "q", "k", "v")})
    host_out = [(torch.empty(o.shape, dtype=o.dtype).pin_memory(), torch.empty(o2.shape, dtype=o2.dtype).pin_memory(),
                 torch.empty(v.shape, dtype=v.dtype).pin_memory(), torch.empty(v2.shape, dtype=v2.dtype).pin_memory())
                for o, o2, v, v2 in zip(out_h, out_l, vic_h, vic_l)]
    h2d = sum(x.numel() * x.element_size() for hi in host_in for x in hi.values())
    d2h = sum(x.numel() * x.element_size() for ho in host_out for x in ho)

    copy_stream = torch.cuda.Stream()
    ready = [torch.cuda.Event() for _ in range(NL)]
    ready_dec = torch.cuda.Event()
    h2o_done = torch.cuda.Event()
    out_h_home = torch.cuda.Event()
    # raw device addresses of every per-step argument, computed once (the
    # binding takes plain integers; no tensor views per call)
    def rows(x):
        base, stride = x.data_ptr(), x.stride(0) * x.element_size()
        return [base + t * stride for t in range(x.shape[0])]
    ptr = [{k: rows(layers[li][k]) for k in ("q", "k", "v")} for li in range(NL)]
    optr = [(rows(out_h[li]), rows(out_l[li]), rows(vic_h[li]), rows(vic_l[li])) for li in range(NL)]
    hh = [int(h) for h in h2o]
    hl = [int(h) for h in lsh]

    def step():
        # inputs stream in on a copy stream: every layer's prompt rows first
        # (each layer's prompt phase waits only for its own), the decode
        # steps' rows last; the H2O outputs go home while the HashEvict
        # steps run
        with torch.cuda.stream(copy_stream):
            copy_stream.wait_stream(stream)
            for li in range(NL):
                for k in ("Q", "K", "V"):
                    layers[li][k].copy_(host_in[li][k], non_blocking=True)
                ready[li].record(copy_stream)
            for li in range(NL):
                for k in ("q", "k", "v"):
                    layers[li][k].copy_(host_in[li][k], non_blocking=True)
            ready_dec.record(copy_stream)
        with torch.cuda.stream(stream):
            for li in range(NL):
                stream.wait_event(ready[li])
                g = layers[li]
                L.h2o_prefill(h2o[li], g["Q"], g["K"], g["V"], T)
                L.lsh_prefill(lsh[li], g["Q"], g["K"], g["V"], T)
            stream.wait_event(ready_dec)
            for t in range(S):
                for li in range(NL):
                    pp, op = ptr[li], optr[li]
                    L.h2o_decode_step(hh[li], pp["q"][t], pp["k"][t], pp["v"][t], op[0][t], op[2][t])
            h2o_done.record(stream)
        with torch.cuda.stream(copy_stream):
            copy_stream.wait_event(h2o_done)
            for li in range(NL):
                host_out[li][0].copy_(out_h[li], non_blocking=True)
                host_out[li][2].copy_(vic_h[li], non_blocking=True)
            out_h_home.record(copy_stream)
        with torch.cuda.stream(stream):
            for t in range(S):
                for li in range(NL):
                    pp, op = ptr[li], optr[li]
                    L.lsh_decode_step(hl[li], pp["q"][t], pp["k"][t], pp["v"][t], op[1][t], op[3][t])
            for li in range(NL):
                host_out[li][1].copy_(out_l[li], non_blocking=True)
                host_out[li][3].copy_(vic_l[li], non_blocking=True)
            stream.wait_event(out_h_home)

    step()
    torch.cuda.synchronize()
    # One step's calls -- the input copies, every prompt and decode call and
    # the output copies -- captured once into a CUDA graph (all step state
    # lives on the device, so a replay is a new step); a replay still moves
    # every input in and every output out.  Eager launches are the fallback.
    run = step
    mode = "eager"
    try:
        gr = torch.cuda.CUDAGraph()
        with torch.cuda.stream(stream):
            gr.capture_begin()
            step()
            gr.capture_end()
        torch.cuda.synchronize()

        def run():
            with torch.cuda.stream(stream):
                gr.replay()
        run()
        torch.cuda.synchronize()
        mode = "graph"
    except Exception as e:  # capture unsupported: keep the eager loop
        print("e2e: graph capture failed (%s); timing eager calls" % e, file=sys.stderr)
        torch.cuda.synchronize()
    secs, each = time_e2e_steps(args, run, torch)
    value = world * 2 * S * NL / secs
    return {"value": value, "unit": UNIT, "h2d_bytes_per_step": h2d, "d2h_bytes_per_step": d2h,
            "ms_per_step": secs * 1000.0, "steps": len(each), "ms_each": each, "statistic": "median",
            "launch": mode}


def time_e2e_steps(args, run, torch):
    """Each end-to-end step timed on its own (host clock, device synchronised
    on both sides); returns the median seconds and every step's ms.  The
    host-device link is shared with other GPUs of the machine, so single
    steps can be slowed by traffic that is not this job's."""
    n = max(1, min(args.steps, 5))
    each = []
    for _ in range(n):
        torch.cuda.synchronize()
        t0 = time.perf_counter()
        run()
        torch.cuda.synchronize()
        each.append(time.perf_counter() - t0)
    return statistics.median(each), [round(1000.0 * x, 3) for x in each]


def run_single(args, variant):
    """One eviction rule alone: H2O on the grouped-query layer ("gqa") or the
    persistence-of-importance rule on the OPT-6.7B-shaped layer ("sh").  L
    layer caches, prompt phase then S decode steps token-major over the
    layers, replayed from CUDA graphs with inputs in HBM; e2e through the
    public API with host copies."""
    import torch
    import torch.distributed as dist

    from kv_cache_eviction_h2o_gb300 import binding as L
    from kv_cache_eviction_h2o_gb300 import build as lib_build
    from kv_cache_eviction_h2o_gb300 import workloads as wl

    world, rank, local = dist_setup(args)
    torch.cuda.set_device(local)
    if world > 1:
        dist.init_process_group("nccl", device_id=torch.device("cuda", local))
    lib_build.build()
    L.lib()
    gqa = variant == "gqa"
    w = wl.WORKLOADS[GQA_WORKLOAD if gqa else WORKLOAD]
    S = args.decode_steps or w.steps
    NL = args.layers
    U, G, T, d, B = w.units, w.groups, w.prompt, w.head_dim, w.budget
    dt = L.H2O_BF16 | (L.H2O_KV8 if args.kv8 else 0)
    stream = torch.cuda.Stream()
    layers = []
    with torch.cuda.stream(stream):
        for li in range(NL):
            layers.append(wl.generate_device(w, seed_offset=li + 1000 * rank, steps=S))
    torch.cuda.synchronize()
    if gqa:
        hs = [L.h2o_init_gqa(B, w.heavy, w.recent, w.batch, w.heads, G, d, dt, w.scale, stream) for _ in range(NL)]
        prefill, step = L.h2o_prefill, L.h2o_decode_step
    else:
        hs = [L.sh_init(B, w.heavy, w.recent, w.batch, w.heads, d, dt, w.scale, stream) for _ in range(NL)]
        prefill, step = L.sh_prefill, L.sh_decode_step
    if args.split:
        for h in hs:
            L.h2o_set_decode_split(h, args.split)
    outs = [torch.empty((S, U * G, d), dtype=torch.float32, device="cuda") for _ in range(NL)]
    vics = [torch.empty((S, U), dtype=torch.int32, device="cuda") for _ in range(NL)]

    def pre():
        for li in range(NL):
            g = layers[li]
            prefill(hs[li], g["Q"], g["K"], g["V"], T)

    def dec():
        for t in range(S):
            for li in range(NL):
                g = layers[li]
                step(hs[li], g["q"][t], g["k"][t], g["v"][t], outs[li][t], vics[li][t])

    phases = [("h2o_prefill", pre), ("h2o_decode", dec)]
    with torch.cuda.stream(stream):
        for _, f in phases:
            f()
    for h in hs:
        L.h2o_sync(h)
    graphs = []
    with torch.cuda.stream(stream):
        for name, f in phases:
            gr = torch.cuda.CUDAGraph()
            gr.capture_begin()
            f()
            gr.capture_end()
            graphs.append((name, gr))
    torch.cuda.synchronize()

    def one_step(evs=None):
        with torch.cuda.stream(stream):
            for i, (_, gr) in enumerate(graphs):
                gr.replay()
                if evs is not None:
                    evs[i].record(stream)

    for _ in range(args.warmup):
        one_step()
    torch.cuda.synchronize()
    for h in hs:
        L.h2o_sync(h)

    clocks = Clocks(local)
    if world > 1:
        dist.barrier()
    torch.cuda.synchronize()
    clocks.start()
    time.sleep(0.3)
    start = torch.cuda.Event(enable_timing=True)
    end = torch.cuda.Event(enable_timing=True)
    step_events = [[torch.cuda.Event(enable_timing=True) for _ in graphs] for _ in range(args.steps)]
    start.record(stream)
    for i in range(args.steps):
        one_step(step_events[i])
    end.record(stream)
    torch.cuda.synchronize()
    if world > 1:
        dist.barrier()
    clk = clocks.stop()
    elapsed_ms = start.elapsed_time(end)
    phase_ms = {name: 0.0 for name, _ in graphs}
    for i in range(args.steps):
        prev = start if i == 0 else step_events[i - 1][-1]
        for j, (name, _) in enumerate(graphs):
            phase_ms[name] += prev.elapsed_time(step_events[i][j])
            prev = step_events[i][j]
    for h in hs:
        L.h2o_sync(h)
    elapsed_ms = max_over_ranks(elapsed_ms, world, device="cuda")
    K = args.steps
    ms_per_step = elapsed_ms / K
    value = world * S * NL / (ms_per_step / 1000.0)
    hbm, tf_burst, tf_sus, peak_src = load_peaks()

    t_dec = phase_ms["h2o_decode"] / (S * NL * K) / 1000.0
    by = decode_bytes_gqa(U, G, B, d, 2, args.kv8) if gqa else decode_bytes_sh(U, B, d, 2)
    ach = by / t_dec / 1e9
    dname = "h2o_decode_gqa" if gqa else "sh_decode"
    rl = [{"kernel": dname, "bound": "hbm", "achieved": ach, "peak": hbm, "unit": "GB/s",
           "frac": ach / hbm, "traffic": ncu_traffic(("h2o_gqa" if gqa else "sh") + ("_kv8" if args.kv8 else "")),
           "algorithmic_bytes": by, "launch_us": t_dec * 1e6, "peak_source": peak_src,
           "share": phase_ms["h2o_decode"] / elapsed_ms}]
    t_pre = phase_ms["h2o_prefill"] / (NL * K) / 1000.0
    if gqa:
        fl = prefill_flops(U * G, T, d)
        ach = fl / t_pre / 1e12
        rl.append({"kernel": "h2o_prefill_gqa", "bound": "tensor", "achieved": ach, "peak": tf_sus,
                   "unit": "TFLOP/s", "frac": ach / tf_sus, "traffic": None, "algorithmic_flops": fl,
                   "launch_us": t_pre * 1e6, "peak_source": peak_src,
                   "share": phase_ms["h2o_prefill"] / elapsed_ms})
    else:
        rl.append({"kernel": "sh_prefill", "bound": "latency", "launch_us": t_pre * 1e6,
                   "share": phase_ms["h2o_prefill"] / elapsed_ms})
    dominant = max((r for r in rl if "achieved" in r), key=lambda r: r["share"])
    main_rl = {k: dominant[k] for k in ("bound", "achieved", "peak", "unit", "frac", "traffic")}
    main_rl["kernel"] = dominant["kernel"]
    main_rl["peak_source"] = peak_src

    e2e = None
    if not args.no_e2e:
        e2e = run_e2e_single(args, L, torch, layers, hs, outs, vics, S, NL, T, stream, world, prefill, step)
    cpu = None
    if rank == 0 and world == 1 and not args.no_cpu:
        n = max(1, args.oracle_units // 4)
        if gqa:
            secs, threads = oracle_job_gqa(w, list(range(n)), S, args.kv8)
        else:
            secs, threads = oracle_job_sh(w, list(range(n)), S)
        cpu = {"value": S / (secs * U / n), "unit": UNIT, "cores": threads, "kind": "oracle",
               "sample": "%d of %d cache units of one layer (prompt %d, %d decode steps, %s), %.1f s"
                         % (n, U, T, S, "H2O" if gqa else "persistence of importance", secs)}
    line = {
        "metric": METRIC, "value": value, "unit": UNIT, "n_gpus": world, "steps": K, "warmup": args.warmup,
        "ms_per_step": ms_per_step, "higher_is_better": True, "scaling": "weak", "vs_baseline": None,
        "dtype": "bf16", "data": "synthetic",
        "config": {"workload": gqa_config_name(w, S, NL, args.kv8) if gqa else sh_config_name(w, S, NL),
                   "cache": "int8 codes + fp32 scale per row" if args.kv8 else "bf16",
                   "batch": w.batch, "kv_heads": w.heads, "groups": G, "head_dim": d, "prompt": T,
                   "decode_steps": S, "budget": B, "layers": NL, "global_batch": w.batch * world,
                   "parallelism": "replicas" if world > 1 else "single",
                   "l2": "inputs larger than L2: %d layer caches (%.0f MB) + prompts (%.0f MB); a cache is reused "
                         "only after %d others" % (NL, NL * by / 1e6, NL * (G + 2) * U * T * d * 2 / 1e6, NL - 1),
                   "step": "one decode step = all %d cache units (%d query heads) of one layer cache advance one "
                           "token; prompt phases inside the timed step" % (U, U * G)},
        "roofline": main_rl,
        "rooflines": rl,
        "phases_ms_per_step": {k: v / K for k, v in phase_ms.items()},
        "cpu_baseline": cpu,
        "clocks": clk,
        "e2e": e2e,
        # prompt launches per layer: row statistics, column sums, head sums,
        # selection, gather (grouped-query); row statistics, flags, selection,
        # gather (persistence rule, tensor-core path); one launch per decode step
        "gpu_launches": (NL * (5 if gqa else 4) + S * NL) * K,
    }
    for h in hs:
        L.h2o_destroy(h)
    if rank == 0:
        print(json.dumps(line))
    if world > 1:
        dist.destroy_process_group()


def run_e2e_single(args, L, torch, layers, hs, outs, vics, S, NL, T, stream, world, prefill, step_call):
    """The single-rule job through the public API: every input copied in
    from pinned host memory and every output copied out inside the timed
    region, one step captured into a CUDA graph."""
    host_in = [{k: g[k].cpu().pin_memory() for k in ("Q", "K", "V", "q", "k", "v")} for g in layers]
    host_out = [(torch.empty(o.shape, dtype=o.dtype).pin_memory(), torch.empty(v.shape, dtype=v.dtype).pin_memory())
                for o, v in zip(outs, vics)]
    h2d = sum(x.numel() * x.element_size() for hi in host_in for x in hi.values())
    d2h = sum(x.numel() * x.element_size() for ho in host_out for x in ho)
    copy_stream = torch.cuda.Stream()
    ready = [torch.cuda.Event() for _ in range(NL)]
    ready_dec = torch.cuda.Event()

    def step():
        with torch.cuda.stream(copy_stream):
            copy_stream.wait_stream(stream)
            for li in range(NL):
                for k in ("Q", "K", "V"):
                    layers[li][k].copy_(host_in[li][k], non_blocking=True)
                ready[li].record(copy_stream)
            for li in range(NL):
                for k in ("q", "k", "v"):
                    layers[li][k].copy_(host_in[li][k], non_blocking=True)
            ready_dec.record(copy_stream)
        with torch.cuda.stream(stream):
            for li in range(NL):
                stream.wait_event(ready[li])
                g = layers[li]
                prefill(hs[li], g["Q"], g["K"], g["V"], T)
            stream.wait_event(ready_dec)
            for t in range(S):
                for li in range(NL):
                    g = layers[li]
                    step_call(hs[li], g["q"][t], g["k"][t], g["v"][t], outs[li][t], vics[li][t])
            for li in range(NL):
                host_out[li][0].copy_(outs[li], non_blocking=True)
                host_out[li][1].copy_(vics[li], non_blocking=True)

    step()
    torch.cuda.synchronize()
    gr = torch.cuda.CUDAGraph()
    with torch.cuda.stream(stream):
        gr.capture_begin()
        step()
        gr.capture_end()
    torch.cuda.synchronize()

    def run():
        with torch.cuda.stream(stream):
            gr.replay()
    run()
    torch.cuda.synchronize()
    secs, each = time_e2e_steps(args, run, torch)
    return {"value": world * S * NL / secs, "unit": UNIT, "h2d_bytes_per_step": h2d, "d2h_bytes_per_step": d2h,
            "ms_per_step": secs * 1000.0, "steps": len(each), "ms_each": each, "statistic": "median",
            "launch": "graph"}


def main():
    args = parse()
    if args.impl == "reference":
        run_reference(args)
    elif args.gqa or args.sh:
        run_single(args, "gqa" if args.gqa else "sh")
    else:
        run_ours(args)


if __name__ == "__main__":
    main()
