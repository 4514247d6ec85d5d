#!/usr/bin/env python3
"""Whole-job throughput of the budgeted-KV decode path on GB300.

One bench step is one pass of the hot path over one batch of synthetic input
shaped like an attention layer of the named configuration:

  for each of L layer caches: the prompt phase (H2O: row statistics and
  column sums on the tensor cores, top-k, gather; HashEvict: sign codes,
  replacement replay, gather), then S decode steps (attend, accumulate,
  evict, insert), token-major over the L layers, as a model decodes.

The default configuration is the OPT-30B-shaped layer in its throughput
regime (64 x 56 heads, head_dim 128, prompt 512, 1024 decode steps, budget
308 = 154 heavy + 154 recent, bf16): the largest single-GPU configuration,
the one the headline value is quoted on.  Its value is H2O decode steps per
second, one decode step being all batch x head units of one layer cache
advancing one token.  The same run then measures the other configurations as
sub-records (each with its own timed region, rooflines and CPU baseline):
the OPT-6.7B-shaped layer, the Llama-7B-shaped 32K-token context and the
HashEvict variant on the OPT-6.7B shapes.

Every layer cache is used again only after the L - 1 others, and the caches
plus the prompts exceed L2, so decode reads come from HBM.  The device-timed
value replays the step from CUDA graphs with inputs already in HBM; the e2e
value drives the same job through the public API with pinned host inputs
copied in and outputs copied out inside the timed region.  The CPU oracle is
timed on a bounded sample of the same job.

    python bench.py [--gpus N] [--steps K] [--warmup W] [--config NAME]
                    [--rule h2o|sh] [--kv8 | --kv4] [--impl reference] [--no-sub]
"""
import argparse
import hashlib
import json
import os
import statistics
import subprocess
import sys
import time

import numpy as np

ROOT = os.path.dirname(os.path.abspath(__file__))
if ROOT not in sys.path:
    sys.path.insert(0, ROOT)

METRIC = "H2O decode steps/s (batch×heads) at 1 GB300; achieved HBM GB/s vs peak"
UNIT = "steps/s"
TRAFFIC_FILE = os.path.join(ROOT, "profiles", "ncu_traffic.json")

# name -> (workload, eviction rule, layer caches in rotation, quantised slots:
# 0 = bf16 rows, 8 = int8 codes, 4 = 4-bit codes).
# The layer count keeps the caches plus prompts well above L2 (129 MB) and
# makes every cache wait for the others before it is read again.
CONFIGS = {
    "opt-30b": ("opt-30b", "h2o", 2, 0),                    # 2 x 594 MB caches
    "opt-6.7b": ("opt-6.7b", "h2o", 8, 0),                  # 8 x 113 MB
    "llama-7b-32k": ("llama-7b-32k", "h2o", 8, 0),          # 8 x 70 MB
    "hashevict-opt-6.7b": ("hashevict-opt-6.7b", "lsh", 8, 0),
    "fastgen-opt-6.7b": ("fastgen-opt-6.7b", "fg", 8, 0),   # per-head policies, mixed budgets
    "gqa-8x8x4": ("gqa-8x8x4", "h2o", 8, 0),                # caches shared by 4 query heads
    "opt-30b-int8": ("opt-30b", "h2o", 2, 8),               # the main layer with int8 slots
    "opt-30b-int4": ("opt-30b", "h2o", 2, 4),               # ... and with 4-bit slots
}
DEFAULT_CONFIG = "opt-30b"
SUB_CONFIGS = ("opt-6.7b", "llama-7b-32k", "hashevict-opt-6.7b", "fastgen-opt-6.7b", "gqa-8x8x4", "opt-30b-int8",
               "opt-30b-int4")


def parse(argv=None):
    p = argparse.ArgumentParser()
    p.add_argument("--gpus", type=int, default=1)
    p.add_argument("--steps", type=int, default=10)
    p.add_argument("--warmup", type=int, default=3)
    p.add_argument("--impl", default="ours", choices=["ours", "reference"])
    p.add_argument("--config", default=DEFAULT_CONFIG, choices=sorted(CONFIGS))
    p.add_argument("--rule", default=None, choices=["h2o", "sh"],
                   help="eviction rule on an H2O workload: h2o (accumulated attention) or sh "
                        "(persistence of importance); default: the configuration's own")
    p.add_argument("--layers", type=int, default=None, help="layer caches in rotation (default per config)")
    p.add_argument("--decode-steps", type=int, default=None)
    p.add_argument("--split", type=int, default=0, help="CTAs per unit in decode (0 = automatic)")
    p.add_argument("--oracle-seconds", type=float, default=10.0,
                   help="CPU work the oracle sample of the main configuration aims at")
    p.add_argument("--oracle-units", type=int, default=0,
                   help="units per oracle sample of the reference arm (default: the host's threads)")
    p.add_argument("--no-e2e", action="store_true")
    p.add_argument("--no-cpu", action="store_true")
    p.add_argument("--no-sub", action="store_true", help="measure the main configuration only")
    p.add_argument("--sub", default=None, help="comma-separated sub-record configurations (default: %s)"
                   % ",".join(SUB_CONFIGS))
    p.add_argument("--kv8", action="store_true", help="int8 cache slots (one fp32 scale per row)")
    p.add_argument("--kv4", action="store_true", help="4-bit cache slots (one fp32 scale per row)")
    # older spellings
    p.add_argument("--gqa", action="store_true", help="same as --config gqa-8x8x4")
    p.add_argument("--sh", action="store_true", help="same as --config opt-6.7b --rule sh")
    a = p.parse_args(argv)
    if a.gqa:
        a.config = "gqa-8x8x4"
    if a.sh:
        a.config, a.rule = ("opt-6.7b" if a.config == DEFAULT_CONFIG else a.config), "sh"
    if a.kv8 and a.kv4:
        p.error("--kv8 and --kv4 are exclusive")
    return a


def qbits(args, q0):
    """Cache row form of a run: the flags, else the configuration's own."""
    return 8 if args.kv8 else 4 if args.kv4 else q0


def code_row(d, eb, qb):
    """Bytes of one stored row: the input type, int8 or 4-bit codes."""
    return d if qb == 8 else d // 2 if qb == 4 else d * eb


# ------------------------------------------------------------------ helpers

def load_peaks():
    path = os.path.join(ROOT, "MEASURED_PEAKS.json")
    try:
        with open(path) as f:
            d = json.load(f)
        return (float(d["hbm_gbs"]), float(d["bf16_tflops"]),
                float(d.get("bf16_tflops_sustained", d["bf16_tflops"])), "measured")
    except Exception:
        return 6800.0, 1900.0, 1700.0, "fallback"


def file_digest(*names):
    h = hashlib.sha256()
    for n in names:
        with open(os.path.join(ROOT, "kv_cache_eviction_h2o_gb300", "csrc", n), "rb") as f:
            h.update(f.read())
    return h.hexdigest()[:16]


def ncu_traffic(key):
    """Per-launch DRAM bytes from the committed ncu capture, if it was taken
    on the current kernel source; None otherwise."""
    try:
        with open(TRAFFIC_FILE) as f:
            d = json.load(f)
        e = d[key]
        if e["source_digest"] != file_digest(*e["sources"]):
            return None
        return float(e["bytes_per_launch"])
    except Exception:
        return None


class Clocks:
    """nvidia-smi sampler for the timed regions."""
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
        return summarize_clocks(out)


def summarize_clocks(text):
    rows = []
    for line in text.strip().splitlines():
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


def dist_setup():
    world = int(os.environ.get("WORLD_SIZE", "1"))
    rank = int(os.environ.get("RANK", "0"))
    local = int(os.environ.get("LOCAL_RANK", "0"))
    return world, rank, local


# ------------------------------------------------------------ algorithmic

def decode_bytes(U, B, d, eb, lsh, qb=0):
    """Algorithmic HBM bytes of one full-cache decode launch over U units:
    per live slot K and V rows (int8 or 4-bit codes plus an 8-byte scale
    pair with qb 8 or 4), plus score read+write (8-byte fp32 pair) and position read (H2O)
    or code and position read (HashEvict); per unit q, k, v in, fp32 out,
    one K/V row written (and its scale pair), victim score/code and
    position written, unit state read and written; plus the projection
    matrix once."""
    row = d * eb
    crow = code_row(d, eb, qb)
    sc = 8 if qb else 0
    if lsh:
        per_slot = 2 * crow + sc + 4 + 4
        fixed = 3 * row + 4 * d + 2 * crow + sc + 4 + 4 + 16
        return U * (B * per_slot + fixed) + d * 32 * 4
    per_slot = 2 * crow + sc + 8 + 8 + 4
    fixed = 3 * row + 4 * d + 2 * crow + sc + 8 + 4 + 16
    return U * (B * per_slot + fixed)


def method_bytes(U, B, d, eb):
    """The method's own bytes per H2O step (one fp32 score per slot, no
    pair): 2 rows + 4 + 4 + 4 per live slot, 1804 B per unit at d = 128."""
    return U * (B * (2 * d * eb + 12) + 3 * d * eb + 4 * d + 2 * d * eb + 12)


def decode_bytes_gqa(U, G, B, d, eb, qb=0):
    """Algorithmic HBM bytes of one full-cache grouped-query H2O decode launch
    over U cache units of G query heads: per live slot K and V rows (int8 or
    4-bit codes plus an 8-byte scale pair with qb 8 or 4), score read+write and position
    read, each once per unit (the heads share them); per query head q in and
    fp32 out; per unit k, v in, one K/V row written (and its scale pair),
    victim score and position written, unit state read and written."""
    row = d * eb
    crow = code_row(d, eb, qb)
    sc = 8 if qb else 0
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


def prefill_bytes(U, G, T, d, B, qb=0, fg=False):
    """Algorithmic HBM bytes of one H2O prompt phase (U cache units, G query
    heads each): each score pass reads Q and K once; pass 1 writes the row
    max and normaliser (4 + 4 B per query row) that pass 2 reads; pass 2
    writes the fp64 column sums that the selection reads (per query head,
    then per unit, for G > 1); the gather reads the kept prompt rows of K
    and V and writes the slots' rows (codes and a scale pair when
    quantised), positions and 8-byte score pairs.  Per-head policies add
    two fp64 band sums per key, written and read."""
    rows = U * G * T * d * 2 + U * T * d * 2
    stats = 2 * U * G * T * 8
    cols = 2 * U * G * T * 8 + (2 * U * T * 8 if G > 1 else 0)
    kept = min(B, T)
    gather = U * kept * d * 2 * 2 + U * B * (2 * code_row(d, 2, qb) + (8 if qb else 0) + 4 + 8)
    band = 2 * 2 * U * T * 8 if fg else 0
    return 2 * rows + stats + cols + gather + band


def lsh_code_flops(U, T, d):
    """Prompt sign codes: 32 fp32 multiply-add chains of d terms for every
    query and key row (2 flops per multiply-add)."""
    return 2 * U * T * 2 * d * 32


def prompt_launches(rule, G):
    """Kernels one prompt phase launches: row statistics, column sums,
    selection, gather (H2O; + head sums for a grouped-query cache); sign
    codes, replay, gather (HashEvict); row statistics, flags, selection,
    gather (persistence rule, tensor-core path)."""
    if rule == "lsh":
        return 3
    if rule == "sh":
        return 4
    if rule == "fg":
        return 6          # row statistics, column and band sums, selection, policy, unit lists, gather
    return 5 if G > 1 else 4


# ------------------------------------------------------------------ oracle

ORACLE_MAX_PROMPT = 4096


def oracle_job(w, rule, units, S, qb=0, prompt=None):
    """The CPU oracle on a sample of units of workload w: the prompt phase
    (of `prompt` tokens, default the workload's) and S decode steps of the
    rule.  Returns (prompt seconds, decode seconds, threads)."""
    import oracle
    from kv_cache_eviction_h2o_gb300 import workloads as wl
    T = prompt or w.prompt
    g = wl.generate(w, units=units, steps=S, prompt=T)
    t0 = time.perf_counter()
    if rule == "lsh":
        W = g["W"]
        st = oracle.lsh_prefill(g["Q"], g["K"], g["V"], W, w.budget, w.recent)
        if qb:
            oracle.kv8(st, qb)
        t1 = time.perf_counter()
        for t in range(S):
            oracle.lsh_decode_step(st, g["q"][t], g["k"][t], g["v"][t], W, T + t, w.recent, w.scale)
    elif rule == "sh":
        st, _, _, _ = oracle.sh_prefill(g["Q"], g["K"], g["V"], w.budget, w.heavy, w.recent, w.scale)
        t1 = time.perf_counter()
        for t in range(S):
            oracle.sh_decode_step(st, g["q"][t], g["k"][t], g["v"][t], T + t, w.recent, w.scale)
    elif rule == "fg":
        _, states, params = oracle.fg_prefill(g["Q"], g["K"], g["V"], w.budget, w.heavy, w.recent, w.scale, w.tau,
                                              w.full_budget)
        t1 = time.perf_counter()
        for t in range(S):
            oracle.fg_decode_step(states, params, g["q"][t], g["k"][t], g["v"][t], T + t, w.scale)
    elif w.groups > 1:
        st, _, _, _, _ = oracle.h2o_prefill_gqa(g["Q"], g["K"], g["V"], w.budget, w.heavy, w.recent, w.scale)
        if qb:
            oracle.kv8(st, qb)
        t1 = time.perf_counter()
        for t in range(S):
            oracle.h2o_decode_step_gqa(st, g["q"][t], g["k"][t], g["v"][t], T + t, w.recent, w.scale)
    else:
        st, _, _, _ = oracle.h2o_prefill(g["Q"], g["K"], g["V"], w.budget, w.heavy, w.recent, w.scale)
        if qb:
            oracle.kv8(st, qb)
        t1 = time.perf_counter()
        for t in range(S):
            oracle.h2o_decode_step(st, g["q"][t], g["k"][t], g["v"][t], T + t, w.recent, w.scale)
    t2 = time.perf_counter()
    return t1 - t0, t2 - t1, oracle.get_threads()


class OracleSample:
    """The oracle timed on a bounded sample of a configuration's job, scaled
    to the metric (decode steps per second, one step = all units of one
    layer cache advancing one token, the prompt phase included).  Units:
    the host's thread count, then once more with as many as the target time
    allows.  A prompt longer than ORACLE_MAX_PROMPT (H2O only, whose prompt
    work grows with the causal pair count) is timed on its first
    ORACLE_MAX_PROMPT rows and scaled by the pair count."""

    def __init__(self, w, rule, qb, target_s, units=None, steps=None):
        import oracle
        self.w, self.rule, self.qb = w, rule, qb
        self.S = steps or w.steps
        self.Tp = w.prompt
        if w.prompt > ORACLE_MAX_PROMPT:
            assert rule == "h2o", "prompt truncation is only scaled for the H2O prompt phase"
            self.Tp = ORACLE_MAX_PROMPT
        self.pair_scale = (w.prompt * (w.prompt + 1)) / (self.Tp * (self.Tp + 1))
        n = min(w.units, units or max(1, oracle.get_threads()))
        tp, td, th = oracle_job(w, rule, list(range(n)), self.S, qb, self.Tp)
        if units is None and tp + td < target_s / 2 and n < w.units:
            n = min(w.units, max(n + 1, int(n * target_s / max(tp + td, 1e-3))))
            tp, td, th = oracle_job(w, rule, list(range(n)), self.S, qb, self.Tp)
        self.n, self.tp, self.td, self.threads = n, tp, td, th

    def seconds(self):
        return self.tp + self.td

    def layer_job_seconds(self):
        return (self.tp * self.pair_scale + self.td) * self.w.units / self.n

    def rate(self):
        return self.S / self.layer_job_seconds()

    def describe(self):
        w = self.w
        if self.Tp != w.prompt:
            pr = "prompt phase on the first %d of %d rows, scaled x%.1f by the causal pair count" % (
                self.Tp, w.prompt, self.pair_scale)
        else:
            pr = "prompt %d" % w.prompt
        return "%d of %d units of one layer (%s, %d decode steps, %s), %.1f s" % (
            self.n, w.units, pr, self.S, rule_name(self.rule, w), self.seconds())

    def record(self, single_thread=False):
        rec = {"value": self.rate(), "unit": UNIT, "cores": self.threads, "kind": "oracle",
               "sample": self.describe()}
        if single_thread and self.threads > 1:
            # the same oracle on one thread, over the units one of the
            # sample's threads took
            import oracle
            n1 = max(1, self.n // self.threads)
            try:
                oracle.set_threads(1)
                tp, td, _ = oracle_job(self.w, self.rule, list(range(n1)), self.S, self.qb, self.Tp)
            finally:
                oracle.set_threads(self.threads)
            rate = self.S / ((tp * self.pair_scale + td) * self.w.units / n1)
            rec["single_thread"] = {"value": rate, "unit": UNIT, "cores": 1,
                                    "sample": "%d units on one thread, %.1f s" % (n1, tp + td)}
        return rec


# -------------------------------------------------------------- reference

def run_reference(args):
    """The oracle, as it stands, timed on the host cores on this run's
    configuration: each step a bounded sample of the job (the prompt phase
    and the decode steps of as many units as the host has threads)."""
    world, rank, _ = dist_setup()
    if rank != 0:
        return
    from kv_cache_eviction_h2o_gb300 import workloads as wl
    import oracle
    wname, rule0, _, q0 = CONFIGS[args.config]
    rule = args.rule or rule0
    qb = qbits(args, q0)
    w = wl.WORKLOADS[wname]
    n = min(w.units, args.oracle_units or max(1, oracle.get_threads()))
    S = args.decode_steps or w.steps
    for _ in range(args.warmup):
        OracleSample(w, rule, qb, 0, units=n, steps=S)
    samples = [OracleSample(w, rule, qb, 0, units=n, steps=S) for _ in range(args.steps)]
    per = sum(x.layer_job_seconds() for x in samples) / len(samples)
    value = S / per
    line = {
        "impl": "reference", "metric": METRIC, "value": value, "unit": UNIT, "n_gpus": world,
        "steps": args.steps, "warmup": args.warmup,
        "ms_per_step": 1000.0 * per, "higher_is_better": True, "scaling": "weak",
        "vs_baseline": None, "dtype": "f64", "data": "synthetic (seeded, shaped like the configuration's layer)",
        "config": {"workload": config_name(w, rule, S, 1, qb)},
        "cpu_baseline": {"value": value, "unit": UNIT, "cores": samples[0].threads, "kind": "oracle",
                         "sample": "per step: " + samples[0].describe()},
        "e2e": {"value": value, "unit": UNIT, "h2d_bytes_per_step": 0, "d2h_bytes_per_step": 0},
    }
    print(json.dumps(line))


def rule_name(rule, w):
    if rule == "lsh":
        return "HashEvict"
    if rule == "fg":
        return "per-head policies (local / frequency + local / full, tau %g, full budget %d)" % (w.tau, w.full_budget)
    if rule == "sh":
        return "persistence of importance"
    return "H2O" + (" grouped-query" if w.groups > 1 else "")


def config_name(w, rule, S, NL, qb):
    heads = ("%d x %d key/value heads x %d query heads" % (w.batch, w.heads, w.groups) if w.groups > 1
             else "%d x %d heads" % (w.batch, w.heads))
    split = ("recent %d" % w.recent) if rule == "lsh" else ("%d heavy + %d recent" % (w.heavy, w.recent))
    return ("%s-shaped layer x%d (%s, head_dim %d): %s, prompt %d -> %d decode steps, budget %d (%s)%s"
            % (w.name, NL, heads, w.head_dim, rule_name(rule, w), w.prompt, S, w.budget, split,
               {8: ", int8 cache slots", 4: ", 4-bit cache slots"}.get(qb, "")))


# -------------------------------------------------------------------- ours

class Job:
    """L layer caches of one configuration on the device: inputs resident
    in HBM, the handles, the prompt and decode phases as callables over the
    public API, and their algorithmic work."""

    def __init__(self, L, torch, w, rule, NL, S, qb, split, stream, rank):
        from kv_cache_eviction_h2o_gb300 import workloads as wl
        self.L, self.torch, self.w, self.rule, self.NL, self.S, self.qb = L, torch, w, rule, NL, S, qb
        self.stream = stream
        U, G, d, B = w.units, w.groups, w.head_dim, w.budget
        dt = L.H2O_BF16 | {0: 0, 8: L.H2O_KV8, 4: L.H2O_KV4}[qb]
        self.layers = []
        with torch.cuda.stream(stream):
            for li in range(NL):
                self.layers.append(wl.generate_device(w, seed_offset=li + 1000 * rank, steps=S))
        torch.cuda.synchronize()
        if rule == "lsh":
            self.W = self.layers[0]["W"]
            self.hs = [L.lsh_init(B, w.recent, w.batch, w.heads, d, dt, w.scale, self.W, stream) for _ in range(NL)]
            self.prefill_call, self.step_call = L.lsh_prefill, L.lsh_decode_step
        elif rule == "sh":
            self.hs = [L.sh_init(B, w.heavy, w.recent, w.batch, w.heads, d, dt, w.scale, stream) for _ in range(NL)]
            self.prefill_call, self.step_call = L.sh_prefill, L.sh_decode_step
        elif rule == "fg":
            self.hs = [L.fg_init(B, w.heavy, w.recent, w.full_budget, w.tau, w.batch, w.heads, d, dt, w.scale, stream)
                       for _ in range(NL)]
            self.prefill_call, self.step_call = L.fg_prefill, L.fg_decode_step
        elif G > 1:
            self.hs = [L.h2o_init_gqa(B, w.heavy, w.recent, w.batch, w.heads, G, d, dt, w.scale, stream)
                       for _ in range(NL)]
            self.prefill_call, self.step_call = L.h2o_prefill, L.h2o_decode_step
        else:
            self.hs = [L.h2o_init(B, w.heavy, w.recent, w.batch, w.heads, d, dt, w.scale, stream)
                       for _ in range(NL)]
            self.prefill_call, self.step_call = L.h2o_prefill, L.h2o_decode_step
        if split:
            for h in self.hs:
                L.h2o_set_decode_split(h, split)
        self.outs = [torch.empty((S, U * G, d), dtype=torch.float32, device="cuda") for _ in range(NL)]
        self.vics = [torch.empty((S, U), dtype=torch.int32, device="cuda") for _ in range(NL)]
        # raw device addresses of every per-step argument (the binding takes
        # plain integers; no tensor views per call)

        def rows(x):
            base, stride = x.data_ptr(), x.stride(0) * x.element_size()
            return [base + t * stride for t in range(x.shape[0])]
        self.ptr = [{k: rows(g[k]) for k in ("q", "k", "v")} for g in self.layers]
        self.optr = [(rows(o), rows(v)) for o, v in zip(self.outs, self.vics)]
        self.hh = [int(h) for h in self.hs]
        self.graphs = None

    # the two phases, over the public API
    def prefill(self):
        T = self.w.prompt
        for li in range(self.NL):
            g = self.layers[li]
            self.prefill_call(self.hs[li], g["Q"], g["K"], g["V"], T)

    def decode(self, t0=0, t1=None):
        step = self.step_call
        for t in range(t0, self.S if t1 is None else t1):
            for li in range(self.NL):
                pp, op = self.ptr[li], self.optr[li]
                step(self.hh[li], pp["q"][t], pp["k"][t], pp["v"][t], op[0][t], op[1][t])

    def sync(self):
        for h in self.hs:
            self.L.h2o_sync(h)

    def capture(self):
        torch = self.torch
        phases = [("prefill", self.prefill), ("decode", self.decode)]
        with torch.cuda.stream(self.stream):      # eager pass: scratch, kernel attributes, errors
            for _, f in phases:
                f()
        self.sync()
        self.graphs = []
        with torch.cuda.stream(self.stream):
            for name, f in phases:
                gr = torch.cuda.CUDAGraph()
                gr.capture_begin()
                f()
                gr.capture_end()
                self.graphs.append((name, gr))
        torch.cuda.synchronize()

    def one_step(self, evs=None):
        with self.torch.cuda.stream(self.stream):
            for i, (_, gr) in enumerate(self.graphs):
                gr.replay()
                if evs is not None:
                    evs[i].record(self.stream)

    def time(self, K, W, world):
        """W warm-up steps, then K steps bracketed by a barrier and device
        synchronisation; device events after every phase.  Returns
        (elapsed ms max over ranks, per-phase ms summed over the K steps)."""
        torch = self.torch
        import torch.distributed as dist
        for _ in range(W):
            self.one_step()
        torch.cuda.synchronize()
        self.sync()
        if world > 1:
            dist.barrier()
        torch.cuda.synchronize()
        start = torch.cuda.Event(enable_timing=True)
        end = torch.cuda.Event(enable_timing=True)
        evs = [[torch.cuda.Event(enable_timing=True) for _ in self.graphs] for _ in range(K)]
        start.record(self.stream)
        for i in range(K):
            self.one_step(evs[i])
        end.record(self.stream)
        torch.cuda.synchronize()
        if world > 1:
            dist.barrier()
        elapsed = start.elapsed_time(end)
        phase = {name: 0.0 for name, _ in self.graphs}
        for i in range(K):
            prev = start if i == 0 else evs[i - 1][-1]
            for j, (name, _) in enumerate(self.graphs):
                phase[name] += prev.elapsed_time(evs[i][j])
                prev = evs[i][j]
        self.sync()
        return max_over_ranks(elapsed, world, device="cuda"), phase

    # algorithmic work of one launch / phase
    def l2_hot(self, n=64, reps=5):
        """Decode launches on ONE layer cache, repeated: for caches that fit
        in L2 (129 MB) the rows then come from L2, so this is labelled apart
        from the HBM numbers.  Layer 0 is prompted, its first n decode steps
        captured in a graph and replayed; the median replay per launch."""
        torch = self.torch
        n = min(n, self.S)
        g = self.layers[0]
        h, pp, op = self.hh[0], self.ptr[0], self.optr[0]
        step = self.step_call

        def steps():
            for t in range(n):
                step(h, pp["q"][t], pp["k"][t], pp["v"][t], op[0][t], op[1][t])
        with torch.cuda.stream(self.stream):
            self.prefill_call(self.hs[0], g["Q"], g["K"], g["V"], self.w.prompt)
            steps()
            gr = torch.cuda.CUDAGraph()
            gr.capture_begin()
            steps()
            gr.capture_end()
        torch.cuda.synchronize()
        each = []
        for _ in range(reps):
            a, b = torch.cuda.Event(enable_timing=True), torch.cuda.Event(enable_timing=True)
            with torch.cuda.stream(self.stream):
                self.prefill_call(self.hs[0], g["Q"], g["K"], g["V"], self.w.prompt)
                a.record(self.stream)
                gr.replay()
                b.record(self.stream)
            torch.cuda.synchronize()
            each.append(a.elapsed_time(b) * 1000.0 / (n * self.decode_launches()))
        self.sync()
        by = self.decode_launch_bytes() / self.decode_launches()
        us = statistics.median(each)
        fits = by < 129e6
        return {"decode_us_per_launch": us, "launches": n * self.decode_launches(),
                "bytes_per_launch": by, "gb_s": by / us / 1e3,
                "note": ("one layer cache decoded %d steps in a row: %.0f MB %s L2 (129 MB), so the rows %s; not an HBM "
                         "number" % (n, by / 1e6, "fits in" if fits else "exceeds",
                                     "come from L2" if fits else "still stream from HBM"))}

    def decode_kernel(self):
        if self.rule == "lsh":
            return "lsh_decode"
        if self.rule == "fg":
            return "fg_decode"
        if self.rule == "sh":
            return "sh_decode"
        return "h2o_decode_gqa" if self.w.groups > 1 else "h2o_decode"

    def decode_launch_bytes(self):
        w = self.w
        U, G, d, B = w.units, w.groups, w.head_dim, w.budget
        if self.rule == "lsh":
            return decode_bytes(U, B, d, 2, True, self.qb)
        if self.rule == "sh":
            return decode_bytes_sh(U, B, d, 2)
        if self.rule == "fg":
            # every unit on its own policy's budget; a full-cache unit grows by
            # one slot a step: the average over the S steps of each launch
            L = self.L
            pol = np.empty(U, np.int32)
            L.h2o_sync(self.hs[0])
            L.fg_get_policy(self.hs[0], pol)
            tot = 0.0
            for u in range(U):
                Bu = w.full_budget if pol[u] == 2 else B
                n0 = min(Bu, w.prompt)
                avg_n = sum(min(Bu, n0 + t) for t in range(self.S)) / self.S
                tot += decode_bytes(1, avg_n, d, 2, False)
            self.policy_mix = {int(k): int((pol == k).sum()) for k in (0, 1, 2)}
            return tot
        if G > 1:
            return decode_bytes_gqa(U, G, B, d, 2, self.qb)
        return decode_bytes(U, B, d, 2, False, self.qb)

    def traffic_key(self):
        return "%s%s@%s" % (self.decode_kernel(), {8: "_kv8", 4: "_kv4"}.get(self.qb, ""), self.w.name)

    def decode_launches(self):
        """Kernels one decode step launches: per-head policies take two (the
        compressed policies' units, then the full caches'), the rest one."""
        return 2 if self.rule == "fg" else 1

    def launches_per_step(self):
        return self.NL * (prompt_launches(self.rule, self.w.groups) + self.S * self.decode_launches())

    def destroy(self):
        for h in self.hs:
            self.L.h2o_destroy(h)
        self.hs = []
        self.graphs = None
        self.layers = self.outs = self.vics = None
        self.torch.cuda.synchronize()
        self.torch.cuda.empty_cache()


def rooflines(job, phase_ms, elapsed_ms, K):
    """Per-kernel rooflines from the live phase times (per-launch averages
    on the launching stream)."""
    hbm, tf_burst, tf_sus, peak_src = load_peaks()
    w, NL, S = job.w, job.NL, job.S
    U, G, T, d, B = w.units, w.groups, w.prompt, w.head_dim, w.budget
    rl = []
    t_launch = phase_ms["decode"] / (S * NL * K) / 1000.0
    by = job.decode_launch_bytes()
    ach = by / t_launch / 1e9
    rec = {"kernel": job.decode_kernel(), "bound": "hbm", "achieved": ach, "peak": hbm, "unit": "GB/s",
           "frac": ach / hbm, "traffic": ncu_traffic(job.traffic_key()), "algorithmic_bytes": by,
           "launch_us": t_launch * 1e6, "peak_source": peak_src, "share": phase_ms["decode"] / elapsed_ms}
    if job.decode_launches() > 1:
        # bytes and time of the step's launches together
        rec["launches_per_decode_step"] = job.decode_launches()
    if job.rule == "h2o" and G == 1 and not job.qb:
        mb = method_bytes(U, B, d, 2)
        rec["method_bytes"] = mb
        rec["method_frac"] = mb / t_launch / 1e9 / hbm
    rl.append(rec)
    t_pre = phase_ms["prefill"] / (NL * K) / 1000.0
    if job.rule in ("h2o", "fg"):
        fl = prefill_flops(U * G, T, d)
        ach = fl / t_pre / 1e12
        Bp = w.full_budget if job.rule == "fg" else B
        by = prefill_bytes(U, G, T, d, Bp, job.qb, job.rule == "fg")
        hb = by / t_pre / 1e9
        tens = {"bound": "tensor", "achieved": ach, "peak": tf_sus, "unit": "TFLOP/s", "frac": ach / tf_sus,
                "peak_source": peak_src + " (sustained)"}
        mem = {"bound": "hbm", "achieved": hb, "peak": hbm, "unit": "GB/s", "frac": hb / hbm, "peak_source": peak_src}
        # the phase is tensor-bound on long prompts and HBM-bound on short
        # ones: the nearer roof is the one reported, the other beside it
        top, other = (tens, mem) if tens["frac"] >= mem["frac"] else (mem, tens)
        rec = {"kernel": ("fg_prefill" if job.rule == "fg" else "h2o_prefill") + ("_gqa" if G > 1 else "")}
        rec.update(top)
        rec.update({"traffic": None, "algorithmic_flops": fl, "algorithmic_bytes": by, "launch_us": t_pre * 1e6,
                    "share": phase_ms["prefill"] / elapsed_ms,
                    "other_roof": {k: other[k] for k in ("bound", "achieved", "peak", "unit", "frac")}})
        rl.append(rec)
    elif job.rule == "lsh":
        rl.append({"kernel": "lsh_prefill", "bound": "latency", "launch_us": t_pre * 1e6,
                   "serial_steps": max(0, T - B),
                   "ns_per_serial_step": t_pre * 1e9 / max(1, T - B),
                   "code_flops": lsh_code_flops(U, T, d),
                   "share": phase_ms["prefill"] / elapsed_ms})
    else:
        rl.append({"kernel": "sh_prefill", "bound": "latency", "launch_us": t_pre * 1e6,
                   "share": phase_ms["prefill"] / elapsed_ms})
    return rl


def main_roofline(rl):
    measured = [r for r in rl if "achieved" in r]
    dom = max(measured, key=lambda r: r["share"])
    out = {k: dom[k] for k in ("bound", "achieved", "peak", "unit", "frac", "traffic")}
    out["kernel"] = dom["kernel"]
    out["peak_source"] = dom["peak_source"]
    return out


def l2_note(job):
    w = job.w
    by = job.decode_launch_bytes()
    prompts = job.NL * (w.groups + 2) * w.units * w.prompt * w.head_dim * 2
    return ("inputs larger than L2 (129 MB): %d layer caches (%.0f MB) + prompts (%.0f MB); a cache is "
            "reused only after %d others" % (job.NL, job.NL * by / 1e6, prompts / 1e6, job.NL - 1))


def measure(args, L, torch, cname, rule, NL, S, stream, world, rank, want_e2e, cpu_seconds, clocks=None,
            main_record=False):
    """Build, time and describe one configuration's job (clocks sampled
    during its timed region when a sampler is given; the main record's CPU
    baseline adds the oracle's single-thread rate)."""
    from kv_cache_eviction_h2o_gb300 import workloads as wl
    wname, rule0, NL0, q0 = CONFIGS[cname]
    w = wl.WORKLOADS[wname]
    rule = rule or rule0
    NL = NL or NL0
    S = S or w.steps
    qb = qbits(args, q0)
    job = Job(L, torch, w, rule, NL, S, qb, args.split, stream, rank)
    job.capture()
    if clocks is not None:
        clocks.start()
        time.sleep(0.3)
    elapsed, phase = job.time(args.steps, args.warmup, world)
    clk = clocks.stop() if clocks is not None else None
    hot = job.l2_hot()
    K = args.steps
    ms = elapsed / K
    rl = rooflines(job, phase, elapsed, K)
    mix = getattr(job, "policy_mix", None)
    rec = {
        "config": {"workload": config_name(w, rule, S, NL, qb),
                   "cache": {8: "int8 codes + fp32 scale per row", 4: "4-bit codes (two per byte) + fp32 scale per row"}
                   .get(qb, "bf16"),
                   "batch": w.batch, "heads": w.heads, "groups": w.groups, "head_dim": w.head_dim,
                   "prompt": w.prompt, "decode_steps": S, "budget": w.budget, "heavy": w.heavy,
                   "recent": w.recent, "layers": NL, "l2": l2_note(job),
                   "step": "one decode step = all %d units of one layer cache advance one token (%s); prompt "
                           "phases inside the timed step" % (w.units, rule_name(rule, w))},
        "value": world * S * NL / (ms / 1000.0), "unit": UNIT, "ms_per_step": ms,
        "head_steps_per_s": world * S * NL * w.query_units / (ms / 1000.0),
        "roofline": main_roofline(rl), "rooflines": rl,
        "launch_us": {r["kernel"]: r["launch_us"] for r in rl},
        "phases_ms_per_step": {k: v / K for k, v in phase.items()},
        "gpu_launches": job.launches_per_step() * K,
        "l2_hot": hot,
    }
    if want_e2e:
        rec["e2e"] = run_e2e(job, world)
    job.destroy()
    del job
    rec["clocks"] = clk
    rec["cpu_baseline"] = None
    if rank == 0 and world == 1 and cpu_seconds > 0:
        rec["cpu_baseline"] = OracleSample(w, rule, qb, cpu_seconds, steps=S).record(single_thread=main_record)
    if mix:
        rec["policies"] = {"local": mix[0], "frequency+local": mix[1], "full": mix[2]}
    return rec


def run_e2e(job, world, chunk_steps=64):
    """The job through the public API: every input copied in from pinned host
    memory and every output copied out inside the timed region, one step
    captured into a CUDA graph (all step state lives on the device, so a
    replay is a new step that still moves every input in and every output
    out).  The copies are pipelined with the compute on two copy streams:
    each layer's prompt rows ahead of its prompt phase, the decode rows in
    chunks of `chunk_steps` steps ahead of the chunk that reads them, and
    each chunk's outputs out while the next chunk decodes."""
    torch = job.torch
    NL, S, stream = job.NL, job.S, job.stream
    host_in = [{k: g[k].cpu().pin_memory() for k in ("Q", "K", "V", "q", "k", "v")} for g in job.layers]
    host_out = [(torch.empty(o.shape, dtype=o.dtype).pin_memory(), torch.empty(v.shape, dtype=v.dtype).pin_memory())
                for o, v in zip(job.outs, job.vics)]
    h2d = sum(x.numel() * x.element_size() for hi in host_in for x in hi.values())
    d2h = sum(x.numel() * x.element_size() for ho in host_out for x in ho)
    cin, cout = torch.cuda.Stream(), torch.cuda.Stream()
    chunks = [(t0, min(S, t0 + chunk_steps)) for t0 in range(0, S, chunk_steps)]
    ready = [torch.cuda.Event() for _ in range(NL)]
    in_ready = [torch.cuda.Event() for _ in chunks]
    out_ready = [torch.cuda.Event() for _ in chunks]
    start_ev, done_in, done_out = torch.cuda.Event(), torch.cuda.Event(), torch.cuda.Event()
    T = job.w.prompt

    def step():
        start_ev.record(stream)
        with torch.cuda.stream(cin):
            cin.wait_event(start_ev)
            for li in range(NL):
                for k in ("Q", "K", "V"):
                    job.layers[li][k].copy_(host_in[li][k], non_blocking=True)
                ready[li].record(cin)
            for c, (t0, t1) in enumerate(chunks):
                for li in range(NL):
                    for k in ("q", "k", "v"):
                        job.layers[li][k][t0:t1].copy_(host_in[li][k][t0:t1], non_blocking=True)
                in_ready[c].record(cin)
            done_in.record(cin)
        with torch.cuda.stream(stream):
            for li in range(NL):
                stream.wait_event(ready[li])
                g = job.layers[li]
                job.prefill_call(job.hs[li], g["Q"], g["K"], g["V"], T)
            for c, (t0, t1) in enumerate(chunks):
                stream.wait_event(in_ready[c])
                job.decode(t0, t1)
                out_ready[c].record(stream)
        with torch.cuda.stream(cout):
            for c, (t0, t1) in enumerate(chunks):
                cout.wait_event(out_ready[c])
                for li in range(NL):
                    host_out[li][0][t0:t1].copy_(job.outs[li][t0:t1], non_blocking=True)
                    host_out[li][1][t0:t1].copy_(job.vics[li][t0:t1], non_blocking=True)
            done_out.record(cout)
        stream.wait_event(done_in)
        stream.wait_event(done_out)

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
    job.sync()
    n = 9                     # the host link is shared: a median over more steps
    each = []
    for _ in range(n):
        torch.cuda.synchronize()
        t0 = time.perf_counter()
        run()
        torch.cuda.synchronize()
        each.append(time.perf_counter() - t0)
    job.sync()
    secs = statistics.median(each)
    return {"value": world * job.S * NL / secs, "unit": UNIT, "h2d_bytes_per_step": h2d, "d2h_bytes_per_step": d2h,
            "ms_per_step": secs * 1000.0, "steps": n, "ms_each": [round(1000.0 * x, 3) for x in each],
            "statistic": "median (the host link is shared with the machine's other GPUs)", "launch": "graph",
            "copies": "pipelined: prompt rows per layer, decode rows and outputs in chunks of %d steps" % chunk_steps}


def run_ours(args):
    import torch
    import torch.distributed as dist

    from kv_cache_eviction_h2o_gb300 import binding as L
    from kv_cache_eviction_h2o_gb300 import build as lib_build

    world, rank, local = dist_setup()
    torch.cuda.set_device(local)
    if world > 1:
        dist.init_process_group("nccl", device_id=torch.device("cuda", local))
    lib_build.build()
    L.lib()
    stream = torch.cuda.Stream()
    main = measure(args, L, torch, args.config, args.rule, args.layers, args.decode_steps, stream, world, rank,
                   not args.no_e2e, 0 if args.no_cpu else args.oracle_seconds, Clocks(local), main_record=True)
    subs = {}
    if not args.no_sub:
        names = [s for s in (args.sub.split(",") if args.sub else SUB_CONFIGS) if s and s != args.config]
        for name in names:
            subs[name] = measure(args, L, torch, name, None, None, None, stream, world, rank, False,
                                 0 if args.no_cpu else args.oracle_seconds / 2)
    line = {
        "metric": METRIC, "value": main["value"], "unit": UNIT, "n_gpus": world, "steps": args.steps,
        "warmup": args.warmup, "ms_per_step": main["ms_per_step"], "higher_is_better": True, "scaling": "weak",
        "vs_baseline": None, "dtype": "bf16", "data": "synthetic (seeded, shaped like the configuration's layer)",
        "config": dict(main["config"], global_batch=main["config"]["batch"] * world,
                       parallelism="replicas" if world > 1 else "single"),
        "roofline": main["roofline"], "rooflines": main["rooflines"], "launch_us": main["launch_us"],
        "phases_ms_per_step": main["phases_ms_per_step"], "head_steps_per_s": main["head_steps_per_s"],
        "cpu_baseline": main["cpu_baseline"], "clocks": main["clocks"], "e2e": main.get("e2e"),
        "gpu_launches": main["gpu_launches"],
        "l2_hot": main["l2_hot"],
        "sub_records": subs,
    }
    if rank == 0:
        print(json.dumps(line))
    if world > 1:
        dist.destroy_process_group()


def main():
    args = parse()
    if args.impl == "reference":
        run_reference(args)
    else:
        run_ours(args)


if __name__ == "__main__":
    main()
