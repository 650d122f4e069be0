#!/usr/bin/env python
"""Throughput of the FAD-KV per-token KV encoding path on GB300.

A step is one decode step of every dictionary of Llama-3.2-3B (28 layers x
{K, V} = 56 dictionaries, N=4096 binary16 atoms, d=128, n=256, s=8; 8 KV
heads x 16 sequences = 128 vectors per dictionary): encode (screening, Top-n
pool, greedy + ridge), fixed-size adaptation and sparse reconstruction,
through the C ABI.  Inputs are synthetic (seeded sparse mixtures, see
dictionary_sparse_kv_gb300/synthetic.py).

    python bench.py [--gpus N] [--steps K] [--warmup W] [--impl ours|reference] [--coder gm|pl]

--coder pl times the PL coder instead (the Top-s atoms and one ridge fit in
place of the greedy selection; Tables 1-4's "PL" rows).

Prints one JSON line (rank 0).  Under torchrun (N > 1) every rank runs its
own 56 dictionaries (weak scaling, no collective on the data path); the time
is the max over ranks.
"""
from __future__ import annotations

import argparse
import hashlib
import json
import os
import statistics
import subprocess
import sys
import threading
import time
from dataclasses import replace

ROOT = os.path.dirname(os.path.abspath(__file__))
if ROOT not in sys.path:
    sys.path.insert(0, ROOT)

METRIC = "KV vectors encoded/s at N=4096,d=128,n=256,s=8; % HBM / tensor-pipe roofline"
METRIC_PL = "KV vectors encoded/s, PL coder (Top-s + one ridge fit) at N=4096,d=128,s=8; % HBM roofline"
UNIT = "vectors/s"
WORKLOAD = "decode_3b"
L2_FLUSH_BYTES = 256 << 20           # twice the 129 MB L2
FALLBACK_PEAKS = {"hbm_gbs": 6800.0, "bf16_tflops": 1900.0, "bf16_tflops_sustained": 1700.0,
                  "sm_max_mhz": 2070.0}


def parse(argv=None):
    ap = argparse.ArgumentParser()
    ap.add_argument("--gpus", type=int, default=1)
    ap.add_argument("--steps", type=int, default=20)
    ap.add_argument("--warmup", type=int, default=3)
    ap.add_argument("--impl", choices=["ours", "reference"], default="ours")
    ap.add_argument("--workload", default=WORKLOAD)
    ap.add_argument("--no-cpu-baseline", action="store_true")
    ap.add_argument("--no-extra", action="store_true",
                    help="measure only the headline workload (not " + ", ".join(EXTRA_WORKLOADS) + ")")
    ap.add_argument("--coder", choices=["gm", "pl"], default="gm")
    ap.add_argument("--dicts", type=int, default=0,
                    help="run only the first G dictionaries of the workload (profiling captures)")
    ap.add_argument("--vectors", type=int, default=0,
                    help="vectors per dictionary per step instead of the workload's (batch-size sweeps)")
    ap.add_argument("--record-traffic", metavar="CSV", default=None,
                    help="read an ncu --csv capture of dram__bytes_read.sum / dram__bytes_write.sum and record "
                         "the bytes per launch of --traffic-kernel in profiles/traffic.json, then exit")
    ap.add_argument("--traffic-kernel", default="greedy", help="kernel class of --record-traffic")
    ap.add_argument("--traffic-scale", type=float, default=1.0,
                    help="multiply the captured bytes per launch by this (a capture on fewer dictionaries)")
    ap.add_argument("--attend", type=int, default=0, metavar="T",
                    help="time decode attention over packed codes with T cached tokens instead")
    return ap.parse_args(argv)


def dist_env():
    return (int(os.environ.get("RANK", "0")), int(os.environ.get("WORLD_SIZE", "1")),
            int(os.environ.get("LOCAL_RANK", "0")))


def workload_config(w, vectors_per_step, coder="gm"):
    return {
        "coder": "greedy in the Top-n pool + ridge refit" if coder == "gm" else "PL: Top-s + one ridge fit",
        "workload": f"{w.name}: {w.G} dictionaries (layers x K,V), N={w.N}, d={w.d}, n={w.n}, s={w.s}, "
                    f"{w.V} vectors per dictionary per step (8 KV heads x {w.V // 8} sequences)",
        "vectors_per_step": vectors_per_step,
        "step": "encode + adapt + reconstruct",
        "storage": "binary16 atoms and inputs",
        "l2": "flushed between timed steps (256 MiB write outside the step's events)",
    }


L2_FETCH_BYTES = 32


def set_l2_fetch_granularity(nbytes: int):
    """Sets the current CUDA context's L2 fetch granularity hint (the
    driver's CU_LIMIT_MAX_L2_FETCH_GRANULARITY, per context, gone with the
    process).  The greedy's Gram gathers are scattered 4-byte reads: with
    32-byte fetches an L2 miss brings one sector instead of two or four.
    Returns the value the context reports afterwards (None if unknown)."""
    import ctypes
    try:
        cu = ctypes.CDLL("libcuda.so.1")
    except OSError:
        return None
    limit = 0x05                                   # CU_LIMIT_MAX_L2_FETCH_GRANULARITY
    cu.cuCtxSetLimit(limit, ctypes.c_size_t(nbytes))
    got = ctypes.c_size_t(0)
    if cu.cuCtxGetLimit(ctypes.byref(got), limit) != 0:
        return None
    return int(got.value)


def load_peaks():
    path = os.path.join(ROOT, "MEASURED_PEAKS.json")
    if os.path.exists(path):
        with open(path) as f:
            return json.load(f), "measured"
    return dict(FALLBACK_PEAKS), "fallback"


# --------------------------------------------------------------------------
# clocks during the timed region
# --------------------------------------------------------------------------

class ClockSampler:
    QUERY = ("index,clocks.sm,clocks.max.sm,power.draw,clocks_event_reasons.active,"
             "clocks_event_reasons.hw_slowdown,clocks_event_reasons.hw_thermal_slowdown,"
             "clocks_event_reasons.sw_thermal_slowdown,clocks_event_reasons.sw_power_cap")

    def __init__(self, gpu_index: int):
        self.gpu = gpu_index
        self.proc = None
        self.lines = []
        self.t = None

    def start(self):
        try:
            self.proc = subprocess.Popen(["nvidia-smi", f"--query-gpu={self.QUERY}", "--format=csv,noheader,nounits",
                                          "-lms", "200", "-i", str(self.gpu)],
                                         stdout=subprocess.PIPE, stderr=subprocess.DEVNULL, text=True)
        except OSError:
            self.proc = None
            return
        self.t = threading.Thread(target=self._read, daemon=True)
        self.t.start()
        time.sleep(0.3)

    def _read(self):
        for line in self.proc.stdout:
            self.lines.append(line.strip())

    def stop(self):
        if not self.proc:
            return {"sm_mhz": None, "sm_max_mhz": None, "reasons": ["nvidia-smi unavailable"]}
        time.sleep(0.3)
        self.proc.terminate()
        try:
            self.proc.wait(timeout=5)
        except subprocess.TimeoutExpired:
            self.proc.kill()
        if self.t:
            self.t.join(timeout=2)
        sm, mx, reasons = [], [], set()
        names = ["hw_slowdown", "hw_thermal_slowdown", "sw_thermal_slowdown", "sw_power_cap"]
        for ln in self.lines:
            parts = [p.strip() for p in ln.split(",")]
            if len(parts) < 9:
                continue
            try:
                sm.append(float(parts[1]))
                mx.append(float(parts[2]))
            except ValueError:
                continue
            for nm, val in zip(names, parts[5:9]):
                if val.lower() == "active":
                    reasons.add(nm)
        return {"sm_mhz": statistics.median(sm) if sm else None, "sm_max_mhz": max(mx) if mx else None,
                "reasons": sorted(reasons), "samples": len(sm)}


# --------------------------------------------------------------------------
# algorithmic work per kernel launch (the roofline numerators)
# --------------------------------------------------------------------------

def kernel_work(w, kernel: str, vectors: int, coder: str = "gm"):
    """(bound, algorithmic units per launch, unit) for one launch that covers
    `vectors` vectors of every dictionary (G * vectors vectors in total).
    Per-vector figures: screening streams the dictionary once per launch plus
    the inputs (HBM); the greedy gathers the pool's data and (s - 1) Gram
    rows at the pool's ids (HBM)."""
    G, N, d, n, s = w.G, w.N, w.d, w.n, w.s
    esz = 2 if w.dtype.__name__ == "float16" else 4
    nv = G * vectors
    if kernel == "screen":
        return "hbm", float(G * N * d * esz + nv * d * esz), "GB/s"
    if kernel == "topn":
        # the screening records in (per 128 atoms a header and four mask
        # words, and about 1.3 n kept scores per vector) and the pool out
        # (ids and scores: n, or s for the PL coder)
        return "hbm", (4.0 * (5 * (N // 128) + 1.3 * n) + 8.0 * (s if coder == "pl" else n)) * nv, "GB/s"
    if kernel == "greedy" and coder == "pl":
        # the fit: the s rows and x in, ids, coefficients and relres out
        return "hbm", ((s + 1) * d * esz + 8.0 * s + 4.0) * nv, "GB/s"
    if kernel == "greedy":
        # the greedy over the Gram matrix: per vector the pool's ids, scores
        # and G_jj (12 B each), the (s - 1) Gram rows at the pool's ids
        # (4 B per entry), x and the s picked rows for the residual, and the
        # codes out
        return "hbm", (12.0 * n + 4.0 * (s - 1) * n + (s + 1) * d * esz + 8.0 * s + 4.0) * nv, "GB/s"
    if kernel == "gram":
        # the update after an adaptation: the replaced-atom counts (the rows
        # of replaced atoms are data-dependent and not counted)
        return "hbm", 4.0 * G, "GB/s"
    if kernel == "adapt":
        return "hbm", 4.0 * (s + 3) * nv + 4.0 * G * N, "GB/s"
    if kernel == "reconstruct":
        return "hbm", (esz * (s + 1) * d + 4 * (s + 1) + 4 * d) * nv, "GB/s"
    raise KeyError(kernel)


def step_roofline(w, vectors_per_step: int, ms_per_step: float, peaks: dict) -> dict:
    """HBM fraction of the whole step: its algorithmic bytes -- every
    dictionary read once, the inputs read, the codes written (s ids and
    coefficients, relres, replacement id and coefficient per vector) and the
    usage counts scanned -- over the step time, against the HBM peak."""
    esz = 2 if w.dtype.__name__ == "float16" else 4
    V = vectors_per_step // w.G
    algo = (w.G * w.N * w.d * esz + vectors_per_step * w.d * esz
            + vectors_per_step * (8 * w.s + 4 + 8) + w.G * w.N * 4)
    achieved = algo / (ms_per_step / 1e3) / 1e9
    return {"bound": "hbm", "algorithmic_bytes": algo, "bytes_per_vector": round(algo / vectors_per_step, 1),
            "vectors_per_dictionary": V, "achieved": round(achieved, 1), "peak": round(peaks["hbm_gbs"], 1),
            "unit": "GB/s", "frac": round(achieved / peaks["hbm_gbs"], 4)}


def kernel_sources():
    import glob
    out = {}
    for p in glob.glob(os.path.join(ROOT, "dictionary_sparse_kv_gb300", "csrc", "*")):
        with open(p, "rb") as f:
            out[os.path.basename(p)] = hashlib.sha256(f.read()).hexdigest()[:16]
    return out


def kernel_files(coder: str = "gm"):
    """Source file of each kernel class on the binary16 path the bench runs."""
    return {"screen": "k_screen_tc.cu", "topn": "k_select.cu",
            "greedy": "k_pl.cu" if coder == "pl" else "k_gram.cu",
            "adapt": "k_adapt_reconstruct.cu", "reconstruct": "k_adapt_reconstruct.cu", "gram": "k_gram.cu"}


def traffic_for(kernel: str, w, coder: str = "gm"):
    """DRAM bytes per launch from a committed ncu summary, if it was taken on
    the current source of that kernel (profiles/traffic.json; the PL coder's
    entries sit under "<workload>+pl")."""
    path = os.path.join(ROOT, "profiles", "traffic.json")
    if not os.path.exists(path):
        return None
    with open(path) as f:
        tab = json.load(f)
    ent = tab.get(w.name + ("+pl" if coder == "pl" else ""), {}).get(kernel)
    if not ent:
        return None
    src = kernel_sources().get(kernel_files(coder).get(kernel, ""), None)
    if ent.get("source_sha256_16") != src:
        return None
    return ent.get("dram_bytes_per_launch")


# ncu's kernel names of each kernel class (demangled names contain these)
KERNEL_SYMBOLS = {"screen": "screen_tc_kernel", "topn": "select_kernel", "greedy": "greedy_gram_kernel",
                  "adapt": "adapt_kernel", "reconstruct": "reconstruct_kernel", "gram": "gram_kernel"}


def traffic_from_ncu_csv(path, symbol):
    """Mean DRAM bytes (read + write) per launch of the kernels whose name
    contains `symbol`, from `ncu --metrics dram__bytes_read.sum,
    dram__bytes_write.sum --csv` output (one row per launch and metric)."""
    import csv
    unit_scale = {"byte": 1.0, "Kbyte": 1e3, "Mbyte": 1e6, "Gbyte": 1e9, "KB": 1e3, "MB": 1e6, "GB": 1e9}
    per_launch = {}
    with open(path, newline="") as f:
        rows = [r for r in csv.reader(f)]
    head = next(i for i, r in enumerate(rows) if "Metric Name" in r and "Kernel Name" in r)
    cols = rows[head]
    ki, mi, ui, vi, ii = (cols.index(c) for c in ("Kernel Name", "Metric Name", "Metric Unit", "Metric Value", "ID"))
    for r in rows[head + 1:]:
        if len(r) <= vi or symbol not in r[ki]:
            continue
        if r[mi] not in ("dram__bytes_read.sum", "dram__bytes_write.sum"):
            continue
        v = float(r[vi].replace(",", "")) * unit_scale.get(r[ui], 1.0)
        per_launch[r[ii]] = per_launch.get(r[ii], 0.0) + v
    if not per_launch:
        raise ValueError(f"no launch of {symbol} with DRAM metrics in {path}")
    return sum(per_launch.values()) / len(per_launch), len(per_launch)


def record_traffic(args):
    """Writes the DRAM bytes per launch of one kernel class, with the sha256
    of its source file as it is now, into profiles/traffic.json."""
    from dictionary_sparse_kv_gb300 import synthetic as S
    w = S.WORKLOADS[args.workload]
    kern = args.traffic_kernel
    byts, n = traffic_from_ncu_csv(args.record_traffic, KERNEL_SYMBOLS[kern])
    path = os.path.join(ROOT, "profiles", "traffic.json")
    tab = {}
    if os.path.exists(path):
        with open(path) as f:
            tab = json.load(f)
    key = w.name + ("+pl" if args.coder == "pl" else "")
    src = kernel_files(args.coder)[kern]
    tab.setdefault(key, {})[kern] = {
        "kernel": KERNEL_SYMBOLS[kern], "dram_bytes_per_launch": int(round(byts * args.traffic_scale)),
        "launches_captured": n, "scale": args.traffic_scale, "source": src,
        "source_sha256_16": kernel_sources().get(src), "from": os.path.basename(args.record_traffic)}
    with open(path, "w") as f:
        json.dump(tab, f, indent=1, sort_keys=True)
        f.write("\n")
    print(json.dumps(tab[key][kern]))
    return 0


def dominant_kernel(prof):
    """The kernel class with the largest device time in a profile."""
    return max(prof, key=lambda k: prof[k][1]) if prof else None


def roofline(w, prof, timed, vectors_per_launch, peaks, peak_kind, sm_count, sm_mhz_max, coder="gm"):
    """Roofline object for the kernel with the largest share of device time
    (shares from `prof`, a pass with every launch bracketed; the kernel's
    launch duration from `timed`, the timed region, where only it is)."""
    kern = dominant_kernel(prof)
    if kern is None:
        return None, {}
    shares = {}
    tot = sum(v[1] for v in prof.values()) or 1.0
    for k, (n_l, ms) in prof.items():
        shares[k] = {"launches": n_l, "ms_total": round(ms, 4), "share": round(ms / tot, 4)}
    n_launch, ms = timed[kern] if timed.get(kern, (0, 0.0))[1] > 0 else prof[kern]
    bound, work, unit = kernel_work(w, kern, vectors_per_launch, coder)
    sec = ms / 1e3 / n_launch
    if unit == "GB/s":
        achieved = work / sec / 1e9
        peak = peaks["hbm_gbs"]
        pk = f"hbm_gbs ({peak_kind})"
    else:
        achieved = work / sec / 1e12
        if bound == "alu":
            # FP32 pipe: 128 FMA lanes per SM, 2 flops per FMA, max SM clock
            peak = sm_count * 128 * 2 * sm_mhz_max * 1e6 / 1e12
            pk = f"fp32 fma: {sm_count} SMs x 128 lanes x 2 x {sm_mhz_max:.0f} MHz"
        else:
            # binary16 inputs, fp32 accumulation: the dense bf16 rate (same
            # nominal rate as fp16), burst figure for a kernel timed per launch
            peak = peaks["bf16_tflops"]
            pk = f"bf16_tflops ({peak_kind}, burst; fp16 at the same nominal rate)"
    obj = {"kernel": kern, "source": kernel_files(coder).get(kern), "bound": bound, "achieved": round(achieved, 3),
           "peak": round(peak, 3), "unit": unit, "frac": round(achieved / peak, 4),
           "traffic": traffic_for(kern, w, coder), "peak_source": pk,
           "launch_ms": round(ms / n_launch, 5)}
    return obj, shares


# --------------------------------------------------------------------------
# oracle timing (CPU baseline and the reference arm)
# --------------------------------------------------------------------------

def oracle_steps(w, data, steps, threads, coder="gm"):
    """Run the oracle over `steps` decode steps of every dictionary of `data`
    (encode on `threads` host threads, then the sequential adapt and
    reconstruct).  Returns
    (vectors, seconds)."""
    import numpy as np
    from oracle import oracle as O
    p = O.Params(w.N, w.d, w.n, w.s, 1e-4, 0.20, O.F16 if w.dtype.__name__ == "float16" else O.F32)
    atoms = data.atoms.copy()
    usage = data.usage.copy()
    xs = [data.inputs(t) for t in range(steps)]
    t0 = time.perf_counter()
    nvec = 0
    for t in range(steps):
        x = xs[t]
        for g in range(len(data.dicts)):
            r = O.encode_threaded(p, atoms[g], x[g], threads, coder)
            a = O.adapt(p, atoms[g], usage[g], x[g], r.idx, r.coef, r.relres, data.deltas()[g])
            O.reconstruct(p, atoms[g], r.idx, r.coef, a.repl_id, a.repl_coef)
            nvec += x.shape[1]
    return nvec, time.perf_counter() - t0


ARM_PARTS = {"0xd4f": "Arm Neoverse-V2", "0xd40": "Arm Neoverse-V1", "0xd0c": "Arm Neoverse-N1",
             "0xd49": "Arm Neoverse-N2", "0xd8e": "Arm Neoverse-N3", "0xd84": "Arm Neoverse-V3"}


def cpu_model():
    try:
        with open("/proc/cpuinfo") as f:
            for ln in f:
                key = ln.split(":", 1)[0].strip().lower()
                if key == "model name":
                    return ln.split(":", 1)[1].strip()
                if key == "cpu part":
                    part = ln.split(":", 1)[1].strip().lower()
                    return ARM_PARTS.get(part, f"Arm part {part}")
    except OSError:
        pass
    return "unknown"


def run_reference(args):
    rank, world, _ = dist_env()
    if rank != 0:
        return 0
    from dictionary_sparse_kv_gb300 import synthetic as S
    w = S.WORKLOADS[args.workload]
    data = S.WorkloadData(w)
    threads = os.cpu_count() or 1
    # W warm-up steps, then K timed steps; each step is one full decode step
    oracle_steps(w, data, max(0, args.warmup), threads, args.coder)
    nvec, sec = oracle_steps(w, data, args.steps, threads, args.coder)
    value = nvec / sec
    line = {
        "impl": "reference", "metric": METRIC_PL if args.coder == "pl" else METRIC, "value": round(value, 3), "unit": UNIT, "n_gpus": args.gpus,
        "steps": args.steps, "warmup": args.warmup, "ms_per_step": round(sec * 1e3 / args.steps, 3),
        "higher_is_better": True, "scaling": "weak", "vs_baseline": None, "dtype": "f64", "data": "synthetic",
        "config": workload_config(w, w.G * w.V, args.coder),
        "cpu_baseline": {"value": round(value, 3), "unit": UNIT, "cores": threads, "kind": "oracle",
                         "sample": f"{args.steps} full decode steps ({w.G} x {w.V} vectors each), "
                                   f"plain C double-precision oracle, encode split over {threads} host "
                                   f"threads, adapt sequential; CPU: {cpu_model()}"},
        "e2e": {"value": round(value, 3), "unit": UNIT, "h2d_bytes_per_step": 0, "d2h_bytes_per_step": 0},
    }
    print(json.dumps(line), flush=True)
    return 0


# --------------------------------------------------------------------------
# multi-rank plumbing (weak scaling: every rank owns its own dictionaries)
# --------------------------------------------------------------------------

def rank_workload(w0, rank: int):
    """The workload a rank runs: the same shapes, its own dictionaries and
    inputs (seed offset by rank)."""
    return replace(w0, seed=w0.seed + 1000 * rank)


def max_over_ranks(x: float, device=None) -> float:
    """The largest x over all ranks (the step time of the slowest rank)."""
    import torch
    import torch.distributed as dist
    if not (dist.is_available() and dist.is_initialized()) or dist.get_world_size() == 1:
        return float(x)
    t = torch.tensor([float(x)], dtype=torch.float64, device=device)
    dist.all_reduce(t, op=dist.ReduceOp.MAX)
    return float(t.item())


def job_throughput(world: int, steps: int, vectors_per_step: int, ms_max: float) -> float:
    """Whole-job vectors/s: every rank's vectors over the slowest rank's time."""
    return world * steps * vectors_per_step / (ms_max / 1e3)


# --------------------------------------------------------------------------
# our arm
# --------------------------------------------------------------------------

# Workloads measured beside the headline one, in the same run (one GPU).
EXTRA_WORKLOADS = ("prefill_3b_16k", "decode_8b", "adapt_stress")


def screening_fractions(w, prof, steps, peaks):
    """The screening kernel's own fractions over a profiled pass of `steps`
    steps: HBM (each launch streams every dictionary once, plus the inputs)
    and tensor pipe (2 N d flops per vector against the dense bf16 peak,
    binary16 having the same nominal rate)."""
    if "screen" not in prof:
        return None
    launches, ms = prof["screen"]
    esz = 2 if w.dtype.__name__ == "float16" else 4
    vecs = steps * w.G * w.V
    sec = ms / 1e3
    byts = launches * w.G * w.N * w.d * esz + vecs * w.d * esz
    flops = 2.0 * w.N * w.d * vecs
    return {"launches": launches, "ms_per_launch": round(ms / launches, 5),
            "hbm": {"achieved_gbs": round(byts / sec / 1e9, 1), "frac": round(byts / sec / 1e9 / peaks["hbm_gbs"], 4)},
            "tensor": {"achieved_tflops": round(flops / sec / 1e12, 2),
                       "frac": round(flops / sec / 1e12 / peaks["bf16_tflops"], 4)}}


def extra_workload(name, dev, peaks, peak_kind, sm_count, sm_max, coder="gm", K=5, W=3):
    """The headline's step on another workload, device-timed the same way
    (CUDA events around each step, L2 flushed between steps, W warm-up
    steps): ms per step, vectors/s, the dominant kernel's roofline, the
    screening kernel's own HBM and tensor fractions, and the atoms replaced
    in the timed steps.  The adaptation stress takes its inputs from the
    first drift of its sources on (steps 128, 129, ...: the stress case,
    replacements in every step); the 16K prefill alternates two input
    batches of 262 144 vectors."""
    import torch
    from dictionary_sparse_kv_gb300 import fadkv as F
    from dictionary_sparse_kv_gb300 import synthetic as S
    w = S.WORKLOADS[name]
    data = S.WorkloadData(w)
    t0 = w.drift_period if w.drift_period > 0 else 0
    nin = 2 if w.G * w.V > 100_000 else W + 2 * K
    xs = [torch.from_numpy(data.inputs(t0 + t)).to(dev) for t in range(nin)]
    D = F.Dictionary(torch.from_numpy(data.atoms).to(dev), torch.from_numpy(data.usage).to(dev),
                     data.deltas(), w.n, w.s, w.V)
    codes = D.new_codes(w.V)
    xhat = torch.empty((w.G, w.V, w.d), dtype=torch.float32, device=dev)
    flush = torch.empty(L2_FLUSH_BYTES // 4, dtype=torch.float32, device=dev)
    stream = torch.cuda.current_stream(dev)
    step = 0
    for _ in range(W):
        D.step(xs[step % nin], codes, xhat, coder=coder)
        step += 1
    torch.cuda.synchronize(dev)
    F.profile_read(D.h, reset=True)
    F.profile_enable(D.h, True)
    for t in range(K):
        flush.fill_(float(t))
        D.step(xs[step % nin], codes, xhat, coder=coder)
        step += 1
    torch.cuda.synchronize(dev)
    F.profile_enable(D.h, False)
    prof_all = F.profile_read(D.h, reset=True)
    dom = dominant_kernel(prof_all)
    F.profile_select(D.h, [dom] if dom else None)
    F.profile_enable(D.h, True)
    rep0 = sum(s["replaced"] for s in D.stats())
    ev = [(torch.cuda.Event(enable_timing=True), torch.cuda.Event(enable_timing=True)) for _ in range(K)]
    torch.cuda.synchronize(dev)
    for t in range(K):
        flush.fill_(float(t))
        ev[t][0].record(stream)
        D.step(xs[step % nin], codes, xhat, coder=coder)
        ev[t][1].record(stream)
        step += 1
    torch.cuda.synchronize(dev)
    F.profile_enable(D.h, False)
    F.profile_select(D.h, None)
    prof = F.profile_read(D.h, reset=True)
    st = D.stats()
    ms = sum(a.elapsed_time(b) for a, b in ev) / K
    roof, shares = roofline(w, prof_all, prof, w.V, peaks, peak_kind, sm_count, sm_max, coder)
    out = {"workload": workload_config(w, w.G * w.V, coder)["workload"], "steps": K, "warmup": W,
           "ms_per_step": round(ms, 4), "vectors_per_s": round(w.G * w.V / (ms / 1e3), 1),
           "roofline": roof, "kernels": shares, "screening": screening_fractions(w, prof_all, K, peaks),
           "replaced_in_timed_steps": sum(s["replaced"] for s in st) - rep0,
           "status_words": sorted({int(s["status"]) for s in st})}
    if w.drift_period > 0:
        out["inputs"] = f"steps {t0}.. (after the first drift of the sources)"
    if nin == 2:
        out["inputs"] = "two input batches, alternated"
    D.close()
    del D, xs, codes, xhat, flush
    torch.cuda.empty_cache()
    return out


def run_ours(args):
    import numpy as np
    import torch
    from dictionary_sparse_kv_gb300 import build as B
    from dictionary_sparse_kv_gb300 import fadkv as F
    from dictionary_sparse_kv_gb300 import synthetic as S

    rank, world, local = dist_env()
    if world > 1:
        import torch.distributed as dist
        torch.cuda.set_device(local)
        dist.init_process_group("nccl")
    dev = torch.device("cuda", local if world > 1 else 0)
    torch.cuda.set_device(dev)
    torch.zeros(1, device=dev)                     # the context exists from here
    l2_fetch = set_l2_fetch_granularity(L2_FETCH_BYTES)
    if rank == 0:
        B.build()
    if world > 1:
        dist.barrier()
    F.lib()

    w = rank_workload(S.WORKLOADS[args.workload], rank)
    if args.dicts > 0:
        w = replace(w, G=min(args.dicts, w.G))
    if args.vectors > 0:
        w = replace(w, V=args.vectors)
    data = S.WorkloadData(w)
    K, W = args.steps, max(3, args.warmup)
    G, V, d = w.G, w.V, w.d
    xs_host = [torch.from_numpy(data.inputs(t)).pin_memory() for t in range(W + K)]
    xs_dev = [x.to(dev) for x in xs_host]
    D = F.Dictionary(torch.from_numpy(data.atoms).to(dev), torch.from_numpy(data.usage).to(dev),
                     data.deltas(), w.n, w.s, V)
    codes = D.new_codes(V)
    xhat = torch.empty((G, V, d), dtype=torch.float32, device=dev)
    flush = torch.empty(L2_FLUSH_BYTES // 4, dtype=torch.float32, device=dev)
    stream = torch.cuda.current_stream(dev)

    for t in range(W):
        D.step(xs_dev[t], codes, xhat, coder=args.coder)
    torch.cuda.synchronize(dev)
    F.profile_read(D.h, reset=True)

    # ---- per-kernel shares: an untimed pass with every launch bracketed ----
    F.profile_enable(D.h, True)
    for t in range(min(K, 10)):
        flush.fill_(float(t))
        D.step(xs_dev[W + t], codes, xhat, coder=args.coder)
    torch.cuda.synchronize(dev)
    F.profile_enable(D.h, False)
    prof_all = F.profile_read(D.h, reset=True)

    # ---- device-resident timed region (events bracket only the dominant
    #      kernel, whose launch duration the roofline needs) ----
    dom = dominant_kernel(prof_all)
    F.profile_select(D.h, [dom] if dom else None)
    F.profile_enable(D.h, True)
    clocks = ClockSampler(torch.cuda.current_device())
    if rank == 0:
        clocks.start()
    ev = [(torch.cuda.Event(enable_timing=True), torch.cuda.Event(enable_timing=True)) for _ in range(K)]
    if world > 1:
        dist.barrier()
    torch.cuda.synchronize(dev)
    wall0 = time.perf_counter()
    for t in range(K):
        flush.fill_(float(t))
        ev[t][0].record(stream)
        D.step(xs_dev[W + t], codes, xhat, coder=args.coder)
        ev[t][1].record(stream)
    torch.cuda.synchronize(dev)
    wall = time.perf_counter() - wall0
    clk = clocks.stop() if rank == 0 else None
    F.profile_enable(D.h, False)
    F.profile_select(D.h, None)
    prof = F.profile_read(D.h, reset=True)
    dev_ms = max_over_ranks(sum(a.elapsed_time(b) for a, b in ev), dev)
    launches = sum(n for n, _ in prof.values())

    # ---- end to end: pinned host inputs in, codes out, every step ----
    xin = torch.empty_like(xs_dev[0])
    # the codes live in one buffer: one copy brings every array back
    outs = [torch.empty(codes.buf.shape, dtype=codes.buf.dtype).pin_memory()]
    h2d = xs_host[0].numel() * xs_host[0].element_size()
    d2h = sum(o.numel() * o.element_size() for o in outs)
    ev2 = [(torch.cuda.Event(enable_timing=True), torch.cuda.Event(enable_timing=True)) for _ in range(K)]

    def e2e_step(t):
        xin.copy_(xs_host[t], non_blocking=True)
        D.step(xin, codes, xhat, coder=args.coder)
        for o, c in zip(outs, (codes.buf,)):
            o.copy_(c, non_blocking=True)

    # untimed warm-up of the same loop (first touch of the pinned buffers)
    for t in range(W):
        e2e_step(t)
    if world > 1:
        dist.barrier()
    torch.cuda.synchronize(dev)
    for t in range(K):
        flush.fill_(float(t))
        ev2[t][0].record(stream)
        e2e_step(W + t)
        ev2[t][1].record(stream)
    torch.cuda.synchronize(dev)
    e2e_seq_ms = max_over_ranks(sum(a.elapsed_time(b) for a, b in ev2), dev)

    # ---- end to end with the copies overlapped, as a decode loop runs: the
    #      input of step t+1 goes in on a copy stream while step t runs and
    #      the codes of step t come back while step t+1 runs (two input and
    #      two code buffers).  Timed from the first input copy to the last
    #      codes copy on the copy stream, less the L2 flushes between steps
    #      (each bracketed by events on the compute stream) ----
    cs = torch.cuda.Stream(device=dev)
    xin2 = [torch.empty_like(xs_dev[0]) for _ in range(2)]
    codes2 = [D.new_codes(V) for _ in range(2)]
    outs2 = [torch.empty(codes.buf.shape, dtype=codes.buf.dtype).pin_memory() for _ in range(2)]

    def pipelined(t0, n):
        if n <= 0:
            return None
        in_ev = [torch.cuda.Event() for _ in range(n)]
        done = [torch.cuda.Event() for _ in range(n)]
        fl = [(torch.cuda.Event(enable_timing=True), torch.cuda.Event(enable_timing=True)) for _ in range(n)]
        start, end = torch.cuda.Event(enable_timing=True), torch.cuda.Event(enable_timing=True)
        cs.wait_stream(stream)
        start.record(cs)
        with torch.cuda.stream(cs):
            xin2[0].copy_(xs_host[t0], non_blocking=True)
        in_ev[0].record(cs)
        for t in range(n):
            b = t % 2
            if t + 1 < n:
                if t >= 1:
                    cs.wait_event(done[t - 1])          # step t-1 is done with that input buffer
                with torch.cuda.stream(cs):
                    xin2[1 - b].copy_(xs_host[t0 + t + 1], non_blocking=True)
                in_ev[t + 1].record(cs)
            fl[t][0].record(stream)
            flush.fill_(float(t))
            fl[t][1].record(stream)
            stream.wait_event(in_ev[t])
            D.step(xin2[b], codes2[b], xhat, coder=args.coder)
            done[t].record(stream)
            cs.wait_event(done[t])
            with torch.cuda.stream(cs):
                outs2[b].copy_(codes2[b].buf, non_blocking=True)
        end.record(cs)
        return start, end, fl

    pipelined(0, W)                                   # untimed
    if world > 1:
        dist.barrier()
    torch.cuda.synchronize(dev)
    # the same launches bracketed as in the device-resident timed region (the
    # dominant kernel's), so the two figures time the same step
    F.profile_select(D.h, [dom] if dom else None)
    F.profile_enable(D.h, True)
    start, end, fl = pipelined(W, K)
    torch.cuda.synchronize(dev)
    F.profile_enable(D.h, False)
    F.profile_select(D.h, None)
    F.profile_read(D.h, reset=True)
    e2e_ms = max_over_ranks(start.elapsed_time(end) - sum(a.elapsed_time(b) for a, b in fl), dev)
    stats = D.stats()

    if rank != 0:
        dist.barrier() if world > 1 else None
        return 0

    vectors_per_step = G * V
    value = job_throughput(world, K, vectors_per_step, dev_ms)
    e2e = job_throughput(world, K, vectors_per_step, e2e_ms)
    e2e_seq = job_throughput(world, K, vectors_per_step, e2e_seq_ms)
    peaks, peak_kind = load_peaks()
    props = torch.cuda.get_device_properties(dev)
    sm_max = float(peaks.get("sm_max_mhz") or clk.get("sm_max_mhz") or 2070.0)
    roof, shares = roofline(w, prof_all, prof, V, peaks, peak_kind, props.multi_processor_count, sm_max,
                            args.coder)

    cpu = None
    if not args.no_cpu_baseline:
        threads = os.cpu_count() or 1
        sub = S.WorkloadData(w)
        nvec, sec = oracle_steps(w, sub, 2, threads, args.coder)
        cpu = {"value": round(nvec / sec, 3), "unit": UNIT, "cores": threads, "kind": "oracle",
               "sample": f"first 2 decode steps of all {w.G} dictionaries ({nvec} vectors), oracle encode "
                         f"over {threads} host threads + sequential adapt; CPU: {cpu_model()}"}
    line = {
        "metric": METRIC_PL if args.coder == "pl" else METRIC, "value": round(value, 1), "unit": UNIT, "n_gpus": world, "steps": K, "warmup": W,
        "ms_per_step": round(dev_ms / K, 4), "higher_is_better": True, "scaling": "weak", "vs_baseline": None,
        "dtype": "f32", "data": "synthetic",
        "config": dict(workload_config(w, vectors_per_step, args.coder), l2_fetch_granularity_bytes=l2_fetch),
        "e2e": {"value": round(e2e, 1), "unit": UNIT, "h2d_bytes_per_step": h2d, "d2h_bytes_per_step": d2h,
                "copies": "overlapped with the neighbouring steps on a copy stream",
                "sequential": {"value": round(e2e_seq, 1), "unit": UNIT,
                               "copies": "in line: input copy, step, codes copy, one step at a time"}},
        "gpu_launches": launches, "roofline": roof, "kernels": shares, "clocks": clk, "cpu_baseline": cpu,
        "step_roofline": step_roofline(w, vectors_per_step, dev_ms / K, peaks),
        "wall_s_timed": round(wall, 4),
        "adapt": {"replaced": sum(s["replaced"] for s in stats), "overflow": sum(s["overflow"] for s in stats)},
        "topn_slow_path_vectors": sum(s["topn_slow_path"] for s in stats),
    }
    scr = screening_fractions(w, prof_all, min(K, 10), peaks)
    if scr:
        line["screening"] = scr
    if world == 1 and args.workload == WORKLOAD and not args.no_extra and args.dicts == 0 and args.vectors == 0:
        D.close()
        del D, codes, xhat, flush, xs_dev, xin
        torch.cuda.empty_cache()
        line["workloads"] = {nm: extra_workload(nm, dev, peaks, peak_kind, props.multi_processor_count, sm_max,
                                                args.coder) for nm in EXTRA_WORKLOADS}
    print(json.dumps(line), flush=True)
    if world > 1:
        dist.barrier()
    return 0


def run_attend(args):
    """Decode attention of Llama-3.2-3B (28 layers, 16 sequences, 24 query /
    8 KV heads, d = 128) over packed codes (N = 4096, s = 8, s + 1 words per
    token) with T cached tokens per sequence, one fadkv_attend launch for all
    layers (three kernels: U = Q D_K^T, the token pass, O = W D_V).  Prints
    one JSON line; value = query-token pairs per second."""
    import numpy as np
    import torch
    from dictionary_sparse_kv_gb300 import build as B
    from dictionary_sparse_kv_gb300 import fadkv as F
    from dictionary_sparse_kv_gb300 import synthetic as S

    B.build()
    dev = torch.device("cuda", 0)
    L, Bs, Hq, Hkv, d, N, s, T = 28, 16, 24, 8, 128, 4096, 8, args.attend
    K, W = args.steps, max(3, args.warmup)
    g = np.random.default_rng(60)
    atoms = torch.from_numpy(np.stack([S.make_dictionary(N, d, np.float16, 61, i) for i in range(2 * L)])).to(dev)
    words = (L, 2, Bs, Hkv, T, s + 1)
    coefs = torch.randn(words, device=dev, dtype=torch.float32).mul_(0.3)
    ids = torch.randint(0, N, words, device=dev, dtype=torch.int32)
    cache = (coefs.view(torch.int32) & -8192) | ids               # random packed words
    del coefs, ids
    lengths = torch.full((Bs,), T, dtype=torch.int32, device=dev)
    q = torch.randn((L, Bs, Hq, d), device=dev, dtype=torch.float32)
    out = torch.empty_like(q)
    p = F.AttnParams(L, Bs, Hq, Hkv, d, N, s, T, F.F16, 1.0 / np.sqrt(d), 2 * N * d, 2 * Bs * Hkv * T * (s + 1))
    ck, cv = cache[:, 0], cache[:, 1]
    flush = torch.empty(L2_FLUSH_BYTES // 4, dtype=torch.float32, device=dev)
    ws = torch.empty(max(1, F.attend_workspace_bytes(p)), dtype=torch.uint8, device=dev)
    for _ in range(W):
        F.attend(p, atoms[0], atoms[1], ck, cv, lengths, q, out, ws)
    torch.cuda.synchronize()
    clocks = ClockSampler(0)
    clocks.start()
    ev = [(torch.cuda.Event(enable_timing=True), torch.cuda.Event(enable_timing=True)) for _ in range(K)]
    stream = torch.cuda.current_stream(dev)
    for t in range(K):
        flush.fill_(float(t))
        ev[t][0].record(stream)
        F.attend(p, atoms[0], atoms[1], ck, cv, lengths, q, out, ws)
        ev[t][1].record(stream)
    torch.cuda.synchronize()
    clk = clocks.stop()
    ms = sum(a.elapsed_time(b) for a, b in ev) / K
    pairs = L * Bs * Hq * T
    code_bytes = L * 2 * Bs * Hkv * T * (s + 1) * 4
    dict_bytes = L * 2 * N * d * 2
    algo = code_bytes + dict_bytes + 2 * q.numel() * 4
    peaks, peak_kind = load_peaks()
    achieved = algo / (ms / 1e3) / 1e9
    dense = L * 2 * Bs * Hkv * T * d * 2
    line = {
        "metric": "decode attention over packed codes: query-token pairs/s (Llama-3.2-3B shape)",
        "value": round(pairs / (ms / 1e3), 1), "unit": "pairs/s", "n_gpus": 1, "steps": K, "warmup": W,
        "ms_per_step": round(ms, 4), "higher_is_better": True, "dtype": "f32",
        "data": "synthetic (random packed words, random queries)",
        "config": {"workload": f"{L} layers x {Bs} sequences x {Hq} query / {Hkv} KV heads, d={d}, N={N}, "
                               f"s={s}, {T} cached tokens per sequence", "launches_per_step": 3,
                   "l2": "flushed between timed steps"},
        "roofline": {"kernel": "attend_kernel", "bound": "hbm", "achieved": round(achieved, 1),
                     "peak": round(peaks["hbm_gbs"], 1), "unit": "GB/s",
                     "frac": round(achieved / peaks["hbm_gbs"], 4), "traffic": None,
                     "algorithmic_bytes": algo, "peak_source": f"hbm_gbs ({peak_kind})"},
        "kv_bytes": {"codes": code_bytes, "dense_bf16": dense, "ratio": round(dense / code_bytes, 3)},
        "clocks": clk,
    }
    print(json.dumps(line), flush=True)
    return 0


def main(argv=None):
    args = parse(argv)
    if args.record_traffic:
        return record_traffic(args)
    if args.impl == "reference":
        return run_reference(args)
    if args.attend > 0:
        return run_attend(args)
    return run_ours(args)


if __name__ == "__main__":
    sys.exit(main())
