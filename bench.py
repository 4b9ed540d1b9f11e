#!/usr/bin/env python3
"""Benchmark of the row-parallel linear epilogue hot path on GB300.

One step = one pass of the whole hot path over one batch of synthetic input:

  gemm_rs            R=8, M=N=8192, K=4096: 8 partial BF16 GEMMs, ring-order
                     fp32 sum, reduce-scatter into 8 owner segments of 1024 rows
  gemm_ar            R=8, M=4096, N=7168, K=2048: 8 partial GEMMs rounded to
                     bf16, all-reduced into 8 rank views
  allreduce_rmsnorm  R=8 bf16 partials [4096, 7168] (1% -0.0), bf16 residual,
                     fp32 gamma: Lamport all-reduce + residual + RMSNorm

Every input is larger than the 129 MB L2, so no flush is needed between
steps.  ``value`` is the step's roofline fraction: the sum over the three
kernels of max(FLOPs / bf16 peak, algorithmic bytes / HBM bandwidth),
divided by the measured step time (per GPU; summed over GPUs for N > 1,
where every rank runs its own replica).  The bf16 peak is the burst figure
when the clock samples of the timed region show the SM clock at its maximum
with no power capping, the sustained figure otherwise.

After the step, ``configs`` times every workload at every size one by one
(CUDA graphs of calls), with the kernel each call launched.

    python bench.py [--gpus N] [--steps K] [--warmup W] [--impl reference]

``--impl reference`` times the CPU oracle (the only reference implementation
that exists for this method) on one bounded sample of the workload per step.
"""
from __future__ import annotations

import argparse
import json
import os
import statistics
import subprocess
import tempfile
import sys
import time

ROOT = os.path.dirname(os.path.abspath(__file__))
if ROOT not in sys.path:
    sys.path.insert(0, ROOT)

METRIC = "fused GEMM+RS TFLOP/s and AR+RMSNorm GB/s on 1 GB300, % of roofline"
UNIT = "% of one GB300's roofline"
WORKLOAD = {
    "gemm_rs": dict(R=8, M=8192, N=8192, K=4096, seed_cfg=4),
    "gemm_ar": dict(R=8, M=4096, N=7168, K=2048, seed_cfg=2),
    "allreduce_rmsnorm": dict(R=8, M=4096, N=7168, seed_cfg=3),
}
EPS = 1e-6
L2_BYTES = 129e6
# Fallback denominators (one earlier GB300 measurement), used only when the
# measured peaks file is absent.
FALLBACK_PEAKS = {"hbm_gbs": 6800.0, "bf16_tflops": 1900.0, "bf16_tflops_sustained": 1700.0}
# DRAM traffic per launch (dram__bytes_read.sum + dram__bytes_write.sum) of each
# part's kernel at this workload, from one ncu capture, keyed to the SHA-256
# (first 16 hex digits) of the kernel's source file at capture time: when the
# source has changed since, the figure no longer describes the kernel and the
# line reports null.
KERNEL_SOURCES = {"gemm_rs": "gemm_reduce.cu", "gemm_ar": "gemm_reduce.cu", "allreduce_rmsnorm": "ar_rmsnorm.cu"}
NCU_TRAFFIC = {
    "gemm_rs": (6671.4e6, "2c6dcb19e836f1c9"),
    "gemm_ar": (2707.8e6, "2c6dcb19e836f1c9"),
    "allreduce_rmsnorm": (626.4e6, "a4af1f7bd1f46c00"),
}


def source_sha16(name: str) -> str:
    import hashlib
    path = os.path.join(ROOT, "all_reduce_epilogue_gb300", "csrc", name)
    return hashlib.sha256(open(path, "rb").read()).hexdigest()[:16]


def ncu_traffic(part: str):
    val, sha = NCU_TRAFFIC[part]
    if val is None or sha != source_sha16(KERNEL_SOURCES[part]):
        return None
    return val


# --------------------------------------------------------------------------- work model

def work_of(op: str, R: int, M: int, N: int, K: int = 0, residual: bool = True):
    """(FLOPs, algorithmic bytes) of one call.  GEMMs: 2RMNK; bytes = the R
    operand pairs read once plus the output written once (GEMM+AR: R views).
    AR+RMSNorm: R partial rows + the residual row read, the output row
    written, gamma read once."""
    if op == "allreduce_rmsnorm":
        return 0.0, float(2 * M * N * (R + (2 if residual else 1)) + 4 * N)
    flops = 2.0 * R * M * N * K
    if op == "gemm_rs":
        return flops, float(2 * (R * M * K + R * K * N + M * N))
    if op == "gemm_ar":
        return flops, float(2 * (R * M * K + R * K * N + R * M * N))
    raise ValueError(op)


def work(part: str):
    w = WORKLOAD[part]
    return work_of(part, w["R"], w["M"], w["N"], w.get("K", 0))


def load_peaks():
    path = os.path.join(ROOT, "MEASURED_PEAKS.json")
    peaks = dict(FALLBACK_PEAKS)
    source = "fallback"
    if os.path.exists(path):
        try:
            d = json.load(open(path))
            flat = {}

            def walk(x, pre=""):
                if isinstance(x, dict):
                    for k, v in x.items():
                        walk(v, f"{pre}{k}.")
                else:
                    flat[pre[:-1]] = x
            walk(d)
            for key in ("hbm_gbs", "bf16_tflops", "bf16_tflops_sustained"):
                cands = [v for k, v in flat.items() if k.split(".")[-1] == key and isinstance(v, (int, float))]
                if cands:
                    peaks[key] = float(cands[0])
                    source = "measured"
        except Exception:
            pass
    return peaks, source


def bf16_peak(peaks, regime: str) -> float:
    return peaks["bf16_tflops"] if regime == "burst" else peaks["bf16_tflops_sustained"]


def roofline_seconds_of(flops: float, byts: float, peaks, regime: str) -> float:
    return max(flops / (bf16_peak(peaks, regime) * 1e12), byts / (peaks["hbm_gbs"] * 1e9))


def roofline_seconds(part: str, peaks, regime: str = "burst") -> float:
    return roofline_seconds_of(*work(part), peaks, regime)


def peak_regime(clocks) -> tuple:
    """Which bf16 peak the timed region ran under: 'burst' (the GEMM peak timed
    alone) when its clock samples show the SM clock at (or within 3% of) its
    maximum and no power capping, 'sustained' (the seconds-long figure under
    the power cap) when the power cap was active or the clock sat lower.  With
    no sample inside the region the burst peak is taken: the higher
    denominator, so the fraction is not overstated."""
    sm, smax, reasons = clocks.get("sm_mhz"), clocks.get("sm_max_mhz"), clocks.get("reasons") or []
    if clocks.get("window") != "timed region" or not sm or not smax:
        return "burst", "no clock sample inside the timed region: burst peak (the larger denominator)"
    if "sw_power_cap" in reasons or sm < 0.97 * smax:
        return "sustained", f"median SM clock {sm:.0f} of {smax:.0f} MHz, reasons {reasons}: sustained peak"
    return "burst", f"median SM clock {sm:.0f} of {smax:.0f} MHz, no power capping: burst peak"


# --------------------------------------------------------------------------- clocks

CLOCK_QUERY = ("timestamp,index,clocks.sm,clocks.max.sm,power.draw,clocks_event_reasons.active,"
               "clocks_event_reasons.hw_slowdown,clocks_event_reasons.hw_thermal_slowdown,"
               "clocks_event_reasons.sw_thermal_slowdown,clocks_event_reasons.sw_power_cap")
CLOCK_PERIOD_MS = int(os.environ.get("ARE_CLOCK_PERIOD_MS", "20"))


class ClockSampler:
    """nvidia-smi clock / throttle-reason samples every CLOCK_PERIOD_MS, read
    back per host wall-clock window (the timed region, the per-workload
    timings)."""

    def __init__(self, device_index: int):
        self.dev = device_index
        self.proc = None
        self.path = None
        self.rows = None

    def start(self):
        try:
            # the raw samples go to ARE_CLOCKS_DIR (default: the system temporary directory)
            out_dir = os.environ.get("ARE_CLOCKS_DIR") or tempfile.gettempdir()
            os.makedirs(out_dir, exist_ok=True)
            self.path = os.path.join(out_dir, f"clocks_bench_{os.getpid()}.csv")
            self.fh = open(self.path, "w")
            self.proc = subprocess.Popen(["nvidia-smi", f"--id={self.dev}", f"--query-gpu={CLOCK_QUERY}",
                                          "--format=csv,noheader,nounits", "-lms", str(CLOCK_PERIOD_MS)],
                                         stdout=self.fh, stderr=subprocess.DEVNULL)
        except Exception:
            self.proc = None

    def stop(self):
        if self.proc is None:
            return
        time.sleep(0.1)
        self.proc.terminate()
        try:
            self.proc.wait(timeout=5)
        except Exception:
            self.proc.kill()
        self.fh.close()
        import datetime
        names = ["hw_slowdown", "hw_thermal_slowdown", "sw_thermal_slowdown", "sw_power_cap"]
        self.rows = []
        for line in open(self.path):
            f = [x.strip() for x in line.split(",")]
            if len(f) < 10:
                continue
            try:
                ts = datetime.datetime.strptime(f[0], "%Y/%m/%d %H:%M:%S.%f").timestamp()
                self.rows.append((ts, float(f[2]), float(f[3]), float(f[4]),
                                  {n for n, v in zip(names, f[6:10]) if v.lower() == "active"}))
            except ValueError:
                continue

    def summary(self, window) -> dict:
        """Median SM clock, maximum clock, power and the throttle reasons of the
        samples inside `window` (host wall-clock seconds)."""
        if self.proc is None or self.rows is None:
            return {"sm_mhz": None, "sm_max_mhz": None, "reasons": ["nvidia-smi unavailable"], "window": "none"}
        inside = [r for r in self.rows if window[0] <= r[0] <= window[1]]
        use, where = (inside, "timed region") if inside else (self.rows, "whole sampling run (no sample fell inside)")
        if not use:
            return {"sm_mhz": None, "sm_max_mhz": None, "reasons": ["no samples"], "window": "none"}
        reasons = sorted(set().union(*[r[4] for r in use]))
        return {"sm_mhz": statistics.median(r[1] for r in use), "sm_max_mhz": max(r[2] for r in use),
                "reasons": reasons, "samples": len(use), "power_w_median": statistics.median(r[3] for r in use),
                "period_ms": CLOCK_PERIOD_MS, "window": where}


# --------------------------------------------------------------------------- distributed plumbing

def dist_env():
    world = int(os.environ.get("WORLD_SIZE", "1"))
    rank = int(os.environ.get("RANK", "0"))
    local = int(os.environ.get("LOCAL_RANK", "0"))
    return world, rank, local


def init_dist(world, backend):
    if world > 1:
        import torch.distributed as dist
        os.environ.setdefault("MASTER_ADDR", "127.0.0.1")
        dist.init_process_group(backend)
        return dist
    return None


def max_over_ranks(dist, value: float, device=None) -> float:
    if dist is None:
        return value
    import torch
    t = torch.tensor([value], dtype=torch.float64, device=device)
    dist.all_reduce(t, op=dist.ReduceOp.MAX)
    return float(t.item())


# --------------------------------------------------------------------------- inputs

def host_inputs():
    """Seeded synthetic host inputs (numpy bf16 bit patterns) for one step."""
    import synth
    w = WORKLOAD
    out = {}
    g = w["gemm_rs"]
    out["gemm_rs"] = synth.gemm_inputs(g["R"], g["M"], g["N"], g["K"], synth.config_seed(g["seed_cfg"]))
    g = w["gemm_ar"]
    out["gemm_ar"] = synth.gemm_inputs(g["R"], g["M"], g["N"], g["K"], synth.config_seed(g["seed_cfg"]))
    g = w["allreduce_rmsnorm"]
    out["allreduce_rmsnorm"] = synth.ar_inputs(g["R"], g["M"], g["N"], synth.config_seed(g["seed_cfg"]))
    return out


# --------------------------------------------------------------------------- CPU oracle timing

_ORACLE_INPUTS = {}


def oracle_sample_step(nthreads: int = 0, gemm_rows: int = 64):
    """Time the oracle as it stands on one bounded sample of the step: `gemm_rows`
    rows (spread over the matrix, every rank, full N and K) of each GEMM part
    and all rows of the AR+RMSNorm part.  Returns a dict: the measured seconds
    of the sample, the sampled fraction of each part's rows, the full step's
    time extrapolated linearly in rows, threads used and a description.  The
    synthetic operands are drawn once per process (outside the timed calls)."""
    import numpy as np

    import oracle
    import synth
    o = oracle.Oracle(0, nthreads)
    threads = o.max_threads() if nthreads == 0 else nthreads
    measured = 0.0
    full = 0.0
    frac = {}
    desc = []
    for part in ("gemm_rs", "gemm_ar"):
        w = WORKLOAD[part]
        R, M, N, K = w["R"], w["M"], w["N"], w["K"]
        rows = np.linspace(0, M - 1, gemm_rows).astype(np.int64)
        if part not in _ORACLE_INPUTS:
            seed = synth.config_seed(w["seed_cfg"])
            s = 1.0 / np.sqrt(K)
            _ORACLE_INPUTS[part] = ([synth.normal_bf16((M, K), seed, synth.T_A, r, 0.0, s) for r in range(R)],
                                    [synth.normal_bf16((K, N), seed, synth.T_B, r, 0.0, s) for r in range(R)])
        A, B = _ORACLE_INPUTS[part]
        t0 = time.perf_counter()
        o.gemm_reduce_rows(A, B, rows, "rs" if part == "gemm_rs" else "ar")
        dt = time.perf_counter() - t0
        measured += dt
        full += dt * M / gemm_rows
        frac[part] = gemm_rows / M
        desc.append(f"{part}: {gemm_rows} of {M} rows in {dt:.2f} s")
    w = WORKLOAD["allreduce_rmsnorm"]
    R, M, N = w["R"], w["M"], w["N"]
    if "allreduce_rmsnorm" not in _ORACLE_INPUTS:
        _ORACLE_INPUTS["allreduce_rmsnorm"] = synth.ar_inputs(R, M, N, synth.config_seed(w["seed_cfg"]))
    parts, res, gamma = _ORACLE_INPUTS["allreduce_rmsnorm"]
    t0 = time.perf_counter()
    o.allreduce_rmsnorm(parts, res, gamma, EPS)
    dt = time.perf_counter() - t0
    measured += dt
    full += dt
    frac["allreduce_rmsnorm"] = 1.0
    desc.append(f"allreduce_rmsnorm: all {M} rows in {dt:.3f} s")
    return {"seconds": measured, "full_step_seconds_extrapolated": full, "fraction": frac, "threads": threads,
            "sample": "; ".join(desc)}


def sample_roofline_seconds(frac, peaks, regime="burst") -> float:
    """Roofline time of the sampled work: each part's roofline time scaled by
    the fraction of its rows in the sample (the GEMMs' work is linear in rows)."""
    return sum(roofline_seconds(p, peaks, regime) * frac[p] for p in WORKLOAD)


def run_reference(args):
    """The reference arm: the oracle on the host cores.  Each step is one bounded
    sample of the workload (a row sample of each GEMM, all rows of AR+RMSNorm);
    ms_per_step is the measured time of that sample, and value is the oracle's
    throughput on it as a fraction of the roofline of the same sampled work."""
    world, rank, _ = dist_env()
    if rank != 0:
        return 0
    peaks, source = load_peaks()
    # smaller row samples when many steps are asked for, so that the run stays
    # within a few minutes
    gemm_rows = max(8, min(64, (64 * 10) // max(1, args.steps)))
    for _ in range(args.warmup):
        oracle_sample_step(gemm_rows=gemm_rows)
    runs = [oracle_sample_step(gemm_rows=gemm_rows) for _ in range(args.steps)]
    step_s = statistics.mean(r["seconds"] for r in runs)
    roof = sample_roofline_seconds(runs[0]["fraction"], peaks)
    value = 100.0 * roof / step_s
    line = {
        "impl": "reference", "metric": METRIC, "value": value, "unit": UNIT, "n_gpus": args.gpus,
        "steps": args.steps, "warmup": args.warmup, "ms_per_step": step_s * 1e3, "higher_is_better": True,
        "scaling": "weak", "vs_baseline": None, "dtype": "f32", "data": "synthetic",
        "config": config_block(),
        "step": f"one bounded sample of the workload per step: {runs[0]['sample']}",
        "ms_per_step_full_extrapolated": statistics.mean(r["full_step_seconds_extrapolated"] for r in runs) * 1e3,
        "extrapolation": "ms_per_step_full_extrapolated scales each GEMM part's measured time by M / sampled rows; "
                         "value and ms_per_step are measured on the sample, not extrapolated",
        "cpu_baseline": {"value": value, "unit": UNIT, "cores": runs[0]["threads"], "kind": "oracle",
                         "sample": runs[0]["sample"]},
        "e2e": {"value": value, "unit": UNIT, "h2d_bytes_per_step": 0, "d2h_bytes_per_step": 0},
        "peaks": {"source": source, "regime": "burst", **peaks},
    }
    print(json.dumps(line), flush=True)
    return 0


def config_block():
    return {"workload": "epilogue hot path: gemm_rs R=8 M=N=8192 K=4096 (8 owner segments) + gemm_ar R=8 "
                        "M=4096 N=7168 K=2048 (8 views) + allreduce_rmsnorm R=8 M=4096 N=7168",
            "parts": {k: {kk: vv for kk, vv in v.items() if kk != "seed_cfg"} for k, v in WORKLOAD.items()},
            "parallelism": "replicas (one full step per GPU; the ranks are emulated on each GPU)",
            "l2": "inputs larger than L2 (each part streams >= 369 MB), no flush"}


# --------------------------------------------------------------------------- every workload, one by one

# (name, op, R, M list, N, K, seed config, input distribution, chunks per owner segment)
CONFIGS = [
    ("tiny gemm_rs + rmsnorm", "gemm_rs_rmsnorm", 2, [64], 256, 128, 0, "uniform", 0),
    ("gemm_rs R=4", "gemm_rs", 4, [256, 1024, 4096, 8192], 4096, 2048, 1, "normal", 0),
    ("gemm_ar R=8", "gemm_ar", 8, [64, 512, 4096], 7168, 2048, 2, "normal", 0),
    ("allreduce_rmsnorm R=8", "allreduce_rmsnorm", 8, [1, 16, 128, 1024, 4096], 7168, 0, 3, "normal", 0),
    ("large gemm_rs R=8", "gemm_rs", 8, [8192], 8192, 4096, 4, "normal", 0),
    # the same with chunked owner-segment completion (8 chunks per segment) and the
    # destination-rotated tile order striped every 4 tile columns: the cost of the
    # counters and of the order
    ("large gemm_rs R=8, chunked + rotated", "gemm_rs", 8, [8192], 8192, 4096, 4, "normal", 8),
]


def time_calls(calls, dev, replays: int = 3, idle_s: float = 0.1):
    """Capture the callables `calls` (one library call each, on the current
    stream) in one CUDA graph, replay it once untimed, then `replays` times
    timed with CUDA events on the replay stream, each after `idle_s` seconds
    idle so that every replay starts at the burst clock (a replay of several
    milliseconds of GEMMs right after another one runs under the power cap).
    Returns the per-call times (us) of the replays."""
    import torch
    s = torch.cuda.Stream(dev)
    s.wait_stream(torch.cuda.current_stream(dev))
    with torch.cuda.stream(s):
        for c in calls[:2]:
            c()  # outside the capture once (lazy set-up)
    torch.cuda.synchronize(dev)
    g = torch.cuda.CUDAGraph()
    with torch.cuda.graph(g, stream=s):
        for c in calls:
            c()
    cur = torch.cuda.current_stream(dev)
    g.replay()
    torch.cuda.synchronize(dev)
    out = []
    for _ in range(replays):
        time.sleep(idle_s)
        e0 = torch.cuda.Event(enable_timing=True)
        e1 = torch.cuda.Event(enable_timing=True)
        e0.record(cur)
        g.replay()
        e1.record(cur)
        torch.cuda.synchronize(dev)
        out.append(e0.elapsed_time(e1) * 1e3 / len(calls))
    del g
    return out


def run_configs(ws, dev, dev_step, peaks, sampler_windows):
    """Every workload at every size: microseconds per call (CUDA graph of
    calls, median and best of 3 replays), throughput, the roofline fraction at
    the burst and sustained bf16 peaks, and which kernel ran.  Inputs are
    rotated over enough copies that the calls of one replay stream at least
    twice the L2 size (no L2 flush is needed)."""
    import numpy as np
    import torch

    import all_reduce_epilogue_gb300 as are
    import synth

    def to_dev(bits):
        return torch.from_numpy(np.ascontiguousarray(bits).view(np.int16)).view(torch.bfloat16).to(dev)

    results = []
    for name, op, R, Ms, N, K, cfg, dist_name, chunks in CONFIGS:
        seed = synth.config_seed(cfg)
        Mmax = max(Ms)
        # inputs at the largest size (row prefixes give the smaller ones)
        if op == "allreduce_rmsnorm":
            if Mmax == WORKLOAD["allreduce_rmsnorm"]["M"] and cfg == WORKLOAD["allreduce_rmsnorm"]["seed_cfg"]:
                P_full, res_full, gamma_d = dev_step["allreduce_rmsnorm"]
            else:
                ph, rh, gh = synth.ar_inputs(R, Mmax, N, seed)
                P_full, res_full, gamma_d = [to_dev(x) for x in ph], to_dev(rh), torch.from_numpy(gh).to(dev)
        else:
            key = "gemm_rs" if (op == "gemm_rs" and R == 8) else ("gemm_ar" if op == "gemm_ar" else None)
            if key and WORKLOAD[key]["M"] == Mmax and WORKLOAD[key]["seed_cfg"] == cfg:
                A_full, B_full = dev_step[key]
            else:
                Ah, Bh = synth.gemm_inputs(R, Mmax, N, K, seed, dist=dist_name)
                A_full, B_full = [to_dev(a) for a in Ah], [to_dev(b) for b in Bh]
            if op == "gemm_rs_rmsnorm":
                gamma_d = torch.from_numpy(synth.normal_f32((N,), seed, synth.T_GAMMA, 0, 1.0, 0.1)).to(dev)
        paths = ["default", "oneshot", "lamport"] if op == "allreduce_rmsnorm" else ["default"]
        for M in Ms:
            if op == "gemm_rs_rmsnorm":
                flops, byts = work_of("gemm_rs", R, M, N, K)
                f2, b2 = work_of("allreduce_rmsnorm", 1, M, N, residual=False)
                flops, byts = flops + f2, byts + b2
            elif op == "allreduce_rmsnorm":
                flops, byts = work_of(op, R, M, N)
            else:
                flops, byts = work_of(op, R, M, N, K)
            n_sets = int(min(1024, max(1, -(-2 * L2_BYTES // byts))))
            n_calls = max(n_sets, 20 if flops < 1e12 else 10)
            sets = []
            for k in range(n_sets):
                cp = (lambda t: t) if k == 0 else (lambda t: t.clone())
                if op == "allreduce_rmsnorm":
                    sets.append(([cp(x[:M]) for x in P_full], cp(res_full[:M]),
                                 torch.empty((M, N), dtype=torch.bfloat16, device=dev)))
                elif op == "gemm_ar":
                    sets.append(([cp(a[:M]) for a in A_full], [cp(b) for b in B_full],
                                 [torch.empty((M, N), dtype=torch.bfloat16, device=dev) for _ in range(R)]))
                else:
                    sets.append(([cp(a[:M]) for a in A_full], [cp(b) for b in B_full],
                                 torch.empty((M, N), dtype=torch.bfloat16, device=dev),
                                 torch.empty((M, N), dtype=torch.bfloat16, device=dev)))
            for path in paths:
                ws.set_debug({"default": 0, "oneshot": are.DEBUG_AR_ONESHOT, "lamport": are.DEBUG_AR_LAMPORT}[path])
                ws.set_chunks(chunks, 4)
                kernels = []
                if op == "allreduce_rmsnorm":
                    def mk(st):
                        return lambda: are.allreduce_rmsnorm(st[0], st[1], gamma_d, EPS, st[2], ws)
                    calls = [mk(sets[i % n_sets]) for i in range(n_calls)]
                    calls[0]()
                    kernels.append(ws.last_launch())
                elif op == "gemm_ar":
                    def mk(st):
                        return lambda: are.gemm_ar(st[0], st[1], st[2], ws)
                    calls = [mk(sets[i % n_sets]) for i in range(n_calls)]
                    calls[0]()
                    kernels.append(ws.last_launch())
                elif op == "gemm_rs":
                    def mk(st):
                        return lambda: are.gemm_rs(st[0], st[1], st[2], ws)
                    calls = [mk(sets[i % n_sets]) for i in range(n_calls)]
                    calls[0]()
                    kernels.append(ws.last_launch())
                else:
                    def mk(st):
                        def c():
                            are.gemm_rs(st[0], st[1], st[2], ws)
                            are.allreduce_rmsnorm([st[2]], None, gamma_d, EPS, st[3], ws)
                        return c
                    calls = [mk(sets[i % n_sets]) for i in range(n_calls)]
                    st0 = sets[0]
                    are.gemm_rs(st0[0], st0[1], st0[2], ws)
                    kernels.append(ws.last_launch())
                    are.allreduce_rmsnorm([st0[2]], None, gamma_d, EPS, st0[3], ws)
                    kernels.append(ws.last_launch())
                t0 = time.time()
                us = time_calls(calls, dev)
                t1 = time.time()
                ws.set_debug(0)
                ws.set_chunks(0, 0)
                stw = ws.device_status()
                if stw["code"] != 0:
                    raise RuntimeError(f"device status after {name} M={M} {path}: {stw}")
                med, best = statistics.median(us), min(us)
                d = {"workload": name, "op": op, "R": R, "M": M, "N": N, "path": path, "chunks": chunks,
                     "kernels": [f"{k['kernel']} grid={k['grid']}x{k['block']}"
                                 + (f" rank_block={k['rank_block']}" if k["kernel"] == "gemm_pair_kernel" else "")
                                 for k in kernels],
                     "us_median": med, "us_best": best, "calls_per_replay": n_calls, "input_sets": n_sets,
                     "streamed_per_replay_mb": round(n_calls * byts / 1e6, 1)}
                if K:
                    d["K"] = K
                if flops:
                    d["tflops"] = flops / (med * 1e-6) / 1e12
                d["gbs_algorithmic"] = byts / (med * 1e-6) / 1e9
                for regime in ("burst", "sustained"):
                    d[f"frac_of_roofline_{regime}"] = roofline_seconds_of(flops, byts, peaks, regime) / (med * 1e-6)
                d["bound"] = "tensor" if flops / (peaks["bf16_tflops"] * 1e12) > byts / (peaks["hbm_gbs"] * 1e9) \
                    else "hbm"
                sampler_windows.append((d, (t0, t1)))
                results.append(d)
            del sets
            torch.cuda.empty_cache()
    return results


# --------------------------------------------------------------------------- GPU arm

def run_gpu(args):
    import numpy as np
    import torch

    import all_reduce_epilogue_gb300 as are

    world, rank, local = dist_env()
    torch.cuda.set_device(local)
    dist = init_dist(world, "nccl")
    dev = torch.device("cuda", local)
    peaks, source = load_peaks()

    host = host_inputs()

    def to_dev(bits):
        return torch.from_numpy(np.ascontiguousarray(bits).view(np.int16)).view(torch.bfloat16).to(dev)

    wr, wa, wn = WORKLOAD["gemm_rs"], WORKLOAD["gemm_ar"], WORKLOAD["allreduce_rmsnorm"]
    A_rs = [to_dev(a) for a in host["gemm_rs"][0]]
    B_rs = [to_dev(b) for b in host["gemm_rs"][1]]
    A_ar = [to_dev(a) for a in host["gemm_ar"][0]]
    B_ar = [to_dev(b) for b in host["gemm_ar"][1]]
    parts_h, res_h, gamma_h = host["allreduce_rmsnorm"]
    P_n = [to_dev(x) for x in parts_h]
    res_n = to_dev(res_h)
    gamma_n = torch.from_numpy(gamma_h).to(dev)
    out_rs = torch.empty((wr["M"], wr["N"]), dtype=torch.bfloat16, device=dev)
    out_ar = [torch.empty((wa["M"], wa["N"]), dtype=torch.bfloat16, device=dev) for _ in range(wa["R"])]
    out_n = torch.empty((wn["M"], wn["N"]), dtype=torch.bfloat16, device=dev)
    ws = are.Workspace(R_max=8, M_max=max(wr["M"], wa["M"], wn["M"]), N_max=max(wr["N"], wa["N"], wn["N"]),
                       K_max=max(wr["K"], wa["K"]))
    stream = torch.cuda.current_stream(dev)

    def step(ev=None):
        if ev is not None:
            ev[0].record(stream)
        are.gemm_rs(A_rs, B_rs, out_rs, ws, stream)
        if ev is not None:
            ev[1].record(stream)
        are.gemm_ar(A_ar, B_ar, out_ar, ws, stream)
        if ev is not None:
            ev[2].record(stream)
        are.allreduce_rmsnorm(P_n, res_n, gamma_n, EPS, out_n, ws, stream)
        if ev is not None:
            ev[3].record(stream)

    for _ in range(args.warmup):
        step()
    torch.cuda.synchronize(dev)
    st = ws.device_status()
    if st["code"] != 0:
        raise RuntimeError(f"device status after warm-up: {st}")

    events = [[torch.cuda.Event(enable_timing=True) for _ in range(4)] for _ in range(args.steps)]
    sampler = ClockSampler(local)
    if dist is not None:
        dist.barrier()
    torch.cuda.synchronize(dev)
    sampler.start()
    time.sleep(0.3)
    windows = {}
    t_start = torch.cuda.Event(enable_timing=True)
    t_end = torch.cuda.Event(enable_timing=True)
    w0 = time.time()
    t_start.record(stream)
    for i in range(args.steps):
        step(events[i])
    t_end.record(stream)
    torch.cuda.synchronize(dev)
    windows["step"] = (w0, time.time())
    if dist is not None:
        dist.barrier()
    st = ws.device_status()
    if st["code"] != 0:
        raise RuntimeError(f"device status after timed steps: {st}")
    total_ms = t_start.elapsed_time(t_end)
    per = {p: [] for p in WORKLOAD}
    for ev in events:
        per["gemm_rs"].append(ev[0].elapsed_time(ev[1]))
        per["gemm_ar"].append(ev[1].elapsed_time(ev[2]))
        per["allreduce_rmsnorm"].append(ev[2].elapsed_time(ev[3]))
    ms_step = max_over_ranks(dist, total_ms / args.steps, dev)
    per_ms = {p: statistics.mean(v) for p, v in per.items()}

    # AR+RMSNorm alone, back to back: the Lamport kernel the step runs (inside the
    # step it runs after the GEMMs, which leave dirty lines in L2 and, over long runs,
    # a power-capped clock), and the one-shot kernel on the same workload (forced; the
    # default dispatch sends this size to the Lamport kernel).  A CUDA graph of calls,
    # replayed, so that no host stall between launches shows up as GPU time.
    # Reported beside the step, not part of it.
    def alone(flags):
        ws.set_debug(flags)
        n_alone = 20
        us = time_calls([lambda: are.allreduce_rmsnorm(P_n, res_n, gamma_n, EPS, out_n, ws)] * n_alone, dev)
        ws.set_debug(0)
        st = ws.device_status()
        if st["code"] != 0:
            raise RuntimeError(f"device status after AR+RMSNorm alone ({flags}): {st}")
        return max_over_ranks(dist, statistics.median(us) * 1e-3, dev)

    wa0 = time.time()
    lamport_alone_ms = alone(0)
    windows["lamport_alone"] = (wa0, time.time())
    wa0 = time.time()
    oneshot_ms = alone(are.DEBUG_AR_ONESHOT)
    windows["oneshot_alone"] = (wa0, time.time())

    # every workload at every size, one by one (after the step; outside its timed region)
    cfg_windows = []
    configs = None
    if not args.no_configs:
        configs = run_configs(ws, dev, {"gemm_rs": (A_rs, B_rs), "gemm_ar": (A_ar, B_ar),
                                              "allreduce_rmsnorm": (P_n, res_n, gamma_n)}, peaks, cfg_windows)
    sampler.stop()
    clocks = sampler.summary(windows["step"])
    regime, regime_why = peak_regime(clocks)
    for d, win in cfg_windows:
        c = sampler.summary(win)
        d["clock_mhz_median"] = c.get("sm_mhz")
        d["power_cap"] = "sw_power_cap" in (c.get("reasons") or [])

    roof = {p: roofline_seconds(p, peaks, regime) for p in WORKLOAD}
    value = world * 100.0 * sum(roof.values()) / (ms_step * 1e-3)
    parts = {}
    for p in WORKLOAD:
        flops, byts = work(p)
        d = {"ms": per_ms[p], "roofline_ms": roof[p] * 1e3, "frac_of_roofline": roof[p] / (per_ms[p] * 1e-3)}
        for reg in ("burst", "sustained"):
            d[f"frac_of_roofline_{reg}"] = roofline_seconds(p, peaks, reg) / (per_ms[p] * 1e-3)
        if flops:
            d["tflops"] = flops / (per_ms[p] * 1e-3) / 1e12
        d["gbs_algorithmic"] = byts / (per_ms[p] * 1e-3) / 1e9
        parts[p] = d
    peak_t = bf16_peak(peaks, regime)
    flops_rs, _ = work("gemm_rs")
    ach_rs = flops_rs / (per_ms["gemm_rs"] * 1e-3) / 1e12
    roofline = {"kernel": "gemm_pair_kernel<RS> (gemm_rs)", "bound": "tensor", "achieved": ach_rs,
                "peak": peak_t, "unit": "TFLOP/s", "frac": ach_rs / peak_t, "traffic": ncu_traffic("gemm_rs"),
                "peak_source": f"{source} bf16 {regime}", "peak_regime_reason": regime_why,
                "frac_burst": ach_rs / peaks["bf16_tflops"], "frac_sustained": ach_rs / peaks["bf16_tflops_sustained"],
                "ms_x_mhz": per_ms["gemm_rs"] * (clocks.get("sm_mhz") or 0.0), "note": f"of {source}"}
    _, bytes_n = work("allreduce_rmsnorm")
    ach_n = bytes_n / (per_ms["allreduce_rmsnorm"] * 1e-3) / 1e9
    roofline_ar = {"kernel": "ar_rmsnorm_kernel<4> (allreduce_rmsnorm)", "bound": "hbm", "achieved": ach_n,
                   "peak": peaks["hbm_gbs"], "unit": "GB/s", "frac": ach_n / peaks["hbm_gbs"],
                   "traffic": ncu_traffic("allreduce_rmsnorm"), "peak_source": f"{source} HBM copy",
                   "note": f"of {source}; in the step"}
    ach_alone = bytes_n / (lamport_alone_ms * 1e-3) / 1e9
    roofline_ar["alone"] = {"ms": lamport_alone_ms, "achieved": ach_alone, "frac": ach_alone / peaks["hbm_gbs"],
                            "clock_mhz_median": sampler.summary(windows["lamport_alone"]).get("sm_mhz"),
                            "note": "the same kernel outside the step: CUDA graph of 20 calls, median of 3 replays "
                                    "(inputs larger than L2)"}
    flops_ar, _ = work("gemm_ar")
    ach_ga = flops_ar / (per_ms["gemm_ar"] * 1e-3) / 1e12
    roofline_gemm_ar = {"kernel": "gemm_pair_kernel<AR> (gemm_ar)", "bound": "tensor", "achieved": ach_ga,
                        "peak": peak_t, "unit": "TFLOP/s", "frac": ach_ga / peak_t, "traffic": ncu_traffic("gemm_ar"),
                        "peak_source": f"{source} bf16 {regime}"}

    # ---- end to end: pinned host inputs -> device, the three calls, results -> host
    e2e_steps = max(1, min(args.steps, 5))
    pin = lambda bits: torch.from_numpy(np.ascontiguousarray(bits).view(np.int16)).pin_memory()  # noqa: E731
    hA_rs = [pin(a) for a in host["gemm_rs"][0]]
    hB_rs = [pin(b) for b in host["gemm_rs"][1]]
    hA_ar = [pin(a) for a in host["gemm_ar"][0]]
    hB_ar = [pin(b) for b in host["gemm_ar"][1]]
    hP = [pin(x) for x in parts_h]
    hres = pin(res_h)
    hgamma = torch.from_numpy(gamma_h).pin_memory()
    ho_rs = torch.empty(out_rs.shape, dtype=torch.int16).pin_memory()
    ho_ar = [torch.empty(o.shape, dtype=torch.int16).pin_memory() for o in out_ar]
    ho_n = torch.empty(out_n.shape, dtype=torch.int16).pin_memory()
    h2d = sum(t.numel() * t.element_size() for t in hA_rs + hB_rs + hA_ar + hB_ar + hP + [hres, hgamma])
    d2h = sum(t.numel() * t.element_size() for t in [ho_rs, ho_n] + ho_ar)

    # Three streams: host->device copies, the three calls, device->host copies.
    # A part starts as soon as its inputs have landed and its outputs go back while
    # the next part runs; every step still copies all of its inputs in and all of
    # its outputs out inside the timed region.  Buffers are reused across steps, so
    # a part's input copy waits for the previous step's call of that part, and its
    # call waits for the previous step's read-back of its outputs.
    s_in = torch.cuda.Stream(dev)
    s_out = torch.cuda.Stream(dev)
    parts_io = [
        (list(zip(hA_rs + hB_rs, A_rs + B_rs)), lambda: are.gemm_rs(A_rs, B_rs, out_rs, ws, stream),
         [(ho_rs, out_rs)]),
        (list(zip(hA_ar + hB_ar, A_ar + B_ar)), lambda: are.gemm_ar(A_ar, B_ar, out_ar, ws, stream),
         list(zip(ho_ar, out_ar))),
        (list(zip(hP + [hres], P_n + [res_n])),
         lambda: are.allreduce_rmsnorm(P_n, res_n, gamma_n, EPS, out_n, ws, stream), [(ho_n, out_n)]),
    ]
    prev = {"computed": [None] * 3, "out_done": [None] * 3}

    def e2e_step():
        in_ready = []
        for i, (ins, _, _) in enumerate(parts_io):
            with torch.cuda.stream(s_in):
                if prev["computed"][i] is not None:
                    s_in.wait_event(prev["computed"][i])
                for h, d in ins:
                    d.view(torch.int16).copy_(h, non_blocking=True)
                if i == 2:
                    gamma_n.copy_(hgamma, non_blocking=True)
                ev = torch.cuda.Event()
                ev.record(s_in)
                in_ready.append(ev)
        computed, out_done = [], []
        for i, (_, call, outs) in enumerate(parts_io):
            stream.wait_event(in_ready[i])
            if prev["out_done"][i] is not None:
                stream.wait_event(prev["out_done"][i])
            call()
            ev = torch.cuda.Event()
            ev.record(stream)
            computed.append(ev)
            with torch.cuda.stream(s_out):
                s_out.wait_event(ev)
                for h, d in outs:
                    h.copy_(d.view(torch.int16), non_blocking=True)
                ev2 = torch.cuda.Event()
                ev2.record(s_out)
                out_done.append(ev2)
        prev["computed"], prev["out_done"] = computed, out_done

    e2e_step()
    torch.cuda.synchronize(dev)
    # the host link on its own, just before: one step's input copies alone (pinned host ->
    # device, one stream), so the e2e figure can be read against the link it ran on (the host
    # memory and its link are shared with other jobs on the machine)
    l0 = torch.cuda.Event(enable_timing=True)
    l1 = torch.cuda.Event(enable_timing=True)
    l0.record(s_in)
    for ins, _, _ in parts_io:
        for h, d in ins:
            d.view(torch.int16).copy_(h, non_blocking=True)
    l1.record(s_in)
    torch.cuda.synchronize(dev)
    link_h2d_gbs = (h2d - hgamma.numel() * 4) / (l0.elapsed_time(l1) * 1e-3) / 1e9
    if dist is not None:
        dist.barrier()
    e0 = torch.cuda.Event(enable_timing=True)
    e1 = torch.cuda.Event(enable_timing=True)
    e0.record(stream)
    s_in.wait_event(e0)
    s_out.wait_event(e0)
    for _ in range(e2e_steps):
        e2e_step()
    for ev in prev["out_done"]:
        stream.wait_event(ev)
    e1.record(stream)
    torch.cuda.synchronize(dev)
    e2e_ms = max_over_ranks(dist, e0.elapsed_time(e1) / e2e_steps, dev)
    e2e_value = world * 100.0 * sum(roof.values()) / (e2e_ms * 1e-3)
    st = ws.device_status()
    if st["code"] != 0:
        raise RuntimeError(f"device status after e2e steps: {st}")

    cpu = None
    if rank == 0 and world == 1 and not args.no_cpu_baseline:
        # the oracle on the host cores, on one bounded sample of the step: the value is
        # its throughput on that sample as a fraction of the sampled work's roofline
        r = oracle_sample_step()
        cpu = {"value": 100.0 * sample_roofline_seconds(r["fraction"], peaks, regime) / r["seconds"], "unit": UNIT,
               "cores": r["threads"], "kind": "oracle", "sample": r["sample"], "ms_sample_measured": r["seconds"] * 1e3,
               "ms_per_step_full_extrapolated": r["full_step_seconds_extrapolated"] * 1e3}
        # the same oracle on one thread, on a smaller row sample
        r1 = oracle_sample_step(nthreads=1, gemm_rows=8)
        cpu["single_thread"] = {"value": 100.0 * sample_roofline_seconds(r1["fraction"], peaks, regime) / r1["seconds"],
                                "cores": 1, "sample": r1["sample"], "ms_sample_measured": r1["seconds"] * 1e3,
                                "ms_per_step_full_extrapolated": r1["full_step_seconds_extrapolated"] * 1e3}

    if rank == 0:
        line = {
            "metric": METRIC, "value": value, "unit": UNIT, "n_gpus": world, "steps": args.steps,
            "warmup": args.warmup, "ms_per_step": ms_step, "higher_is_better": True, "scaling": "weak",
            "vs_baseline": None, "dtype": "bf16", "data": "synthetic (seeded generator, shapes of the workloads)",
            "config": config_block(),
            "parts": parts,
            "roofline": roofline,
            "roofline_gemm_ar": roofline_gemm_ar,
            "roofline_allreduce_rmsnorm": roofline_ar,
            "configs": configs,
            "allreduce_rmsnorm_oneshot": {
                "kernel": "ar_oneshot_kernel<4> (same workload, path forced; outside the step)",
                "ms": oneshot_ms, "gbs_algorithmic": work("allreduce_rmsnorm")[1] / (oneshot_ms * 1e-3) / 1e9,
                "timing": "CUDA graph of 20 calls, median of 3 replays",
                "clock_mhz_median": sampler.summary(windows["oneshot_alone"]).get("sm_mhz"),
                "frac": work("allreduce_rmsnorm")[1] / (oneshot_ms * 1e-3) / 1e9 / peaks["hbm_gbs"],
                "vs_lamport_in_step": per_ms["allreduce_rmsnorm"] / oneshot_ms},
            "cpu_baseline": cpu,
            "clocks": clocks,
            "e2e": {"value": e2e_value, "unit": UNIT, "h2d_bytes_per_step": h2d, "d2h_bytes_per_step": d2h,
                    "ms_per_step": e2e_ms, "steps": e2e_steps,
                    "overlap": "host->device copies, the calls and device->host copies on three streams",
                    "link_h2d_gbs": link_h2d_gbs},
            "gpu_launches": 3 * args.steps,
            "peaks": {"source": source, "regime": regime, **peaks},
        }
        print(json.dumps(line), flush=True)
    ws.close()
    if dist is not None:
        dist.barrier()
        dist.destroy_process_group()
    return 0


def main():
    ap = argparse.ArgumentParser(description=__doc__, formatter_class=argparse.RawDescriptionHelpFormatter)
    ap.add_argument("--gpus", type=int, default=1)
    ap.add_argument("--steps", type=int, default=None,
                    help="timed steps (default: 300 for this implementation, about a second of timed work so "
                         "that the clock samples fall under load; 10 for --impl reference)")
    ap.add_argument("--warmup", type=int, default=3)
    ap.add_argument("--impl", default="ours", choices=["ours", "reference"])
    ap.add_argument("--no-cpu-baseline", action="store_true", help="skip the oracle timing (profiling runs)")
    ap.add_argument("--no-configs", action="store_true", help="skip the per-workload timings (profiling runs)")
    args = ap.parse_args()
    if args.steps is None:
        args.steps = 10 if args.impl == "reference" else 300
    if args.warmup < 3 and args.impl == "ours":
        sys.stderr.write("note: fewer than 3 warm-up steps\n")
    if args.impl == "reference":
        return run_reference(args)
    return run_gpu(args)


if __name__ == "__main__":
    sys.exit(main())
