#!/usr/bin/env python
"""Benchmark of the MoE FFN layer forward on B300: prints ONE JSON line (rank 0).

    python bench.py [--gpus N] [--steps K] [--warmup W] [--workload NAME] [--extra-workloads LIST]
                    [--impl ours|reference]

A step is one moe_layer_forward over one batch of synthetic input (router ->
grouping -> grouped SwiGLU GEMMs -> combine). The headline workload (the line's
own keys) is the Mixtral-8x7B-shaped prefill layer (T=4096, d=4096, 8 experts,
top-2, d_ff=14336); the other four model-shaped layers (Qwen3-30B-A3B-shaped,
DeepSeek-V3-shaped with capacity drops and a shared expert, the decode-shaped
batch of 32 tokens, the tiny float32 layer) are measured the same way in the same
run and reported under "workloads", one entry each.

value        tokens/s with inputs resident in HBM: K steps timed with CUDA events
             (barrier + synchronize on both sides, max over ranks); the expert
             weights exceed the 126 MB L2, so every step streams them from HBM.
             The K moe_layer_forward calls run as one CUDA-graph replay; about one
             layer in 25 (at least two) carries CUDA events at the stage boundaries,
             so the stage times come from the timed replay itself, under the same
             clocks and power. --eager: K separate calls with the stage events.
e2e          the same metric through the same C-ABI call with the activations in
             pinned host memory: each step copies x host->device, runs the layer and
             copies out device->host. Steps with at least 1 MB of activations run their
             copies on their own streams, overlapping the neighbouring steps' layers;
             smaller steps run serially on one stream. Both loops are reported.
roofline     the dominant kernel (the gate/up grouped GEMM), timed by events recorded
             around it on the launching stream, in the layers that carry them.
cpu_baseline the fp64 CPU oracle on a bounded sample of the same workload: the whole
             batch's routing and grouping, the expert MLPs and combine of a token sample.
--impl reference  times that oracle alone on the host cores, step by step, each step
             the same kind of bounded sample of the headline workload.
N > 1 (torchrun): every rank runs its own replica of the layer (the layer has no
exchange step), value = all ranks' tokens / max time.
"""
from __future__ import annotations

import argparse
import hashlib
import json
import math
import os
import re
import statistics
import subprocess
import sys
import tempfile
import time

ROOT = os.path.dirname(os.path.abspath(__file__))
sys.path.insert(0, ROOT)

METRIC = "MoE layer tokens/s on 1 B300"
UNIT = "tokens/s"
OVERLAP_MIN_BYTES = 1 << 20          # end-to-end loop: overlap the copies from this size
E2E_WARM_S = 0.3                     # end-to-end loops: warm-up wall time
E2E_MIN_S = 0.3                      # end-to-end loops: least timed device time
PEAKS_FILE = os.path.join(ROOT, "MEASURED_PEAKS.json")
TRAFFIC_FILE = os.path.join(ROOT, "profiles", "traffic.json")
FALLBACK_PEAKS = {"hbm_gbs": 6400.0, "bf16_tflops": 1800.0, "bf16_tflops_sustained": 1400.0}
HEADLINE = "mixtral_8x7b"
EXTRA_WORKLOADS = ("qwen3_30b_a3b", "deepseek_v3", "decode_qwen3", "tiny_f32")
# tokens whose expert MLPs the CPU oracle runs (the routing and grouping always cover the whole
# batch); sized for a few seconds of fp64 work each, weights generated outside the timing
CPU_SAMPLE_TOKENS = {"mixtral_8x7b": 512, "qwen3_30b_a3b": 512, "deepseek_v3": 16, "decode_qwen3": 32,
                     "tiny_f32": 64}
REF_TOKENS_PER_STEP = {"mixtral_8x7b": 512, "qwen3_30b_a3b": 64, "deepseek_v3": 2, "decode_qwen3": 32,
                       "tiny_f32": 64}
CPU_MIN_S = 0.5                      # CPU baseline: repeat a small sample to at least this much time
CPU_MAX_REPS = 200
# float32 FMA rate of the CUDA cores: 148 SMs x 128 lanes x 2 flops x 2.032 GHz
F32_FMA_TFLOPS = 148 * 128 * 2 * 2.032e9 / 1e12
NOMINAL_HBM_GBS = 8000.0             # HBM3e's nominal ~8 TB/s (the measured copy bandwidth is the roofline)


def parse_args(argv=None):
    ap = argparse.ArgumentParser()
    ap.add_argument("--gpus", type=int, default=1)
    ap.add_argument("--steps", type=int, default=100)
    ap.add_argument("--warmup", type=int, default=10)
    ap.add_argument("--workload", default=HEADLINE)
    ap.add_argument("--extra-workloads", default=None,
                    help="comma-separated workloads measured after the headline one and reported under "
                         "'workloads' (default: the other four model-shaped layers when the headline is "
                         f"{HEADLINE}, none otherwise; 'none' for none)")
    ap.add_argument("--impl", choices=["ours", "reference"], default="ours")
    ap.add_argument("--e2e-steps", type=int, default=None,
                    help="end-to-end steps per loop (default: at least 100 and 0.3 s of layers)")
    ap.add_argument("--no-cpu-baseline", action="store_true")
    ap.add_argument("--cpu-sample-tokens", type=int, default=None,
                    help="tokens whose expert MLPs the CPU oracle runs (default: per workload)")
    ap.add_argument("--weights", choices=["bf16", "fp8", "w8a8"], default="bf16",
                    help="expert weights as stored: bf16, or FP8 E4M3 codes with per-row scales (fp8), or "
                         "those weights with the expert inputs quantised to E4M3 per row as well (w8a8)")
    ap.add_argument("--traffic-kind", choices=["bf16", "fp8", "w8a8", "fused", "w8a8_fused"], default=None,
                    help="with --write-traffic: which kernels the CSVs hold (default: --weights)")
    ap.add_argument("--write-traffic", metavar="CSV_DIR", default=None,
                    help="write profiles/traffic.json from ncu CSVs traffic_<workload>.csv in CSV_DIR (see "
                         "write_traffic) and exit")
    ap.add_argument("--combine", choices=["separate", "fused"], default="separate",
                    help="combine as its own kernel (default), or fused into the down projection's "
                         "epilogue as float32 reductions (sets MOE_FUSED_COMBINE=1)")
    ap.add_argument("--no-w8a8", action="store_true",
                    help="skip the W8A8 (E4M3 weights and activations) measurement of each bf16 workload that "
                         "the default multi-workload line adds under 'w8a8'")
    ap.add_argument("--eager", action="store_true",
                    help="time K separate launches of the layer instead of CUDA-graph replays")
    return ap.parse_args(argv)


def extra_workloads(args) -> list:
    if args.extra_workloads is None:
        return list(EXTRA_WORKLOADS) if args.workload == HEADLINE and args.gpus == 1 else []
    if args.extra_workloads.strip().lower() in ("", "none"):
        return []
    return [n.strip() for n in args.extra_workloads.split(",") if n.strip() and n.strip() != args.workload]


# ----------------------------------------------------------------- helpers

def dist_env():
    world = int(os.environ.get("WORLD_SIZE", "1"))
    rank = int(os.environ.get("RANK", "0"))
    local = int(os.environ.get("LOCAL_RANK", "0"))
    return world, rank, local


def load_peaks():
    try:
        with open(PEAKS_FILE) as f:
            p = json.load(f)
        return p, "measured"
    except (OSError, ValueError):
        return dict(FALLBACK_PEAKS), "fallback"


def algorithmic(w, kept_pairs: int, groups_touched: int, weight_bytes: float = 2.0):
    """Work of one layer forward, from the realised routing (counted, not estimated).
    weight_bytes: bytes per stored expert weight (2 for bf16, 4 for float32, 1 for FP8 codes,
    whose per-row float32 scales are counted too). Activations are bf16 (float32 layers: 4 bytes)."""
    rows = kept_pairs + w.n_shared * w.T
    d, F = w.d_model, w.d_ff
    e = 2 if w.dtype == "bf16" else 4   # bytes per activation
    scales = 4.0 if weight_bytes < 2 else 0.0
    gu_w = groups_touched * 2.0 * F * (d * weight_bytes + scales)
    dn_w = groups_touched * 1.0 * d * (F * weight_bytes + scales)
    return {
        "gateup_flops": 4.0 * d * F * rows,
        "down_flops": 2.0 * d * F * rows,
        "router_flops": 2.0 * w.T * d * w.n_experts,
        "gateup_bytes": gu_w + rows * d * e + rows * F * e,
        "down_bytes": dn_w + rows * F * e + rows * d * e,
        "weight_bytes": gu_w + dn_w,
    }


def layer_totals(w, kept_pairs: int, groups_touched: int, weight_bytes: float = 2.0) -> dict:
    """Flops and HBM bytes of one whole layer forward with its intermediate round trips: the
    expert MLPs and the router; the touched experts' weights, x in, the grouped x rows written
    and read, h written and read, the grouped outputs written and read, and the output."""
    rows = kept_pairs + w.n_shared * w.T
    d, F = w.d_model, w.d_ff
    e = 2 if w.dtype == "bf16" else 4
    flops = 6.0 * d * F * rows + 2.0 * w.T * d * w.n_experts
    weights = groups_touched * 3.0 * d * F * weight_bytes
    bytes_ = (weights + w.T * d * e + kept_pairs * d * e * 2 + rows * F * e * 2 + rows * d * e * 2
              + w.T * d * e)
    return {"flops": flops, "bytes": bytes_}


class ClockSampler:
    """nvidia-smi clocks and throttle reasons sampled every 200 ms during the timed region."""
    FIELDS = ("index,clocks.sm,clocks.max.sm,power.draw,clocks_event_reasons.active,"
              "clocks_event_reasons.hw_slowdown,clocks_event_reasons.hw_thermal_slowdown,"
              "clocks_event_reasons.sw_thermal_slowdown,clocks_event_reasons.sw_power_cap")

    def __init__(self, gpu_id: str):
        self.gpu_id = gpu_id
        self.proc = None
        self.tmp = None

    def start(self):
        self.tmp = tempfile.NamedTemporaryFile("w+", suffix=".csv", delete=False)
        try:
            self.proc = subprocess.Popen(["nvidia-smi", f"--id={self.gpu_id}", f"--query-gpu={self.FIELDS}",
                                          "--format=csv,noheader,nounits", "-lms", "200"],
                                         stdout=self.tmp, stderr=subprocess.DEVNULL)
        except OSError:
            self.proc = None
        time.sleep(0.25)

    def stop(self):
        if self.proc is None:
            return {"sm_mhz": None, "sm_max_mhz": None, "reasons": ["nvidia-smi unavailable"]}
        time.sleep(0.25)
        self.proc.terminate()
        try:
            self.proc.wait(timeout=5)
        except subprocess.TimeoutExpired:
            self.proc.kill()
        self.tmp.flush()
        self.tmp.seek(0)
        text = self.tmp.read()
        os.unlink(self.tmp.name)
        return self.parse(text)

    @staticmethod
    def parse(text: str) -> dict:
        """Median SM clock, highest max clock and power, and every throttle reason seen active,
        from nvidia-smi CSV lines in FIELDS order (malformed lines are skipped)."""
        sm, smax, power, reasons = [], [], [], set()
        names = ["hw_slowdown", "hw_thermal_slowdown", "sw_thermal_slowdown", "sw_power_cap"]
        for line in text.splitlines():
            parts = [p.strip() for p in line.split(",")]
            if len(parts) < 9:
                continue
            try:
                sm.append(float(parts[1]))
                smax.append(float(parts[2]))
                power.append(float(parts[3]))
            except ValueError:
                continue
            for n, v in zip(names, parts[5:9]):
                if v.lower() == "active":
                    reasons.add(n)
        return {"sm_mhz": statistics.median(sm) if sm else None, "sm_max_mhz": max(smax) if smax else None,
                "power_w_max": max(power) if power else None, "samples": len(sm), "reasons": sorted(reasons)}


GEMM_SOURCES = {"bf16": ("gemm_tc.cu", "epilogue.cuh", "gemm_common.cuh", "tc_ptx.cuh"),
                "fused": ("gemm_fused.cu", "epilogue.cuh", "gemm_common.cuh", "tc_ptx.cuh"),
                "fp8": ("gemm_fp8w.cu", "gemm_common.cuh", "tc_ptx.cuh"),
                "w8a8": ("gemm_w8a8.cu", "epilogue.cuh", "fp8_quant.cuh", "gemm_common.cuh", "tc_ptx.cuh"),
                "w8a8_fused": ("gemm_w8a8_fused.cu", "epilogue.cuh", "fp8_quant.cuh", "gemm_common.cuh", "tc_ptx.cuh")}


def code_only(src: str) -> str:
    """C/CUDA source without its comments and blank lines (none of the hashed files has a
    comment marker inside a string literal), so that editing comments keeps the hash."""
    src = re.sub(r"/\*.*?\*/", "", src, flags=re.S)
    src = re.sub(r"//[^\n]*", "", src)
    return "\n".join(line.rstrip() for line in src.splitlines() if line.strip())


def kernel_source_hash(weights: str = "bf16") -> str:
    """SHA-256 of the GEMM kernel's code (comments removed): a traffic capture stays valid
    exactly as long as this is unchanged."""
    h = hashlib.sha256()
    for fn in GEMM_SOURCES[weights]:
        with open(os.path.join(ROOT, "sparse_expert_mlp_router_b300", "csrc", fn)) as f:
            h.update(code_only(f.read()).encode())
    return h.hexdigest()


def measured_traffic(workload: str, weights: str = "bf16"):
    """DRAM bytes per launch of the gate/up GEMM from a committed ncu capture, if that capture
    was taken of the current kernel source; otherwise None."""
    try:
        with open(TRAFFIC_FILE) as f:
            t = json.load(f)
    except (OSError, ValueError):
        return None
    e = t.get(workload if weights == "bf16" else workload + "+" + weights)
    if not e or e.get("source_sha256") != kernel_source_hash(weights):
        return None
    return e.get("bytes_per_launch")


def write_traffic(csv_dir: str, weights: str) -> None:
    """profiles/traffic.json from one-pass ncu captures, one CSV per workload, made with

        ncu --metrics dram__bytes_read.sum,dram__bytes_write.sum,gpu__time_duration.sum \\
            --clock-control none -k regex:grouped_gemm -s 2 -c 2 --csv --log-file traffic_<workload>.csv \\
            python bench.py --workload <workload> --steps 3 --warmup 1 --e2e-steps 1 --no-cpu-baseline \\
            --eager [--weights fp8]

    (the second layer forward's gate/up and down GEMMs; with --weights fused, -k regex:grouped_mlp_fused -c 1 on a
    layer that runs the expert MLP as one launch). Each entry records the hash of the GEMM source it was measured
    on; the roofline reports the traffic only while that source is unchanged.
    """
    import csv
    import glob
    out = json.load(open(TRAFFIC_FILE)) if os.path.exists(TRAFFIC_FILE) else {}
    sha = kernel_source_hash(weights)
    for fn in sorted(glob.glob(os.path.join(csv_dir, "traffic_*.csv"))):
        wl = os.path.basename(fn)[len("traffic_"):-len(".csv")]
        rows = [r for r in csv.reader(open(fn)) if len(r) > 10]
        hdr = rows[0]
        ki, mi, vi, ids = (hdr.index(c) for c in ("Kernel Name", "Metric Name", "Metric Value", "ID"))
        per = {}
        for r in rows[1:]:
            per.setdefault(r[ids], {"k": r[ki]})[r[mi]] = float(r[vi].replace(",", ""))
        gu = list(per.values())[0]                 # gate/up is launched before down
        key = wl if weights == "bf16" else wl + "+" + weights
        out[key] = {"source_sha256": sha, "kernel": gu["k"][:60],
                    "bytes_per_launch": gu["dram__bytes_read.sum"] + gu["dram__bytes_write.sum"],
                    "read": gu["dram__bytes_read.sum"], "write": gu["dram__bytes_write.sum"],
                    "ns_under_ncu": gu["gpu__time_duration.sum"]}
        if weights not in ("fused", "w8a8_fused"):  # the one-launch MLP has no separate down kernel
            dn = list(per.values())[1]
            out[key]["down_bytes_per_launch"] = dn["dram__bytes_read.sum"] + dn["dram__bytes_write.sum"]
    out["_comment"] = ("DRAM bytes per launch of the gate/up grouped GEMM (and of the down GEMM) from one-pass ncu "
                       "captures; written by `python bench.py --write-traffic DIR`, see write_traffic().")
    with open(TRAFFIC_FILE, "w") as f:
        json.dump(out, f, indent=1, sort_keys=True)


def cpu_threads() -> int:
    try:
        from threadpoolctl import threadpool_info
        n = [i["num_threads"] for i in threadpool_info() if i.get("user_api") == "blas"]
        if n:
            return int(max(n))
    except Exception:
        pass
    return os.cpu_count() or 1


def cpu_model() -> str:
    try:
        with open("/proc/cpuinfo") as f:
            for line in f:
                if line.startswith("model name"):
                    return line.split(":", 1)[1].strip()
    except OSError:
        pass
    return "unknown"


def config_of(w, kept: int, touched: int, world: int, weights: str) -> dict:
    """The `config` object of a bench line: what the workload is, identical in both arms."""
    fp8 = weights in ("fp8", "w8a8")
    return {"workload": w.name, "T": w.T, "d_model": w.d_model, "n_experts": w.n_experts,
            "n_shared": w.n_shared, "top_k": w.top_k, "d_ff": w.d_ff, "score": w.score,
            "renormalize": bool(w.renormalize), "capacity_factor": w.capacity_factor, "kept_pairs": int(kept),
            "groups_touched": int(touched),
            "l2": "inputs larger than L2: %.2f GB of expert weights streamed per step"
                  % (touched * 3.0 * w.d_model * w.d_ff * (1 if fp8 else (2 if w.dtype == "bf16" else 4)) / 1e9)
                  if touched * 3.0 * w.d_model * w.d_ff * 2 > 126e6 else
                  "inputs smaller than L2 (%.1f MB of expert weights): a latency-bound layer"
                  % (touched * 3.0 * w.d_model * w.d_ff * (2 if w.dtype == "bf16" else 4) / 1e6),
            "parallelism": "replicas" if world > 1 else "single GPU",
            "weights": ("fp8 e4m3, per-row float32 scales" + (
                "; activations e4m3 per row too (w8a8)" if weights == "w8a8" else "")) if fp8 else w.dtype}


# ----------------------------------------------------------- the CPU oracle

class OracleSample:
    """The fp64 oracle's layer forward on a bounded sample of a workload.

    Each call routes and groups the whole batch (admission under a capacity limit depends on
    the whole batch) and runs the expert MLPs and the combine for `n_tokens` tokens of it.
    Expert weights are generated on the host and converted to float64 either once before any
    timing (`preload`, when they fit in `max_cached_bytes`) or on demand, one expert at a
    time; the time spent generating them is measured and excluded from the oracle's time.
    """

    def __init__(self, w, n_tokens: int, seed: int = 0, max_cached_bytes: float = 24e9):
        import numpy as np
        import oracle as O
        import synth
        self.w, self.O, self.synth, self.np = w, O, synth, np
        self.x64 = synth.as_f64(synth.host_tensor(w, "x"), w.dtype)
        self.wr64 = synth.as_f64(synth.host_tensor(w, "w_router"), w.dtype)
        self.bias = synth.router_bias(w.n_experts, w.bias_s)
        self.n = max(1, min(n_tokens, w.T))
        self.rng = np.random.default_rng(seed)
        self.kw = dict(top_k=w.top_k, score=w.score, renormalize=w.renormalize,
                       capacity_factor=w.capacity_factor, n_shared=w.n_shared)
        self.gen_s = 0.0
        self.cache = {}
        self.per_expert = 3.0 * w.d_model * w.d_ff * 8
        self.max_cached = max_cached_bytes
        self.lazy = True

    def preload(self, token_sets) -> None:
        """Generate before timing the experts the given token sets will touch, if they fit."""
        np, O = self.np, self.O
        idx, _, _ = O.route(self.x64, self.wr64, self.bias, self.w.top_k, self.w.score, self.w.renormalize)
        need = set()
        for toks in token_sets:
            need |= set(np.unique(idx[toks]).tolist())
        need |= set(range(self.w.n_experts, self.w.n_experts + self.w.n_shared))
        if len(need) * self.per_expert > self.max_cached:
            return
        for g in sorted(need):
            self.cache[g] = self._gen(g)
        self.lazy = False

    def _gen(self, g):
        return tuple(self.synth.as_f64(a, self.w.dtype) for a in self.synth.host_expert(self.w, g))

    def experts(self, g):
        if g in self.cache:
            return self.cache[g]
        t0 = time.perf_counter()
        if self.lazy:
            self.cache.clear()
        v = self.cache[g] = self._gen(g)
        self.gen_s += time.perf_counter() - t0
        return v

    def draw(self):
        return self.np.sort(self.rng.choice(self.w.T, size=self.n, replace=False))

    def run(self, toks) -> tuple:
        """One oracle layer forward restricted to `toks`; returns (tokens, oracle seconds)."""
        g0 = self.gen_s
        t0 = time.perf_counter()
        self.O.layer_forward(self.x64, self.wr64, self.bias, self.experts, tokens=toks, **self.kw)
        dt = time.perf_counter() - t0 - (self.gen_s - g0)
        return len(toks), dt

    def describe(self, steps: int = 1) -> str:
        per = f"expert MLPs and combine of {self.n} sampled tokens" + (" per step" if steps > 1 else "")
        return (f"{self.w.name}: routing and grouping of the whole {self.w.T}-token batch, {per}; "
                f"weight generation excluded")


ONE_CORE_ENV = {"OMP_NUM_THREADS": "1", "OPENBLAS_NUM_THREADS": "1", "MKL_NUM_THREADS": "1",
                "BLIS_NUM_THREADS": "1", "NUMEXPR_NUM_THREADS": "1"}


def cpu_baseline(w, n_tokens: int, one_core: bool = False) -> dict:
    """The oracle timed once on a bounded sample of workload w, on all host cores, or (one_core)
    in a child process whose BLAS and OpenMP thread pools are limited to one thread."""
    if one_core:
        code = ("import json, sys; sys.path.insert(0, %r); import bench, synth; "
                "print(json.dumps(bench.cpu_baseline(synth.WORKLOADS[%r], %d)))" % (ROOT, w.name, n_tokens))
        r = subprocess.run([sys.executable, "-c", code], env=dict(os.environ, **ONE_CORE_ENV), capture_output=True,
                           text=True, timeout=600)
        if r.returncode != 0:
            return {"value": None, "error": r.stderr.strip().splitlines()[-1:] or ["failed"]}
        res = json.loads(r.stdout.strip().splitlines()[-1])
        res["cores"] = 1
        res["threads"] = "BLAS / OpenMP pools limited to 1 thread (" + ", ".join(sorted(ONE_CORE_ENV)) + ")"
        return res
    s = OracleSample(w, n_tokens)
    toks = s.draw()
    s.preload([toks])
    n, dt, reps = 0, 0.0, 0
    while reps < CPU_MAX_REPS and (reps == 0 or dt < CPU_MIN_S):   # small layers: repeat to a measurable time
        a, b = s.run(toks)
        n, dt, reps = n + a, dt + b, reps + 1
    return {"value": n / dt, "unit": UNIT, "cores": cpu_threads(), "kind": "oracle",
            "sample": s.describe() + (f", {reps} repetitions" if reps > 1 else ""),
            "seconds": dt, "cpu_model": cpu_model(), "nproc": os.cpu_count()}


def max_over_ranks(ms: float, dist=None, device="cuda") -> float:
    """The slowest rank's time (every rank passes its own; all get the maximum)."""
    if dist is None:
        return ms
    import torch
    t = torch.tensor([ms], dtype=torch.float64, device=device)
    dist.all_reduce(t, op=dist.ReduceOp.MAX)
    return float(t.item())


def whole_job_rate(tokens_per_step: int, steps: int, world: int, max_ms: float) -> float:
    """Tokens per second of the whole job: every rank's tokens over the slowest rank's time."""
    return tokens_per_step * steps * world / (max_ms / 1e3)


def run_reference(args, w):
    """The reference arm: the fp64 oracle alone on the host cores. Each step is one oracle layer
    forward over the whole batch's routing and grouping with the expert MLPs and combine of a
    fresh token sample, as in the CPU baseline; value = sampled tokens / oracle time."""
    import numpy as np
    world, rank, _ = dist_env()
    if rank != 0:
        return
    n_tok = args.cpu_sample_tokens or REF_TOKENS_PER_STEP.get(w.name, 64)
    s = OracleSample(w, n_tok)
    samples = [s.draw() for _ in range(args.warmup + args.steps)]
    s.preload(samples)
    for i in range(args.warmup):
        s.run(samples[i])
    n, dt = 0, 0.0
    for i in range(args.steps):
        a, b = s.run(samples[args.warmup + i])
        n, dt = n + a, dt + b
    value = n / dt if dt > 0 else 0.0
    idx, _, _ = s.O.route(s.x64, s.wr64, s.bias, w.top_k, w.score, w.renormalize)
    counts = np.bincount(idx.ravel(), minlength=w.n_experts)
    cap = s.O.capacity(w.T, w.top_k, w.n_experts, w.capacity_factor)
    kept_e = counts if cap is None else np.minimum(counts, cap)
    kept, touched = int(kept_e.sum()), int((kept_e > 0).sum()) + w.n_shared
    line = {
        "impl": "reference", "metric": METRIC, "value": value, "unit": UNIT, "n_gpus": args.gpus,
        "steps": args.steps, "warmup": args.warmup, "ms_per_step": 1e3 * dt / max(args.steps, 1),
        "higher_is_better": True, "scaling": "weak", "vs_baseline": None, "dtype": "f64", "data": "synthetic",
        "config": config_of(w, kept, touched, 1, args.weights),
        "cpu_baseline": {"value": value, "unit": UNIT, "cores": cpu_threads(), "kind": "oracle",
                         "sample": s.describe(args.steps), "cpu_model": cpu_model(), "nproc": os.cpu_count()},
        "e2e": {"value": value, "unit": UNIT, "h2d_bytes_per_step": 0, "d2h_bytes_per_step": 0},
    }
    print(json.dumps(line), flush=True)


# ------------------------------------------------------------- our layer

def staged_positions(K: int) -> list:
    """Which of the K timed layers carry the stage events: about one in 25 (at least
    min(K, 2) of them), evenly spread, the last one included."""
    n = min(K, max(2, K // 25))
    return [((j + 1) * K) // n - 1 for j in range(n)]


def measure_workload(args, w, dist, local, rank, world, with_cpu: bool, weights: str = None,
                     with_e2e: bool = True) -> dict:
    """Everything the bench reports for one workload: device-timed value, stage times, roofline,
    end-to-end rate (with_e2e), clocks and (rank 0, N = 1) the CPU oracle baseline. weights:
    bf16, fp8 or w8a8 (default: --weights)."""
    weights = args.weights if weights is None else weights
    import numpy as np
    import torch
    import synth
    import sparse_expert_mlp_router_b300 as moe

    def barrier():
        if dist is not None:
            dist.barrier()
        torch.cuda.synchronize()

    cfg = moe.make_config(T=w.T, d_model=w.d_model, n_experts=w.n_experts, top_k=w.top_k, d_ff=w.d_ff,
                          n_shared=w.n_shared, score=w.score, renormalize=w.renormalize,
                          capacity_factor=w.capacity_factor, dtype=w.dtype)
    dev = synth.device_inputs(w)
    fp8 = weights in ("fp8", "w8a8") and w.dtype == "bf16"
    a8 = fp8 and weights == "w8a8"
    if fp8:
        # FP8 codes and per-row scales made on the device by the library's quantiser; the bf16
        # copies are freed before any timing
        for name in ("w_gate", "w_up", "w_down"):
            dev[name + "_q"], dev[name + "_s"] = moe.moe_quantize_fp8_rows(dev[name])
            del dev[name]
        torch.cuda.synchronize()
        torch.cuda.empty_cache()
        wargs = (dev["w_gate_q"], dev["w_gate_s"], dev["w_up_q"], dev["w_up_s"], dev["w_down_q"], dev["w_down_s"])
        forward, forward_timed = ((moe.moe_layer_forward_w8a8, moe.moe_layer_forward_w8a8_timed) if a8 else
                                  (moe.moe_layer_forward_fp8, moe.moe_layer_forward_fp8_timed))
    else:
        wargs = (dev["w_gate"], dev["w_up"], dev["w_down"])
        forward, forward_timed = moe.moe_layer_forward, moe.moe_layer_forward_timed
    ws = moe.alloc_workspace(cfg)
    dt = dev["x"].dtype
    out = torch.empty(w.T, w.d_model, dtype=dt, device="cuda")
    counts = torch.empty(w.n_experts, dtype=torch.int32, device="cuda")
    args_fwd = (cfg, dev["x"], dev["w_router"], dev["bias"], *wargs, out, ws)

    # one checked forward: status and the realised routing (kept pairs, experts touched)
    forward(*args_fwd, counts_out=counts)
    status = moe.moe_get_device_error(ws)
    if status != moe.MOE_OK:
        raise RuntimeError(f"{w.name}: device status {moe.status_string(status)}")
    cap = moe.moe_capacity(cfg)
    c = counts.cpu().numpy()
    kept = int(np.minimum(c, cap).sum())
    touched = int((np.minimum(c, cap) > 0).sum()) + w.n_shared
    work = algorithmic(w, kept, touched, 1.0 if fp8 else (2.0 if w.dtype == "bf16" else 4.0))

    K, W = args.steps, args.warmup
    # Graph mode: the K timed steps are one CUDA-graph replay of K layer calls; a few of them,
    # evenly spread (staged_positions), are recorded with CUDA events at the five stage
    # boundaries, so the stage times come from the timed replay itself (six event records cost
    # a decode-shaped layer about 8 %, and only these layers carry them). Eager mode (--eager,
    # for profilers): K separate calls, each with the stage events.
    staged_at = staged_positions(K) if not args.eager else list(range(K))
    evs = [[torch.cuda.Event(enable_timing=True) for _ in range(6)] for _ in range(len(staged_at))]
    for row in evs:            # create every event before any capture
        for e in row:
            e.record()
    for i in range(W):
        forward_timed(*args_fwd, evs[i % len(evs)])
    barrier()
    graph = None
    if not args.eager:
        slot = {pos: j for j, pos in enumerate(staged_at)}
        graph = torch.cuda.CUDAGraph()
        with torch.cuda.graph(graph):
            for i in range(K):
                if i in slot:
                    forward_timed(*args_fwd, evs[slot[i]])
                else:
                    forward(*args_fwd)
        graph.replay()             # one untimed replay
        barrier()
    props = torch.cuda.get_device_properties(local)
    try:
        gpu_id = "%08X:%02X:%02X.0" % (props.pci_domain_id, props.pci_bus_id, props.pci_device_id)
    except AttributeError:
        gpu_id = str(local)
    sampler = ClockSampler(gpu_id)
    sampler.start()
    t_start = torch.cuda.Event(enable_timing=True)
    t_end = torch.cuda.Event(enable_timing=True)
    barrier()
    t_start.record()
    if graph is not None:
        graph.replay()
    else:
        for i in range(K):
            forward_timed(*args_fwd, evs[i])
    t_end.record()
    barrier()
    clocks = sampler.stop()
    elapsed_ms = t_start.elapsed_time(t_end)
    stage = np.array([[e[j].elapsed_time(e[j + 1]) for j in range(5)] for e in evs])   # [staged layers, 5] ms
    status = moe.moe_get_device_error(ws)
    if status != moe.MOE_OK:
        raise RuntimeError(f"{w.name}: device status after timing: {moe.status_string(status)}")
    max_ms = max_over_ranks(elapsed_ms, dist)
    value = whole_job_rate(w.T, K, world, max_ms)
    del graph

    e2e = None
    if with_e2e:
        # end to end: activations in pinned host memory, copies inside the timed region. Two loops:
        # serial (one stream: copy x in, run the layer, copy the output out), and overlapped (the
        # copies on their own streams, two device buffers of each, so that step i's copies overlap
        # the layers of steps i-1 and i+1). Cross-stream waits cost a few microseconds a step, more
        # than copies of a few hundred KB take, so the reported loop is the overlapped one when a
        # step's activations reach OVERLAP_MIN_BYTES and the serial one below; both are reported.
        x_host = dev["x"].cpu().pin_memory()
        out_hosts = [torch.empty(out.shape, dtype=dt).pin_memory() for _ in range(2)]
        x_devs = [torch.empty_like(dev["x"]) for _ in range(2)]
        out_devs = [out, torch.empty_like(out)]
        main = torch.cuda.current_stream()
        h2d, d2h = torch.cuda.Stream(), torch.cuda.Stream()
        ev_in = [torch.cuda.Event() for _ in range(2)]      # x_devs[b] holds this step's input
        ev_done = [torch.cuda.Event() for _ in range(2)]    # the layer on buffer pair b finished
        ev_out = [torch.cuda.Event() for _ in range(2)]     # out_devs[b] copied to the host

        def e2e_step(i):
            b = i % 2
            h2d.wait_event(ev_done[b])                       # the layer that read x_devs[b] is done
            with torch.cuda.stream(h2d):
                x_devs[b].copy_(x_host, non_blocking=True)
            ev_in[b].record(h2d)
            main.wait_event(ev_in[b])
            main.wait_event(ev_out[b])                       # out_devs[b] is free again
            forward(cfg, x_devs[b], dev["w_router"], dev["bias"], *wargs, out_devs[b], ws)
            ev_done[b].record(main)
            d2h.wait_event(ev_done[b])
            with torch.cuda.stream(d2h):
                out_hosts[b].copy_(out_devs[b], non_blocking=True)
            ev_out[b].record(d2h)

        def e2e_serial_step():
            x_devs[0].copy_(x_host, non_blocking=True)
            forward(cfg, x_devs[0], dev["w_router"], dev["bias"], *wargs, out_devs[0], ws)
            out_hosts[0].copy_(out_devs[0], non_blocking=True)

        # By default each loop is warmed up for E2E_WARM_S of wall time (the host's clock settles: a
        # cold host doubled the per-step cost of the smallest layers) and timed over at least
        # E2E_MIN_S of steps; --e2e-steps N times exactly N steps after a few warm-up steps.
        auto = args.e2e_steps is None
        K2 = max(100, math.ceil(E2E_MIN_S / (max_ms / K / 1e3))) if auto else max(args.e2e_steps, 1)

        def warm(fn, n_min):
            t_end = time.perf_counter() + (E2E_WARM_S if auto else 0.0)
            i = 0
            while i < n_min or time.perf_counter() < t_end:
                fn(i)
                i += 1
            torch.cuda.synchronize()

        e0 = torch.cuda.Event(enable_timing=True)
        e1 = torch.cuda.Event(enable_timing=True)
        warm(lambda i: e2e_serial_step(), 3)
        barrier()
        e0.record()
        for i in range(K2):
            e2e_serial_step()
        e1.record()
        barrier()
        serial_ms = max_over_ranks(e0.elapsed_time(e1), dist)
        warm(e2e_step, 4)                                    # the two loops share buffer 0: synchronised
        barrier()
        e0.record()
        h2d.wait_stream(main)
        d2h.wait_stream(main)
        for i in range(K2):
            e2e_step(i)
        main.wait_stream(d2h)                                # the last output has reached the host
        e1.record()
        barrier()
        overlap_ms = max_over_ranks(e0.elapsed_time(e1), dist)
        overlapped = x_host.numel() * x_host.element_size() >= OVERLAP_MIN_BYTES
        e2e_value = whole_job_rate(w.T, K2, world, overlap_ms if overlapped else serial_ms)
        if moe.moe_get_device_error(ws) != moe.MOE_OK:
            raise RuntimeError(f"{w.name}: device status after e2e timing")
        e2e = {"value": e2e_value, "unit": UNIT, "h2d_bytes_per_step": int(x_host.numel() * x_host.element_size()),
               "d2h_bytes_per_step": int(out.numel() * out.element_size()), "steps": K2,
               "copies": ("own streams, overlapping the neighbouring steps' layers (double-buffered)"
                          if overlapped else "serial, on the layer's stream (activations under %d bytes)"
                          % OVERLAP_MIN_BYTES),
               "serial_value": whole_job_rate(w.T, K2, world, serial_ms),
               "overlapped_value": whole_job_rate(w.T, K2, world, overlap_ms)}
        del x_host, out_hosts, x_devs, out_devs

    # roofline of the dominant kernel: the gate/up grouped GEMM (stage 2 -> 3). A tensor-bound
    # kernel timed inside a long run of back-to-back layers (>= 1 s, where the GPU settles at
    # its power limit) is compared with the sustained bf16 rate, else with the burst rate; the
    # fraction of the burst rate is reported as well. The float32 layer's MLP runs on the CUDA
    # cores and is compared with their FMA rate.
    # the bf16 layer's expert MLP may run as one launch of both contractions (decode-shaped
    # batches): then the dominant kernel is that launch, timed over both stages, with the flops
    # and bytes of both contractions
    one_mlp = (w.dtype == "bf16" and
               moe.moe_layer_mlp_fused_weights(cfg, "w8a8" if a8 else "fp8" if fp8 else "bf16") == 1)
    peaks, peak_src = load_peaks()
    # the E4M3 x E4M3 tensor-core rate is twice the bf16 one (nominal dense 4.5 vs 2.25 PFLOP/s):
    # W8A8 contractions are compared with twice the measured bf16 rate
    tensor_mult = 2.0 if a8 else 1.0
    pair_ms = float((stage[:, 2] + stage[:, 3]).mean())
    gemm_ms = pair_ms if one_mlp else float(stage[:, 2].mean())
    r_flops = work["gateup_flops"] + (work["down_flops"] if one_mlp else 0.0)
    r_bytes = work["gateup_bytes"] + (work["down_bytes"] if one_mlp else 0.0)
    long_run = max_ms >= 1000.0
    if w.dtype != "bf16":
        achieved = r_flops / (gemm_ms / 1e3) / 1e12
        roof = {"bound": "alu", "achieved": achieved, "peak": F32_FMA_TFLOPS, "unit": "TFLOP/s",
                "kernel": "ffn_gateup_fma_kernel (float32, CUDA cores)",
                "peak_source": "float32 FMA rate: 148 SMs x 128 lanes x 2 flops x 2.032 GHz"}
    else:
        t_tensor = r_flops / (peaks["bf16_tflops"] * tensor_mult * 1e12)
        t_bytes = r_bytes / (peaks["hbm_gbs"] * 1e9)
        if t_tensor >= t_bytes:
            achieved = r_flops / (gemm_ms / 1e3) / 1e12
            peak = tensor_mult * (peaks["bf16_tflops_sustained"] if long_run else peaks["bf16_tflops"])
            roof = {"bound": "tensor", "achieved": achieved, "peak": peak, "unit": "TFLOP/s",
                    "frac_of_burst": achieved / (peaks["bf16_tflops"] * tensor_mult)}
        else:
            achieved = r_bytes / (gemm_ms / 1e3) / 1e9
            roof = {"bound": "hbm", "achieved": achieved, "peak": peaks["hbm_gbs"], "unit": "GB/s"}
        roof["kernel"] = ("grouped_mlp_w8a8_fused_kernel<gate/up + SwiGLU, h to E4M3, then down, one launch> "
                          "(tcgen05 kind::f8f6f4)" if one_mlp and a8 else
                          ("grouped_mlp_fused_kernel<gate/up + SwiGLU, then down and the combine, one launch> (tcgen05)"
                           if os.environ.get("MOE_MLP_COMBINE") == "1" else
                           "grouped_mlp_fused_kernel<gate/up + SwiGLU, then down, one launch> (tcgen05)") if one_mlp else
                          "grouped_gemm_w8a8_kernel<gate/up, E4M3 weights and activations, SwiGLU epilogue> "
                          "(tcgen05 kind::f8f6f4)" if a8 else
                          "grouped_gemm_fp8w_kernel<gate/up, FP8 weights, SwiGLU epilogue> (tcgen05)" if fp8 else
                          "grouped_gemm_kernel<gate/up, SwiGLU epilogue> (tcgen05)")
        roof["peak_source"] = (f"{peak_src} copy bandwidth" if roof["bound"] == "hbm" else
                               (("2 x " if a8 else "") + f"{peak_src} bf16 ") +
                               (f"sustained (timed region {max_ms / 1e3:.1f} s)" if long_run else "burst"))
    roof["frac"] = roof["achieved"] / roof["peak"]
    roof["traffic"] = (measured_traffic(w.name, ("w8a8_fused" if a8 else "fused") if one_mlp else
                                        "w8a8" if a8 else "fp8" if fp8 else "bf16")
                       if w.dtype == "bf16" else None)
    roof["ms_per_launch"] = gemm_ms

    stages_ms = dict(zip(["router", "grouping", "gemm_gate_up", "gemm_down", "combine"],
                         [float(v) for v in stage.mean(axis=0)]))
    pair_flops = work["gateup_flops"] + work["down_flops"]
    layer_work = layer_totals(w, kept, touched, 1.0 if fp8 else (2.0 if w.dtype == "bf16" else 4.0))
    weight_bytes = work["weight_bytes"]
    res = {
        "value": value, "ms_per_step": max_ms / K, "steps": K,
        "config": config_of(w, kept, touched, world, weights if fp8 else "bf16"),
        "e2e": e2e,
        "gpu_launches": K * moe.moe_layer_launch_count_weights(cfg, weights if fp8 else "bf16"),
        "roofline": roof,
        "clocks": clocks,
        "stages_ms": stages_ms,
        "stages_sum_ms": float(stage.sum(axis=1).mean()),
        "grouped_gemm_tflops": pair_flops / (pair_ms / 1e3) / 1e12,
        "grouped_gemm_frac_of_burst": pair_flops / (pair_ms / 1e3) / 1e12 / (peaks["bf16_tflops"] * tensor_mult),
        "expert_weight_gbs": weight_bytes / (pair_ms / 1e3) / 1e9,
        "expert_weight_frac_of_hbm": weight_bytes / (pair_ms / 1e3) / 1e9 / peaks["hbm_gbs"],
        "grouped_gemm_frac_of_sustained": pair_flops / (pair_ms / 1e3) / 1e12 / (peaks["bf16_tflops_sustained"]
                                                                                  * tensor_mult),
        "expert_weight_frac_of_nominal_hbm": weight_bytes / (pair_ms / 1e3) / 1e9 / NOMINAL_HBM_GBS,
        # the whole layer against its own roofline: the longer of (all flops / tensor rate) and
        # (all bytes / HBM bandwidth), over the layer time
        "layer_roofline_frac": max(layer_work["flops"] / (peaks["bf16_tflops"] * tensor_mult * 1e12),
                                   layer_work["bytes"] / (peaks["hbm_gbs"] * 1e9)) / (max_ms / K / 1e3),
    }
    del dev, ws, out, counts, wargs, args_fwd
    torch.cuda.synchronize()
    torch.cuda.empty_cache()
    if with_cpu:
        n = args.cpu_sample_tokens or CPU_SAMPLE_TOKENS.get(w.name, 256)
        res["cpu_baseline"] = cpu_baseline(w, n)
        if w.name == "tiny_f32":
            res["cpu_baseline"]["one_core"] = cpu_baseline(w, n, one_core=True)
    else:
        res["cpu_baseline"] = None
    return res


def run_ours(args, w):
    import torch
    if args.combine == "fused":
        os.environ["MOE_FUSED_COMBINE"] = "1"
    world, rank, local = dist_env()
    torch.cuda.set_device(local)
    dist = None
    if world > 1:
        import torch.distributed as dist
        dist.init_process_group("nccl", device_id=torch.device("cuda", local))
    with_cpu = rank == 0 and world == 1 and not args.no_cpu_baseline
    import synth
    head = measure_workload(args, w, dist, local, rank, world, with_cpu)
    extras = {}
    for name in extra_workloads(args):
        extras[name] = measure_workload(args, synth.WORKLOADS[name], dist, local, rank, world, with_cpu)
    # the FP8 path (E4M3 weights and activations) on every bf16 workload of the line: device-timed
    # value, stages and roofline only
    if args.weights == "bf16" and not args.no_w8a8 and extras:
        for name, res in [(w.name, head)] + list(extras.items()):
            wl = synth.WORKLOADS[name]
            if wl.dtype == "bf16":
                res["w8a8"] = measure_workload(args, wl, dist, local, rank, world, False, weights="w8a8",
                                               with_e2e=False)
    line = {
        "metric": METRIC, "value": head["value"], "unit": UNIT, "n_gpus": world, "steps": args.steps,
        "warmup": args.warmup, "ms_per_step": head["ms_per_step"], "higher_is_better": True, "scaling": "weak",
        "vs_baseline": None, "dtype": "bf16" if w.dtype == "bf16" else "f32", "data": "synthetic",
        "config": head["config"], "launch": "eager" if args.eager else "cuda_graph", "combine": args.combine,
        "e2e": head["e2e"], "gpu_launches": head["gpu_launches"], "roofline": head["roofline"],
        "cpu_baseline": head["cpu_baseline"], "clocks": head["clocks"], "stages_ms": head["stages_ms"],
        "stages_sum_ms": head["stages_sum_ms"], "grouped_gemm_tflops": head["grouped_gemm_tflops"],
        "grouped_gemm_frac_of_burst": head["grouped_gemm_frac_of_burst"],
        "expert_weight_frac_of_hbm": head["expert_weight_frac_of_hbm"],
    }
    for key in ("expert_weight_gbs", "grouped_gemm_frac_of_sustained", "expert_weight_frac_of_nominal_hbm",
                "layer_roofline_frac"):
        line[key] = head[key]
    if "w8a8" in head:
        line["w8a8"] = head["w8a8"]
    if extras:
        line["workloads"] = extras
    if rank == 0:
        print(json.dumps(line), flush=True)
    if dist is not None:
        dist.destroy_process_group()


def main():
    args = parse_args()
    if args.write_traffic:
        write_traffic(args.write_traffic, args.traffic_kind or args.weights)
        return
    import synth
    w = synth.WORKLOADS[args.workload]
    if args.impl == "reference":
        run_reference(args, w)
    else:
        run_ours(args, w)


if __name__ == "__main__":
    main()
