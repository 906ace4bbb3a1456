#!/usr/bin/env python
"""Benchmark of the MoE FFN layer forward on B300: prints ONE JSON line (rank 0).

    python bench.py [--gpus N] [--steps K] [--warmup W] [--workload NAME] [--impl ours|reference]

A step is one moe_layer_forward over one batch of synthetic input (router ->
grouping -> grouped SwiGLU GEMMs -> combine). Default workload: the
Mixtral-8x7B-shaped prefill layer (T=4096, d=4096, 8 experts, top-2, d_ff=14336).

value        tokens/s with inputs resident in HBM, K steps timed with CUDA events
             (barrier + synchronize on both sides, max over ranks); expert weights
             (2.8 GB) exceed the 126 MB L2, so every step streams them from HBM.
             The K moe_layer_forward calls are captured into one CUDA graph and
             replayed (--eager: K separate calls); each captured call enqueues the
             same kernels as an eager one. Stage times (and the roofline's kernel
             time) come from a second replay of the same K calls with CUDA events
             at the stage boundaries (--eager: from the timed calls themselves).
e2e          the same metric through the same C-ABI call with the activations in
             pinned host memory: each step copies x host->device, runs the layer and
             copies out device->host. Steps with at least 1 MB of activations run their
             copies on their own streams, overlapping the neighbouring steps' layers;
             smaller steps run serially on one stream. Both loops are reported.
roofline     the dominant kernel (the gate/up grouped GEMM), timed by events recorded
             around it on the launching stream, in the staged replay of the K layers.
cpu_baseline the fp64 CPU oracle on a bounded sample of the same workload.
--impl reference  times that oracle alone, step by step, on the host cores.
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


def parse_args():
    ap = argparse.ArgumentParser()
    ap.add_argument("--gpus", type=int, default=1)
    ap.add_argument("--steps", type=int, default=500)
    ap.add_argument("--warmup", type=int, default=10)
    ap.add_argument("--workload", default="mixtral_8x7b")
    ap.add_argument("--impl", choices=["ours", "reference"], default="ours")
    ap.add_argument("--e2e-steps", type=int, default=None,
                    help="end-to-end steps per loop (default: at least 100 and 0.3 s of layers)")
    ap.add_argument("--no-cpu-baseline", action="store_true")
    ap.add_argument("--cpu-sample-tokens", type=int, default=4096)
    ap.add_argument("--weights", choices=["bf16", "fp8"], default="bf16",
                    help="expert weights as stored: bf16, or FP8 E4M3 codes with per-row scales")
    ap.add_argument("--write-traffic", metavar="CSV_DIR", default=None,
                    help="write profiles/traffic.json from ncu CSVs traffic_<workload>.csv in CSV_DIR (see "
                         "write_traffic) and exit")
    ap.add_argument("--eager", action="store_true",
                    help="time K separate launches of the layer instead of one CUDA-graph replay of K layers")
    return ap.parse_args()


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
    weight_bytes: bytes per stored expert weight (2 for bf16, 1 for FP8 codes, whose per-row
    float32 scales are counted too)."""
    rows = kept_pairs + w.n_shared * w.T
    d, F = w.d_model, w.d_ff
    e = 2  # bytes per bf16 activation
    scales = 4.0 if weight_bytes < 2 else 0.0
    return {
        "gateup_flops": 4.0 * d * F * rows,
        "down_flops": 2.0 * d * F * rows,
        "router_flops": 2.0 * w.T * d * w.n_experts,
        "gateup_bytes": groups_touched * 2.0 * F * (d * weight_bytes + scales) + rows * d * e + rows * F * e,
        "down_bytes": groups_touched * 1.0 * d * (F * weight_bytes + scales) + rows * F * e + rows * d * e,
    }


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


GEMM_SOURCES = {"bf16": ("gemm_tc.cu", "gemm_common.cuh", "tc_ptx.cuh"),
                "fp8": ("gemm_fp8w.cu", "gemm_common.cuh", "tc_ptx.cuh")}


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

    (the second layer forward's gate/up and down GEMMs). Each entry records the hash of the GEMM
    source it was measured on; the roofline reports the traffic only while that source is unchanged.
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
        gu, dn = list(per.values())[:2]            # gate/up is launched before down
        key = wl if weights == "bf16" else wl + "+" + weights
        out[key] = {"source_sha256": sha, "kernel": gu["k"][:60],
                    "bytes_per_launch": gu["dram__bytes_read.sum"] + gu["dram__bytes_write.sum"],
                    "read": gu["dram__bytes_read.sum"], "write": gu["dram__bytes_write.sum"],
                    "ns_under_ncu": gu["gpu__time_duration.sum"],
                    "down_bytes_per_launch": dn["dram__bytes_read.sum"] + dn["dram__bytes_write.sum"]}
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


# ----------------------------------------------------------- the CPU oracle

def oracle_sample(w, n_tokens: int, one_token_batches: bool):
    """Returns (callable that runs the oracle once, tokens it covers, description).

    The expert weights are generated on the host and converted to float64 before the
    timing starts; the timed call is the oracle's layer forward alone.
    """
    import numpy as np
    import oracle as O
    import synth

    x64 = synth.as_f64(synth.host_tensor(w, "x"), w.dtype)
    wr64 = synth.as_f64(synth.host_tensor(w, "w_router"), w.dtype)
    bias = synth.router_bias(w.n_experts, w.bias_s)
    rng = np.random.default_rng(0)
    toks = np.sort(rng.choice(w.T, size=min(n_tokens, w.T), replace=False))
    if one_token_batches:
        assert w.capacity_factor <= 0, "a one-token batch changes capacity; use a dropless workload"
        need = set()
        idx, _, _ = O.route(x64[toks], wr64, bias, w.top_k, w.score, w.renormalize)
        need |= set(np.unique(idx).tolist())
    else:
        idx, _, _ = O.route(x64, wr64, bias, w.top_k, w.score, w.renormalize)
        need = set(np.unique(idx[toks]).tolist())
    need |= set(range(w.n_experts, w.n_experts + w.n_shared))
    cache = {g: tuple(synth.as_f64(a, w.dtype) for a in synth.host_expert(w, g)) for g in sorted(need)}
    experts = cache.__getitem__
    kw = dict(top_k=w.top_k, score=w.score, renormalize=w.renormalize, capacity_factor=w.capacity_factor,
              n_shared=w.n_shared)
    if one_token_batches:
        state = {"i": 0}

        def run():
            t = toks[state["i"] % len(toks)]
            state["i"] += 1
            O.layer_forward(x64[t:t + 1], wr64, bias, experts, **kw)
            return 1
        desc = f"{w.name}: one token per step (a 1-token dropless batch), tokens drawn from the {w.T}-token batch"
    else:
        def run():
            O.layer_forward(x64, wr64, bias, experts, tokens=toks, **kw)
            return len(toks)
        desc = (f"{w.name}: routing and grouping of all {w.T} tokens, expert MLPs and combine for "
                f"{len(toks)} sampled tokens")
    return run, desc


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
    world, rank, _ = dist_env()
    if rank != 0:
        return
    run, desc = oracle_sample(w, max(args.steps + args.warmup, 1), one_token_batches=True)
    for _ in range(args.warmup):
        run()
    t0 = time.perf_counter()
    n = 0
    for _ in range(args.steps):
        n += run()
    dt = time.perf_counter() - t0
    value = n / dt
    line = {
        "impl": "reference", "metric": METRIC, "value": value, "unit": UNIT, "n_gpus": args.gpus,
        "steps": args.steps, "warmup": args.warmup, "ms_per_step": 1e3 * dt / max(args.steps, 1),
        "higher_is_better": True, "scaling": "weak", "vs_baseline": None, "dtype": "f64", "data": "synthetic",
        "config": {"workload": w.name, "T": w.T, "d_model": w.d_model, "n_experts": w.n_experts,
                   "top_k": w.top_k, "d_ff": w.d_ff},
        "cpu_baseline": {"value": value, "unit": UNIT, "cores": cpu_threads(), "kind": "oracle", "sample": desc},
        "e2e": {"value": value, "unit": UNIT, "h2d_bytes_per_step": 0, "d2h_bytes_per_step": 0},
    }
    print(json.dumps(line), flush=True)


# ------------------------------------------------------------- our layer

def run_ours(args, w):
    import numpy as np
    import torch
    import synth
    import sparse_expert_mlp_router_b300 as moe

    world, rank, local = dist_env()
    torch.cuda.set_device(local)
    dist = None
    if world > 1:
        import torch.distributed as dist
        dist.init_process_group("nccl", device_id=torch.device("cuda", local))

    def barrier():
        if dist is not None:
            dist.barrier()
        torch.cuda.synchronize()

    cfg = moe.make_config(T=w.T, d_model=w.d_model, n_experts=w.n_experts, top_k=w.top_k, d_ff=w.d_ff,
                          n_shared=w.n_shared, score=w.score, renormalize=w.renormalize,
                          capacity_factor=w.capacity_factor, dtype=w.dtype)
    dev = synth.device_inputs(w)
    fp8 = args.weights == "fp8"
    if fp8:
        # FP8 codes and per-row scales made on the device by the library's quantiser; the bf16
        # copies are freed before any timing
        for name in ("w_gate", "w_up", "w_down"):
            dev[name + "_q"], dev[name + "_s"] = moe.moe_quantize_fp8_rows(dev[name])
            del dev[name]
        torch.cuda.synchronize()
        torch.cuda.empty_cache()
        wargs = (dev["w_gate_q"], dev["w_gate_s"], dev["w_up_q"], dev["w_up_s"], dev["w_down_q"], dev["w_down_s"])
        forward, forward_timed = moe.moe_layer_forward_fp8, moe.moe_layer_forward_fp8_timed
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
        raise RuntimeError(f"device status {moe.status_string(status)}")
    cap = moe.moe_capacity(cfg)
    c = counts.cpu().numpy()
    kept = int(np.minimum(c, cap).sum())
    touched = int((np.minimum(c, cap) > 0).sum()) + w.n_shared
    work = algorithmic(w, kept, touched, 1.0 if fp8 else 2.0)

    K, W = args.steps, args.warmup
    evs = [[torch.cuda.Event(enable_timing=True) for _ in range(6)] for _ in range(K)]
    for row in evs:            # create every event before any capture
        for e in row:
            e.record()
    for i in range(W):
        forward_timed(*args_fwd, evs[i % K])
    barrier()
    # Graph mode: the timed region replays K plain moe_layer_forward calls; the stage times come
    # from a second replay of the same K calls with CUDA events recorded at the stage boundaries
    # (six event records a layer cost the decode-shaped layer about 8 %). Eager mode (--eager,
    # for profilers): K calls with the stage events, timed as they run.
    graph = graph_staged = None
    if not args.eager:
        graph = torch.cuda.CUDAGraph()
        with torch.cuda.graph(graph):
            for i in range(K):
                forward(*args_fwd)
        graph_staged = torch.cuda.CUDAGraph()
        with torch.cuda.graph(graph_staged):
            for i in range(K):
                forward_timed(*args_fwd, evs[i])
        graph.replay()         # one untimed replay of each
        graph_staged.replay()
        barrier()
    props = torch.cuda.get_device_properties(local)
    try:
        gpu_id = "%08X:%02X:%02X.0" % (props.pci_domain_id, props.pci_bus_id, props.pci_device_id)
    except AttributeError:
        gpu_id = str(local)
    sampler = ClockSampler(gpu_id)
    sampler.start()
    barrier()
    t_start = torch.cuda.Event(enable_timing=True)
    t_end = torch.cuda.Event(enable_timing=True)
    t_start.record()
    if graph is not None:
        graph.replay()
    else:
        for i in range(K):
            forward_timed(*args_fwd, evs[i])
    t_end.record()
    barrier()
    if graph_staged is not None:
        graph_staged.replay()
        barrier()
    clocks = sampler.stop()
    elapsed_ms = t_start.elapsed_time(t_end)
    stage = np.array([[e[j].elapsed_time(e[j + 1]) for j in range(5)] for e in evs])   # [K, 5] ms
    status = moe.moe_get_device_error(ws)
    if status != moe.MOE_OK:
        raise RuntimeError(f"device status after timing: {moe.status_string(status)}")
    max_ms = max_over_ranks(elapsed_ms, dist)
    value = whole_job_rate(w.T, K, world, max_ms)

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
        raise RuntimeError("device status after e2e timing")

    # roofline of the dominant kernel: the gate/up grouped GEMM (stage 2 -> 3). A tensor-bound
    # kernel timed inside a long run of back-to-back layers (>= 1 s, where the GPU settles at
    # its power limit) is compared with the sustained bf16 rate, else with the burst rate; the
    # fraction of the burst rate is reported as well.
    peaks, peak_src = load_peaks()
    gemm_ms = float(stage[:, 2].mean())
    t_tensor = work["gateup_flops"] / (peaks["bf16_tflops"] * 1e12)
    t_bytes = work["gateup_bytes"] / (peaks["hbm_gbs"] * 1e9)
    long_run = max_ms >= 1000.0
    if t_tensor >= t_bytes:
        achieved = work["gateup_flops"] / (gemm_ms / 1e3) / 1e12
        peak = peaks["bf16_tflops_sustained"] if long_run else peaks["bf16_tflops"]
        roof = {"bound": "tensor", "achieved": achieved, "peak": peak, "unit": "TFLOP/s",
                "frac_of_burst": achieved / peaks["bf16_tflops"]}
    else:
        achieved = work["gateup_bytes"] / (gemm_ms / 1e3) / 1e9
        roof = {"bound": "hbm", "achieved": achieved, "peak": peaks["hbm_gbs"], "unit": "GB/s"}
    roof["frac"] = roof["achieved"] / roof["peak"]
    roof["traffic"] = measured_traffic(w.name, args.weights)
    roof["kernel"] = ("grouped_gemm_fp8w_kernel<gate/up, FP8 weights, SwiGLU epilogue> (tcgen05)" if fp8 else
                      "grouped_gemm_kernel<gate/up, SwiGLU epilogue> (tcgen05)")
    roof["peak_source"] = (f"{peak_src} copy bandwidth" if roof["bound"] == "hbm" else
                           f"{peak_src} sustained (timed region {max_ms / 1e3:.1f} s)" if long_run else
                           f"{peak_src} burst")
    roof["ms_per_launch"] = gemm_ms

    stages_ms = dict(zip(["router", "grouping", "gemm_gate_up", "gemm_down", "combine"],
                         [float(v) for v in stage.mean(axis=0)]))
    gemm_tflops = (work["gateup_flops"] + work["down_flops"]) / ((stage[:, 2] + stage[:, 3]).mean() / 1e3) / 1e12

    cpu = None
    if rank == 0 and world == 1 and not args.no_cpu_baseline:
        run, desc = oracle_sample(w, args.cpu_sample_tokens, one_token_batches=False)
        t0 = time.perf_counter()
        n = run()
        dtc = time.perf_counter() - t0
        cpu = {"value": n / dtc, "unit": UNIT, "cores": cpu_threads(), "kind": "oracle", "sample": desc,
               "seconds": dtc}

    line = {
        "metric": METRIC, "value": value, "unit": UNIT, "n_gpus": world, "steps": K, "warmup": W,
        "ms_per_step": max_ms / K, "higher_is_better": True, "scaling": "weak", "vs_baseline": None,
        "dtype": "bf16" if w.dtype == "bf16" else "f32", "data": "synthetic",
        "config": {"workload": w.name, "T": w.T, "d_model": w.d_model, "n_experts": w.n_experts,
                   "n_shared": w.n_shared, "top_k": w.top_k, "d_ff": w.d_ff, "score": w.score,
                   "capacity_factor": w.capacity_factor, "kept_pairs": kept, "groups_touched": touched,
                   "l2": "inputs larger than L2: %.2f GB of expert weights streamed per step"
                         % (touched * 3.0 * w.d_model * w.d_ff * 2 / 1e9),
                   "parallelism": "replicas" if world > 1 else "single GPU",
                   "launch": "eager" if args.eager else "cuda_graph",
                   "weights": "fp8 e4m3, per-row float32 scales" if fp8 else w.dtype},
        "e2e": {"value": e2e_value, "unit": UNIT, "h2d_bytes_per_step": int(x_host.numel() * x_host.element_size()),
                "d2h_bytes_per_step": int(out.numel() * out.element_size()), "steps": K2,
                "copies": ("own streams, overlapping the neighbouring steps' layers (double-buffered)"
                           if overlapped else "serial, on the layer's stream (activations under %d bytes)"
                           % OVERLAP_MIN_BYTES),
                "serial_value": whole_job_rate(w.T, K2, world, serial_ms),
                "overlapped_value": whole_job_rate(w.T, K2, world, overlap_ms)},
        "gpu_launches": K * moe.moe_layer_launch_count(cfg),
        "roofline": roof,
        "cpu_baseline": cpu,
        "clocks": clocks,
        "stages_ms": stages_ms,
        "grouped_gemm_tflops": gemm_tflops,
    }
    if rank == 0:
        print(json.dumps(line), flush=True)
    if dist is not None:
        dist.destroy_process_group()


def main():
    args = parse_args()
    if args.write_traffic:
        write_traffic(args.write_traffic, args.weights)
        return
    import synth
    w = synth.WORKLOADS[args.workload]
    if args.impl == "reference":
        run_reference(args, w)
    else:
        run_ours(args, w)


if __name__ == "__main__":
    main()
