#!/usr/bin/env python
"""Benchmark of the fused small-M W8A8 FP8 block-scale linear on GB300.

Metric: us/call and achieved HBM GB/s (fraction of the bytes roofline) of the
fused quant + GEMM, M = 1..32.  Default workload: the M sweep
{1,3,4,8,9,16,17,24,32} at N = 5120, K = 4096 (the token counts an EAGLE
verify pass sends through the in_proj_qkvz projection on the page "[AMD]
Small-M FP8 block-scale GEMM with fused activation quant for gfx950
(Qwen3.5)", "Modifications" / "Kernel microbenchmarks").

One step = one pass over one batch: for every M of the sweep, one fused call
on each of 24 independently seeded weight copies (216 calls; the 24 copies
hold 503 MB, far above the 129 MB L2, so every weight byte comes from HBM),
replayed as one CUDA graph.  Value = algorithmic bytes / time, summed over
ranks, in GB/s; us_per_call = time / calls.

Algorithmic bytes per call: N*K (fp8 weight) + (N/128)(K/128)*4 (fp32 block
scales; *1 for e8m0) + 2*M*K (bf16 x) + 2*M*N (bf16 y).

  python bench.py [--gpus N] [--steps K] [--warmup W] [--impl reference]
                  [--workload msweep|smallest|shapes|ue8m0|chain4|chain16|chain32]

The default run also times every other workload (key "workloads": smallest,
shapes, ue8m0, chain4/16/32) and the M sweep per M.

--impl reference times the CPU oracle (the plain restatement of the method the
tests compare against) on this host's cores: each step computes one whole
call of the workload (its distinct calls in turn), so its GB/s is that of
whole weights.  Under
torchrun (N > 1) every rank runs its own replica on its own GPU (each rank
stands for one tensor-parallel shard: the pages' shapes are per-rank shapes),
the timed region is bracketed by barriers, and the slowest rank's time counts.
"""

from __future__ import annotations

import argparse
import hashlib
import json
import re
import os
import statistics
import subprocess
import sys
import time

ROOT = os.path.dirname(os.path.abspath(__file__))
if ROOT not in sys.path:
    sys.path.insert(0, ROOT)

METRIC = "µs/call and achieved HBM GB/s (frac of roofline), fused quant+GEMM, M=1..32"
M_SWEEP = [1, 3, 4, 8, 9, 16, 17, 24, 32]
COPIES = 24
KERNEL_SOURCES = ["fp8_block_scale_x128_gb300/csrc/gemm_fused.cu",
                  "fp8_block_scale_x128_gb300/csrc/ptx.cuh",
                  "fp8_block_scale_x128_gb300/csrc/internal.cuh"]
DRAM_PROFILE = os.path.join(ROOT, "profiles", "fused_quant_gemm_5120x4096_msweep_dram.md")


def algorithmic_bytes(M: int, N: int, K: int, kind: int) -> int:
    scale = 4 if kind == 0 else 1
    return N * K + (N // 128) * (K // 128) * scale + 2 * M * K + 2 * M * N


def workload_plan(name: str):
    """(description, calls of one step as (M, N, K, kind, weight_id))."""
    rot = range(COPIES)
    if name == "msweep":
        return ("M sweep {1,3,4,8,9,16,17,24,32} at N=5120 K=4096, fp32 block scales, "
                "24 rotated weight copies",
                [(M, 5120, 4096, 0, c) for M in M_SWEEP for c in rot])
    if name == "smallest":
        return ("M=1 at N=4096 K=2048, fp32 block scales, 24 rotated weight copies",
                [(1, 4096, 2048, 0, c) for c in rot])
    if name == "shapes":
        return ("(N,K) in {(5120,4096),(4608,4096),(4096,2048)} x M in {1,4,8,16,32}, fp32 block "
                "scales, 24 rotated weight copies per shape",
                [(M, N, K, 0, c) for (N, K) in [(5120, 4096), (4608, 4096), (4096, 2048)]
                 for M in (1, 4, 8, 16, 32) for c in rot])
    if name == "ue8m0":
        return ("ue8m0 scales, (N,K) in {(7168,2048),(1536,7168),(4096,4096)} x M in {1,16,32}, "
                "24 rotated weight copies per shape",
                [(M, N, K, 1, c) for (N, K) in [(7168, 2048), (1536, 7168), (4096, 4096)]
                 for M in (1, 16, 32) for c in rot])
    if name.startswith("chain"):
        M = int(name[5:] or 16)
        return (f"decode chain: 60 layers x (5120x4096, 4608x4096, 4096x2048) at M={M}, "
                "distinct weights per linear (2.9 GB), fresh x per linear",
                [(M, N, K, 0, layer) for layer in range(60)
                 for (N, K) in [(5120, 4096), (4608, 4096), (4096, 2048)]])
    raise SystemExit(f"unknown workload {name}")


def distinct_calls(calls):
    seen, out = set(), []
    for (M, N, K, kind, _w) in calls:
        if (M, N, K, kind) not in seen:
            seen.add((M, N, K, kind))
            out.append((M, N, K, kind))
    return out


def _code_only(text: str) -> str:
    """The source without its comments, whitespace runs collapsed (the kernel
    sources hold no comment markers inside string literals)."""
    text = re.sub(r"/\*.*?\*/", " ", text, flags=re.S)
    text = re.sub(r"//[^\n]*", " ", text)
    return " ".join(text.split())


def kernel_source_hash() -> str:
    """Identity of the fused kernel's code: a hash of its sources without
    comments, so that the recorded DRAM counters stay attached to the code they
    were taken on through comment-only edits, and to nothing else."""
    h = hashlib.sha256()
    for rel in KERNEL_SOURCES:
        with open(os.path.join(ROOT, rel), encoding="utf-8") as f:
            h.update(_code_only(f.read()).encode())
    return h.hexdigest()[:16]


def bench_config(desc: str, calls) -> dict:
    """The workload description both arms report."""
    weight_bytes = sum(N * K for (N, K, _k, _w) in {c[1:] for c in calls})
    return {"workload": desc, "calls_per_step": len(calls),
            "l2": "inputs larger than L2 (rotated weight copies, "
                  f"{weight_bytes // 10**6} MB of distinct weights per step vs 129 MB)",
            "parallelism": "replicas"}


def dram_traffic_per_launch(workload: str):
    """Per-launch DRAM bytes of the fused kernel from the committed ncu summary,
    or None when the kernel source has changed since the counters were taken."""
    try:
        with open(DRAM_PROFILE) as f:
            # "- key: value" lines of the summary
            prof = dict(m.groups() for m in re.finditer(r"^- (\w+): (\S+)\s*$", f.read(), re.M))
        if "bytes_per_launch_mean" in prof:
            prof["bytes_per_launch_mean"] = float(prof["bytes_per_launch_mean"])
    except (OSError, ValueError):
        return None
    if prof.get("kernel_src_sha256") != kernel_source_hash() or workload != "msweep":
        return None
    return prof.get("bytes_per_launch_mean")


class ClockSampler:
    """nvidia-smi clock / throttle samples while the timed region runs."""

    QUERY = ("index,clocks.sm,clocks.max.sm,power.draw,clocks_event_reasons.active,"
             "clocks_event_reasons.hw_slowdown,clocks_event_reasons.hw_thermal_slowdown,"
             "clocks_event_reasons.sw_thermal_slowdown,clocks_event_reasons.sw_power_cap")

    def __init__(self, gpu_index: int):
        self.gpu = gpu_index
        self.proc = None
        self.lines = []

    def __enter__(self):
        try:
            self.proc = subprocess.Popen(
                ["nvidia-smi", f"--id={self.gpu}", f"--query-gpu={self.QUERY}",
                 "--format=csv,noheader,nounits", "-lms", "100"],
                stdout=subprocess.PIPE, stderr=subprocess.DEVNULL, text=True)
        except OSError:
            self.proc = None
        time.sleep(0.2)
        return self

    def __exit__(self, *exc):
        if self.proc is not None:
            self.proc.terminate()
            try:
                out, _ = self.proc.communicate(timeout=5)
            except subprocess.TimeoutExpired:
                self.proc.kill()
                out, _ = self.proc.communicate()
            self.lines = [ln for ln in out.splitlines() if ln.strip()]
        return False

    def summary(self):
        sm, mx, reasons = [], None, set()
        names = ["hw_slowdown", "hw_thermal_slowdown", "sw_thermal_slowdown", "sw_power_cap"]
        for ln in self.lines:
            f = [t.strip() for t in ln.split(",")]
            if len(f) < 9:
                continue
            try:
                sm.append(float(f[1]))
                mx = float(f[2])
            except ValueError:
                continue
            for nm, v in zip(names, f[5:9]):
                if v.lower() == "active":
                    reasons.add(nm)
        if not sm:
            return {"sm_mhz": None, "sm_max_mhz": mx, "reasons": ["no samples"], "samples": 0}
        return {"sm_mhz": statistics.median(sm), "sm_max_mhz": mx, "reasons": sorted(reasons),
                "samples": len(sm)}


def dist_setup():
    world = int(os.environ.get("WORLD_SIZE", "1"))
    rank = int(os.environ.get("RANK", "0"))
    local = int(os.environ.get("LOCAL_RANK", "0"))
    if world > 1:
        import torch
        import torch.distributed as dist
        dist.init_process_group(backend="nccl" if torch.cuda.is_available() else "gloo")
    return world, rank, local


def barrier(world):
    if world > 1:
        import torch.distributed as dist
        dist.barrier()


def max_over_ranks(value: float, world: int, device) -> float:
    """Largest value over the ranks (the slowest rank's time)."""
    if world == 1:
        return value
    import torch
    import torch.distributed as dist
    t = torch.tensor([value], dtype=torch.float64, device=device)
    dist.all_reduce(t, op=dist.ReduceOp.MAX)
    return float(t.item())


def host_cores() -> int:
    try:
        return len(os.sched_getaffinity(0))
    except AttributeError:
        return os.cpu_count() or 1


# ---------------------------------------------------------------------------
# CPU oracle (reference arm and cpu_baseline)
# ---------------------------------------------------------------------------

class OracleSample:
    """The CPU oracle (1x128 quant + fp64 block-scale GEMM) on 128-row weight
    slices of the workload's distinct shapes; inputs from synth."""

    def __init__(self, calls):
        import oracle
        import synth
        oracle.build()
        self.oracle = oracle
        self.cores = host_cores()
        self.calls = distinct_calls(calls)
        self.w = {}
        self.x = {}
        for (M, N, K, kind) in self.calls:
            if (N, K, kind) not in self.w:
                self.w[(N, K, kind)] = oracle.quant_weight_128x128(
                    synth.w_f32(N, K, seed=N + K), kind)
            self.x[(M, K)] = synth.x_bf16(M, K, seed=M + K)

    def whole_call(self, i: int) -> int:
        """The i-th distinct call (cyclically) on its whole weight; returns bytes."""
        M, N, K, kind = self.calls[i % len(self.calls)]
        wq, ws = self.w[(N, K, kind)]
        self.oracle.linear(self.x[(M, K)], wq, ws, kind, nthreads=self.cores)
        return algorithmic_bytes(M, N, K, kind)

    def step(self, i: int, n_tiles: int = 1) -> int:
        """Every distinct call on n_tiles consecutive 128-row slices; returns bytes."""
        nbytes = 0
        for (M, N, K, kind) in self.calls:
            wq, ws = self.w[(N, K, kind)]
            nt = (i * n_tiles) % (N // 128)
            rows = min(n_tiles, N // 128 - nt) * 128
            self.oracle.linear(self.x[(M, K)], wq[nt * 128:nt * 128 + rows],
                               ws[nt:nt + rows // 128], kind, nthreads=self.cores)
            nbytes += algorithmic_bytes(M, rows, K, kind)
        return nbytes

    def sample_desc(self, n_tiles: int) -> str:
        return (f"per step: each of the {len(self.calls)} distinct calls "
                f"{[c[:3] for c in self.calls]} on {n_tiles} x 128 weight rows; oracle 1x128 quant "
                f"+ fp64 GEMM on {self.cores} threads")


def run_reference(args):
    world = int(os.environ.get("WORLD_SIZE", "1"))
    rank = int(os.environ.get("RANK", "0"))
    if world > 1 and rank != 0:
        return 0
    desc, calls = workload_plan(args.workload)
    smp = OracleSample(calls)
    # one step = one whole call of the workload (its distinct calls in turn),
    # so the GB/s is that of whole weights, like the main arm's cpu_baseline
    for i in range(args.warmup):
        smp.whole_call(i)
    nbytes = 0
    t0 = time.perf_counter()
    for i in range(args.steps):
        nbytes += smp.whole_call(args.warmup + i)
    el = time.perf_counter() - t0
    value = nbytes / el / 1e9
    config = bench_config(desc, calls)
    config["calls_per_step"] = 1
    config["reference_step"] = (f"one whole call per step: the {len(smp.calls)} distinct calls "
                                f"{[c[:3] for c in smp.calls]} in turn, each on its whole weight")
    line = {
        "impl": "reference", "metric": METRIC, "value": value, "unit": "GB/s", "n_gpus": world,
        "steps": args.steps, "warmup": args.warmup, "ms_per_step": el * 1e3 / args.steps,
        "higher_is_better": True, "scaling": "weak", "vs_baseline": None, "dtype": "f64",
        "data": "synthetic", "config": config,
        "cpu_baseline": {"value": value, "unit": "GB/s", "cores": smp.cores, "kind": "oracle",
                         "sample": config["reference_step"] + f"; oracle 1x128 quant + fp64 "
                                   f"GEMM on {smp.cores} threads"},
        "e2e": {"value": value, "unit": "GB/s", "h2d_bytes_per_step": 0, "d2h_bytes_per_step": 0},
    }
    print(json.dumps(line), flush=True)
    return 0


def cpu_baseline(calls, budget_s: float):
    """Oracle throughput over whole weights of the distinct shapes, bounded."""
    smp = OracleSample(calls)
    big = max(N // 128 for (_M, N, _K, _k) in smp.calls)
    nbytes, i = 0, 0
    t0 = time.perf_counter()
    while True:
        nbytes += smp.step(i, n_tiles=big)
        i += 1
        el = time.perf_counter() - t0
        if el >= budget_s:
            break
    return {"value": nbytes / el / 1e9, "unit": "GB/s", "cores": smp.cores, "kind": "oracle",
            "sample": f"{i} pass(es), each: every distinct call of the step on its whole weight; "
                      f"oracle 1x128 quant + fp64 GEMM on {smp.cores} threads ({el:.1f} s)"}


# ---------------------------------------------------------------------------
# GPU leg
# ---------------------------------------------------------------------------

class Step:
    """Packed weights, activations and the CUDA graph of one step."""

    def __init__(self, fb, torch, calls, dev, stream, io: bool = False, graph: bool = True,
                 pdl: bool = True, two_launch: bool = False):
        import synth
        self.calls = calls
        self.packs = {}
        for (M, N, K, kind, wid) in calls:
            key = (N, K, kind, wid)
            if key in self.packs:
                continue
            w = synth.w_f32_torch(N, K, seed=104729 * wid + N + K, device=dev)
            wq, ws = fb.fp8bs_quant_weight(w, kind)
            self.packs[key] = fb.fp8bs_prepack_weight(wq, ws, kind)
            del w, wq, ws
        max_n = max(c[1] for c in calls)
        max_k = max(c[2] for c in calls)
        self.workspace = fb.new_workspace(max_n, max_k, dev)
        # one x per (M, K) and one y per (M, N); with host I/O every call has its
        # own x and y, views of one device buffer each, so a step moves all of
        # its inputs in one host->device copy and all of its outputs in one
        # device->host copy
        self.x = {}
        self.y = {}
        if io:
            x_sizes = [M * K for (M, N, K, _k, _w) in calls]
            y_sizes = [M * N for (M, N, K, _k, _w) in calls]
            self.x_all = torch.empty(sum(x_sizes), dtype=torch.bfloat16, device=dev)
            self.y_all = torch.empty(sum(y_sizes), dtype=torch.bfloat16, device=dev)
            xo = yo = 0
            for i, (M, N, K, kind, wid) in enumerate(calls):
                self.x[i] = self.x_all[xo:xo + M * K].view(M, K)
                self.x[i].copy_(synth.x_bf16_torch(M, K, seed=31 * i + M, device=dev))
                self.y[i] = self.y_all[yo:yo + M * N].view(M, N)
                xo += M * K
                yo += M * N
            self.x_host = torch.empty(self.x_all.numel(), dtype=torch.bfloat16).pin_memory()
            self.x_host.copy_(self.x_all.cpu())
            self.y_host = torch.empty(self.y_all.numel(), dtype=torch.bfloat16).pin_memory()
        else:
            for i, (M, N, K, kind, wid) in enumerate(calls):
                if (M, K) not in self.x:
                    self.x[(M, K)] = synth.x_bf16_torch(M, K, seed=31 * i + M, device=dev)
                if (M, N) not in self.y:
                    self.y[(M, N)] = torch.empty((M, N), dtype=torch.bfloat16, device=dev)
        self.io = io
        self.pdl = pdl
        # the two-launch path: fp8bs_quant, then fp8bs_gemm_prequant on its output
        self.two_launch = two_launch
        if two_launch:
            self.xq = {(M, K): torch.empty((M, K), dtype=torch.uint8, device=dev)
                       for (M, N, K, _k, _w) in calls}
            self.xs = {(M, K, kind): torch.empty((M, K // 128), device=dev,
                                                 dtype=torch.uint8 if kind == 1 else torch.float32)
                       for (M, N, K, kind, _w) in calls}
        self.stream = stream
        self.fb = fb
        # weights, x and the workspace's initial zeros were written on the current
        # stream; `stream` does not wait for it, so finish them before any call
        torch.cuda.synchronize()
        with torch.cuda.stream(stream):
            self.enqueue()  # eager pass: module load, kernel attributes
        stream.synchronize()
        self.torch = torch
        self.graph = None
        if graph:
            self.graph = torch.cuda.CUDAGraph()
            with torch.cuda.graph(self.graph, stream=stream):
                self.enqueue()
        torch.cuda.synchronize()

    def replay(self):
        if self.graph is not None:
            self.graph.replay()
        else:
            with self.torch.cuda.stream(self.stream):
                self.enqueue()

    def enqueue(self):
        if self.io:
            self.x_all.copy_(self.x_host, non_blocking=True)
        for i, (M, N, K, kind, wid) in enumerate(self.calls):
            x = self.x[i] if self.io else self.x[(M, K)]
            y = self.y[i] if self.io else self.y[(M, N)]
            if self.two_launch:
                xq, xs = self.xq[(M, K)], self.xs[(M, K, kind)]
                self.fb.fp8bs_quant(x, kind, xq=xq, xs=xs, stream=self.stream)
                self.fb.fp8bs_gemm_prequant(xq, xs, self.packs[(N, K, kind, wid)], N, K, kind, y=y,
                                            workspace=self.workspace, pdl=self.pdl, stream=self.stream)
            else:
                self.fb.fp8bs_gemm_fused(x, self.packs[(N, K, kind, wid)], N, K, kind, y=y,
                                         workspace=self.workspace, pdl=self.pdl, stream=self.stream)
        if self.io:
            self.y_host.copy_(self.y_all, non_blocking=True)


def time_steps(torch, step: Step, steps: int, warmup: int, world: int, dev) -> float:
    for _ in range(warmup):
        step.replay()
    torch.cuda.synchronize()
    barrier(world)
    torch.cuda.synchronize()
    e0 = torch.cuda.Event(enable_timing=True)
    e1 = torch.cuda.Event(enable_timing=True)
    with torch.cuda.stream(step.stream):
        e0.record(step.stream)
        for _ in range(steps):
            step.replay()
        e1.record(step.stream)
    torch.cuda.synchronize()
    barrier(world)
    return max_over_ranks(e0.elapsed_time(e1), world, dev)


M_ABOVE_32 = [33, 48, 64]
OTHER_WORKLOADS = ["smallest", "shapes", "ue8m0", "chain4", "chain16", "chain32"]


def workloads_table(fb, torch, dev, stream, pdl, peak: float, target_s: float = 0.25):
    """us/call, GB/s and fraction of the peak of every other workload of the
    benchmark (graph replay, the same timing rules as the M sweep)."""
    out = {}
    for name in OTHER_WORKLOADS:
        desc, calls = workload_plan(name)
        step_bytes = sum(algorithmic_bytes(M, N, K, kind) for (M, N, K, kind, _) in calls)
        progress(f"workload {name}")
        st = Step(fb, torch, calls, dev, stream, pdl=pdl)
        probe = time_steps(torch, st, 3, 3, 1, dev) / 3
        reps = max(5, min(500, int(target_s * 1e3 / max(probe, 1e-3))))
        ms = time_steps(torch, st, reps, 3, 1, dev)
        rc = fb.fp8bs_check_error(st.workspace, stream)
        if rc != 0:
            raise SystemExit(f"workload {name}: device error {fb.fp8bs_status_string(rc)}")
        gbps = step_bytes * reps / (ms / 1e3) / 1e9
        out[name] = {"workload": desc, "calls_per_step": len(calls), "steps": reps,
                     "us_per_call": round(ms * 1e3 / (reps * len(calls)), 3),
                     "GBps": round(gbps, 1), "frac": round(gbps / peak, 4)}
        del st
        torch.cuda.empty_cache()
    return out


def per_m_table(fb, torch, dev, stream, pdl, two_launch=False, ms=None):
    """us/call and GB/s per M at N=5120 K=4096 (graph of 24 rotated calls);
    two_launch: fp8bs_quant + fp8bs_gemm_prequant per call instead."""
    out = {}
    for M in (M_SWEEP if ms is None else ms):
        st = Step(fb, torch, [(M, 5120, 4096, 0, c) for c in range(COPIES)], dev, stream, pdl=pdl,
                  two_launch=two_launch)
        progress(f"per-M step M={M}")
        reps = 50
        ms = time_steps(torch, st, reps, 5, 1, dev)
        rc = fb.fp8bs_check_error(st.workspace, stream)
        if rc != 0:
            raise SystemExit(f"per-M step M={M}: device error {fb.fp8bs_status_string(rc)}")
        us = ms * 1e3 / (reps * COPIES)
        out[str(M)] = {"us": round(us, 3),
                       "GBps": round(algorithmic_bytes(M, 5120, 4096, 0) / us / 1e3, 1)}
        del st
    torch.cuda.empty_cache()
    return out


PRODUCER_DECODE = [(1, 7168), (4, 7168), (16, 7168), (32, 7168), (32, 4096), (32, 2048)]
PRODUCER_LARGE = (16384, 7168)


def producer_bytes(M: int, K: int, kind: int) -> int:
    """Algorithmic bytes of one RMSNorm + quant call: x and gamma read, codes
    and scales written (the optional bf16 y is not requested when timed)."""
    return 2 * M * K + 2 * K + M * K + (M * K // 128) * (1 if kind == 1 else 4)


def graph_us_per_call(torch, stream, fn, n_calls: int, reps: int, warm: int = 5) -> float:
    """Capture n_calls of fn(i) in one CUDA graph; µs per call over reps replays."""
    torch.cuda.synchronize()
    g = torch.cuda.CUDAGraph()
    with torch.cuda.graph(g, stream=stream):
        for i in range(n_calls):
            fn(i)
    for _ in range(warm):
        g.replay()
    torch.cuda.synchronize()
    e0 = torch.cuda.Event(enable_timing=True)
    e1 = torch.cuda.Event(enable_timing=True)
    with torch.cuda.stream(stream):
        e0.record(stream)
        for _ in range(reps):
            g.replay()
        e1.record(stream)
    torch.cuda.synchronize()
    del g
    return e0.elapsed_time(e1) * 1e3 / (reps * n_calls)


def producer_table(fb, torch, dev, stream, peak: float):
    """The fused RMSNorm + 1x128 quant producer (ue8m0 scales, as the page's
    producer emits).  First, for the roofline, launches of 16384 x 7168 rows
    over 2 rotated inputs (470 MB of x, larger than L2): 4 per graph, 5 warm-up
    and 20 timed replays.  Then µs/call at decode sizes (rows L2-resident, 24
    rotated inputs per graph, 50 replays)."""
    import synth
    kind = fb.FP8BS_SCALE_UE8M0
    out = {"kind": "ue8m0", "eps": 1e-6}
    M, K = PRODUCER_LARGE
    g = synth.x_bf16_torch(1, K, seed=901, device=dev)[0].abs() + 0.5
    xs_in = [synth.x_bf16_torch(M, K, seed=920 + c, device=dev) for c in range(2)]
    xq = torch.empty((M, K), dtype=torch.uint8, device=dev)
    xsc = torch.empty((M, K // 128), dtype=torch.uint8, device=dev)
    us = graph_us_per_call(torch, stream, lambda i: fb.fp8bs_rmsnorm_quant(
        xs_in[i % 2], g, 1e-6, kind, xq=xq, xs=xsc), 4, 20)
    nbytes = producer_bytes(M, K, 1)
    gbps = nbytes / us / 1e3
    out["large"] = {"M": M, "K": K, "us": round(us, 2), "bytes": nbytes, "GBps": round(gbps, 1),
                    "peak": peak, "frac": round(gbps / peak, 3),
                    "kernel": "rmsnorm_quant_kernel", "bound": "hbm"}
    del xs_in, xq, xsc
    torch.cuda.empty_cache()
    out["decode_us"] = {}
    for (M, K) in PRODUCER_DECODE:
        g = synth.x_bf16_torch(1, K, seed=900, device=dev)[0].abs() + 0.5
        xs_in = [synth.x_bf16_torch(M, K, seed=910 + c, device=dev) for c in range(COPIES)]
        xq = torch.empty((M, K), dtype=torch.uint8, device=dev)
        xsc = torch.empty((M, K // 128), dtype=torch.uint8, device=dev)
        us = graph_us_per_call(torch, stream, lambda i: fb.fp8bs_rmsnorm_quant(
            xs_in[i], g, 1e-6, kind, xq=xq, xs=xsc), COPIES, 50)
        out["decode_us"][f"M={M},K={K}"] = round(us, 3)
        del xs_in
    return out


MOE_E, MOE_H, MOE_S = 513, 4096, 11
MOE_CONFIGS = [("TP4", 256, [1, 4, 8, 16, 20]), ("TP8", 128, [1, 16, 48])]


def moe_table(fb, torch, dev, stream, peak: float):
    """The small-M FP8 block-scale MoE layer at Qwen3.5-397B sizes (513 experts,
    11 slots per token, hidden 4096; intermediate 256 at TP4, 128 at TP8).
    Weights: one layer, 1.6 GB (TP4) / 0.8 GB (TP8), larger than L2.  Each
    graph holds 24 calls with 24 different routings, so the active experts
    change from call to call.  Algorithmic bytes of a call: the w13 / w2 bytes
    and block scales of its distinct active experts, plus x, y, ids and
    weights."""
    import synth
    out = {"E": MOE_E, "H": MOE_H, "S": MOE_S, "configs": {}}
    for name, I, ms in MOE_CONFIGS:
        w = synth.w_f32_torch(MOE_E * 2 * I, MOE_H, seed=950, device=dev)
        w13, s13 = fb.fp8bs_quant_weight(w, fb.FP8BS_SCALE_F32)
        del w
        w = synth.w_f32_torch(MOE_E * MOE_H, I, seed=951, device=dev)
        w2, s2 = fb.fp8bs_quant_weight(w, fb.FP8BS_SCALE_F32)
        del w
        torch.cuda.empty_cache()
        w13 = w13.view(MOE_E, 2 * I, MOE_H)
        s13 = s13.view(MOE_E, 2 * I // 128, MOE_H // 128)
        w2 = w2.view(MOE_E, MOE_H, I)
        s2 = s2.view(MOE_E, MOE_H // 128, I // 128)
        per_expert = 3 * I * MOE_H + (3 * I * MOE_H // 16384) * 4
        rows = {}
        for M in ms:
            routes = [synth.moe_routing(M, MOE_S, MOE_E, seed=960 + 31 * M + c) for c in range(COPIES)]
            ids = [torch.from_numpy(r[0]).to(dev) for r in routes]
            tws = [torch.from_numpy(r[1]).to(dev) for r in routes]
            x = synth.x_bf16_torch(M, MOE_H, seed=970 + M, device=dev)
            y = torch.empty((M, MOE_H), dtype=torch.bfloat16, device=dev)
            ws = fb.new_moe_workspace(M, MOE_S, MOE_H, I, dev)
            us = graph_us_per_call(torch, stream, lambda i: fb.fp8bs_moe_w8a16(
                x, ids[i], tws[i], w13, s13, w2, s2, y=y, workspace=ws), COPIES, 20)
            rc = fb.fp8bs_check_error(ws, stream)
            if rc != 0:
                raise SystemExit(f"MoE {name} M={M}: device error {fb.fp8bs_status_string(rc)}")
            active = statistics.mean(len(set(r[0].ravel().tolist())) for r in routes)
            nbytes = active * per_expert + 4 * M * MOE_H + 8 * M * MOE_S
            gbps = nbytes / us / 1e3
            rows[str(M)] = {"us": round(us, 2), "active_experts": round(active, 1),
                            "bytes": int(nbytes), "GBps": round(gbps, 1), "frac": round(gbps / peak, 3)}
            del ids, tws, x, y, ws
        out["configs"][f"{name} I={I}"] = rows
        del w13, s13, w2, s2
        torch.cuda.empty_cache()
    out["peak"] = peak
    out["kernels"] = "moe_gate_up_kernel, moe_down_kernel, moe_combine_kernel"
    out["bound"] = "hbm"
    return out


def hbm_peak():
    """(GB/s, source): the measured copy bandwidth, else the fallback figure."""
    try:
        with open(os.path.join(ROOT, "MEASURED_PEAKS.json")) as f:
            return float(json.load(f)["hbm_gbs"]), "measured hbm_gbs (copy, burst) of MEASURED_PEAKS.json"
    except (OSError, ValueError, KeyError):
        return 6800.0, "fallback 6.8 TB/s"


def progress(msg: str) -> None:
    if os.environ.get("FP8BS_BENCH_VERBOSE"):
        print(f"[bench {time.strftime('%H:%M:%S')}] {msg}", file=sys.stderr, flush=True)


def run_gpu(args):
    import torch

    import fp8_block_scale_x128_gb300 as fb

    world, rank, local = dist_setup()
    if not torch.cuda.is_available():
        raise SystemExit("bench.py needs a CUDA GPU (the fused kernel has no CPU path)")
    torch.cuda.set_device(local)
    dev = torch.device("cuda", local)
    fb.build()
    fb.lib()
    stream = torch.cuda.Stream(device=dev)
    if args.moe_only:
        if rank == 0:
            print(json.dumps({"moe_w8a16": moe_table(fb, torch, dev, stream, hbm_peak()[0])}), flush=True)
        return 0
    if args.producer_only:
        if rank == 0:
            line = {"producer_rmsnorm_quant": producer_table(fb, torch, dev, stream, hbm_peak()[0])}
            print(json.dumps(line), flush=True)
        return 0
    desc, calls = workload_plan(args.workload)
    step_bytes = sum(algorithmic_bytes(M, N, K, kind) for (M, N, K, kind, _) in calls)
    pdl = not args.no_pdl
    progress("building the step (weights, graph)")
    st = Step(fb, torch, calls, dev, stream, graph=not args.no_graph, pdl=pdl)
    with ClockSampler(local) as clk:
        progress("timed region")
        ms = time_steps(torch, st, args.steps, args.warmup, world, dev)
    clocks = clk.summary()
    sec = ms / 1e3
    launches = len(calls) * args.steps
    value = world * step_bytes * args.steps / sec / 1e9
    achieved = step_bytes * args.steps / sec / 1e9
    status = fb.fp8bs_check_error(st.workspace, st.stream)
    if status != 0:
        raise SystemExit(f"device error {status} during the timed region")
    del st
    torch.cuda.empty_cache()

    # end to end through the public call with host buffers: each step copies
    # all of its calls' x from pinned host memory and all of their y back,
    # inside the timed region
    progress("end-to-end step")
    st_io = Step(fb, torch, calls, dev, stream, io=True, pdl=pdl)
    e2e_steps = max(3, args.steps // 4)
    ms_io = time_steps(torch, st_io, e2e_steps, min(args.warmup, 10), world, dev)
    e2e_value = world * step_bytes * e2e_steps / (ms_io / 1e3) / 1e9
    h2d = sum(2 * M * K for (M, N, K, _k, _w) in calls)
    d2h = sum(2 * M * N for (M, N, K, _k, _w) in calls)
    del st_io
    torch.cuda.empty_cache()

    per_m = per_m_two = above_32 = None
    if args.workload == "msweep" and rank == 0 and not args.no_per_m:
        progress("per-M table")
        per_m = per_m_table(fb, torch, dev, stream, pdl)
        progress("per-M table, two-launch path")
        per_m_two = per_m_table(fb, torch, dev, stream, pdl, two_launch=True)
        progress("33..64 tokens (64-token tile)")
        above_32 = {"fused": per_m_table(fb, torch, dev, stream, pdl, ms=M_ABOVE_32),
                    "two_launch": per_m_table(fb, torch, dev, stream, pdl, two_launch=True,
                                              ms=M_ABOVE_32)}

    peak, peak_src = hbm_peak()

    others = None
    if args.workload == "msweep" and rank == 0 and not args.no_workloads:
        others = workloads_table(fb, torch, dev, stream, pdl, peak)

    producer = None
    if rank == 0 and not args.no_producer:
        progress("RMSNorm + quant producer")
        producer = producer_table(fb, torch, dev, stream, peak)
    moe = None
    if rank == 0 and not args.no_moe:
        progress("MoE layer")
        moe = moe_table(fb, torch, dev, stream, peak)

    cpu = None
    if rank == 0 and not args.no_cpu_baseline:
        cpu = cpu_baseline(calls, args.cpu_seconds)

    if rank == 0:
        line = {
            "metric": METRIC, "value": value, "unit": "GB/s", "n_gpus": world,
            "steps": args.steps, "warmup": args.warmup, "ms_per_step": ms / args.steps,
            "higher_is_better": True, "scaling": "weak", "vs_baseline": None,
            "dtype": "e4m3 x e4m3 -> f32 (bf16 in, bf16 out)", "data": "synthetic",
            "us_per_call": ms * 1e3 / launches,
            "config": bench_config(desc, calls),
            "launch": {"graph": ("eager launches" if args.no_graph
                                 else "one CUDA graph replay per step"),
                       "pdl": pdl},
            "per_m_us_and_GBps": per_m,
            "per_m_two_launch_us_and_GBps": per_m_two,
            "m_above_32_us_and_GBps": above_32,
            "workloads": others,
            "producer_rmsnorm_quant": producer,
            "moe_w8a16": moe,
            "roofline": {"bound": "hbm", "achieved": achieved, "peak": peak, "unit": "GB/s",
                         "frac": achieved / peak, "traffic": dram_traffic_per_launch(args.workload),
                         "peak_source": peak_src, "kernel": "fused_quant_gemm_kernel",
                         "achieved_def": "algorithmic bytes per launch / (timed region / launches)"},
            "cpu_baseline": cpu,
            "e2e": {"value": e2e_value, "unit": "GB/s", "h2d_bytes_per_step": h2d,
                    "d2h_bytes_per_step": d2h, "steps": e2e_steps,
                    "path": "per step: one copy of every call's x from pinned host memory, the "
                            "step's fp8bs_gemm_fused calls, one copy of every call's y to pinned "
                            "host memory; one CUDA graph per step"},
            "gpu_launches": launches,
            "clocks": clocks,
        }
        print(json.dumps(line), flush=True)
    if world > 1:
        import torch.distributed as dist
        dist.destroy_process_group()
    return 0


def main(argv=None):
    ap = argparse.ArgumentParser(description=__doc__, formatter_class=argparse.RawTextHelpFormatter)
    ap.add_argument("--gpus", type=int, default=1)
    ap.add_argument("--steps", type=int, default=2000)
    ap.add_argument("--warmup", type=int, default=20)
    ap.add_argument("--impl", choices=["fp8bs", "reference"], default="fp8bs")
    ap.add_argument("--workload", default="msweep")
    ap.add_argument("--cpu-seconds", type=float, default=10.0)
    ap.add_argument("--no-cpu-baseline", action="store_true")
    ap.add_argument("--no-per-m", action="store_true")
    ap.add_argument("--no-workloads", action="store_true",
                    help="skip the table of the other workloads (smallest, shapes, ue8m0, chains)")
    ap.add_argument("--no-producer", action="store_true",
                    help="skip the RMSNorm + quant producer's table")
    ap.add_argument("--producer-only", action="store_true",
                    help="time only the RMSNorm + quant producer and print its table")
    ap.add_argument("--no-moe", action="store_true", help="skip the MoE layer's table")
    ap.add_argument("--moe-only", action="store_true",
                    help="time only the MoE layer and print its table")
    ap.add_argument("--no-pdl", action="store_true",
                    help="plain launches instead of programmatic dependent launch")
    ap.add_argument("--no-graph", action="store_true",
                    help="launch every call eagerly instead of replaying a CUDA graph")
    args = ap.parse_args(argv)
    if args.warmup < 3:
        raise SystemExit("--warmup must be at least 3")
    if args.steps < 1:
        raise SystemExit("--steps must be at least 1")
    if args.impl == "reference":
        return run_reference(args)
    return run_gpu(args)


if __name__ == "__main__":
    sys.exit(main())
