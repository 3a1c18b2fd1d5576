"""Per-phase timeline of the fused GEMM under CUDA-graph replay.

    python -m fp8_block_scale_x128_gb300.timeline [--M 1 8 16 32] [--N 5120] [--K 4096]
                                                  [--kind 0] [--copies 24] [--no-pdl]

Builds the traced variant of the library (FP8BS_TRACE: every CTA of the fused
kernel stamps its phase boundaries with %globaltimer and clock64), captures for
each M a graph of `copies` calls on as many independently seeded weight
copies (the layout of bench.py's steps), replays it, and prints, as medians
over the calls of the last replay:

  period          time between the last CTA exits of consecutive calls
  entry           each CTA's first instruction, after the previous call's
                  last exit (negative: started while that call still ran)
  release         each CTA's return from the wait on the previous kernel,
                  after the previous call's last exit
  phase rows      each CTA's phase stamps after its own release (SM clock
                  cycles converted with that CTA's measured clock), as the
                  median and the maximum over the call's CTAs; "last CTA" is
                  the CTA that exits last

The stamp points are listed in csrc/trace.cuh.  Timing numbers come from the
traced build, whose stamps cost a few instructions each: use bench.py for
throughput, this for where a call's time goes.
"""

from __future__ import annotations

import argparse
import statistics
import sys

POINTS = (["entry", "setup", "wait", "quant_first", "quant_done", "xchg_done", "mma_first",
           "mma_last", "epi_last", "publish", "reduce_end", "teardown", "exit", "xload", "epoch",
           "gather"] + [f"mma_unit{i}" for i in range(10)] + [f"epi_unit{i}" for i in range(10)]
          + [f"refill{j}" for j in range(8)] + [f"mma_issued{i}" for i in range(4)]
          + [f"epi_seen{i}" for i in range(8)]
          + ["iss_wait", "iss_ring", "iss_acc", "iss_issue", "iss_rest"]
          + ["gather_loaded", "gather_polls", "gather_summed"])
# points that hold a count, not a time
COUNTS = ["gather_polls"]
# points that hold a cycle count (a duration), not a time
DURATIONS = ["iss_wait", "iss_ring", "iss_acc", "iss_issue", "iss_rest"]
PHASES = (["xload", "xchg_done", "quant_first", "quant_done", "mma_last",
           "epi_last", "publish", "gather", "epoch", "gather_loaded", "gather_summed", "reduce_end", "teardown", "exit"]
          + [f"mma_unit{i}" for i in range(10)] + [f"epi_unit{i}" for i in range(10)]
          + [f"refill{j}" for j in range(8)] + [f"mma_issued{i}" for i in range(4)]
          + [f"epi_seen{i}" for i in range(8)])


def _med(v):
    return statistics.median(v) if v else float("nan")


def analyse(tr, epochs, grid):
    """Per-call statistics from the trace array for the given call epochs."""
    import numpy as np
    W = POINTS.index("wait")
    E = POINTS.index("exit")
    N0 = POINTS.index("entry")
    calls = []
    for e in epochs:
        rec = tr[e % tr.shape[0], :grid]           # [cta][point][2]
        gt = rec[:, :, 0].astype(np.int64)
        ck = rec[:, :, 1].astype(np.int64)
        # a point taken with clock64 only has globaltimer 1: times within a CTA
        # come from clock64, lining CTAs up from the entry, wait and exit stamps
        ok = (gt[:, N0] > 1) & (gt[:, E] > 1) & (gt[:, W] > 1)
        if not ok.all():
            return None
        # SM clock per CTA (cycles per ns) over entry -> exit
        span_ns = np.maximum(gt[:, E] - gt[:, N0], 1)
        ghz = (ck[:, E] - ck[:, N0]) / span_ns
        phases = {}
        for name in PHASES + DURATIONS + COUNTS:
            j = POINTS.index(name)
            have = gt[:, j] > 0
            if not have.any():
                continue
            if name in COUNTS:
                dt_us = ck[have, j].astype(np.float64)
            elif name in DURATIONS:
                dt_us = ck[have, j] / ghz[have] / 1e3
            else:
                dt_us = (ck[have, j] - ck[have, W]) / ghz[have] / 1e3
            phases[name] = (float(np.median(dt_us)), float(dt_us.max()), int(have.sum()))
        last = int(np.argmax(gt[:, E]))
        last_row = {}
        for name in PHASES + DURATIONS + COUNTS:
            j = POINTS.index(name)
            if gt[last, j] > 0 and name not in COUNTS:
                base = 0 if name in DURATIONS else ck[last, W]
                last_row[name] = float((ck[last, j] - base) / ghz[last] / 1e3)
        calls.append({"entry_min": int(gt[:, N0].min()), "wait": gt[:, W], "entry": gt[:, N0],
                      "exit_max": int(gt[:, E].max()), "phases": phases, "last": last_row,
                      "ghz": float(np.median(ghz))})
    return calls


def report(M, N, K, grid, calls) -> str:
    out = [f"M={M} N={N} K={K}: grid {grid}, {len(calls) - 1} calls after the first "
           f"(SM clock {_med([c['ghz'] for c in calls]):.2f} GHz)"]
    period = [calls[i]["exit_max"] - calls[i - 1]["exit_max"] for i in range(1, len(calls))]
    out.append(f"  period between last exits          {_med(period) / 1e3:7.2f} us")
    for key, label in (("entry", "entry after previous last exit"),
                       ("wait", "release after previous last exit")):
        lo, md, hi = [], [], []
        for i in range(1, len(calls)):
            d = (calls[i][key] - calls[i - 1]["exit_max"]) / 1e3
            lo.append(float(d.min()))
            md.append(float(statistics.median(d.tolist())))
            hi.append(float(d.max()))
        out.append(f"  {label:34s} first {_med(lo):6.2f}  median {_med(md):6.2f}  last {_med(hi):6.2f} us")
    span = [(calls[i]["exit_max"] - int(calls[i]["wait"].max())) / 1e3 for i in range(1, len(calls))]
    out.append(f"  last exit after the last release   {_med(span):7.2f} us")
    out.append("  after each CTA's own release (us)   median   max    CTAs   last CTA")
    for name in PHASES + DURATIONS + COUNTS:
        if name == COUNTS[0]:
            out.append("  counts                               median   max    CTAs")
        if name == DURATIONS[0]:
            out.append("  the MMA issuer's loop, summed (us)   median   max    CTAs   last CTA")
        rows = [c["phases"][name] for c in calls[1:] if name in c["phases"]]
        if not rows:
            continue
        lst = [c["last"][name] for c in calls[1:] if name in c["last"]]
        out.append(f"    {name:30s} {_med([r[0] for r in rows]):7.2f} {_med([r[1] for r in rows]):7.2f}"
                   f" {int(_med([r[2] for r in rows])):6d} {_med(lst):8.2f}")
    return "\n".join(out)


def main(argv=None):
    ap = argparse.ArgumentParser(description=__doc__, formatter_class=argparse.RawTextHelpFormatter)
    ap.add_argument("--M", type=int, nargs="+", default=[1, 8, 16, 32])
    ap.add_argument("--N", type=int, default=5120)
    ap.add_argument("--K", type=int, default=4096)
    ap.add_argument("--kind", type=int, default=0)
    ap.add_argument("--copies", type=int, default=24)
    ap.add_argument("--replays", type=int, default=20)
    ap.add_argument("--no-pdl", action="store_true")
    args = ap.parse_args(argv)
    import numpy as np
    import torch

    import fp8_block_scale_x128_gb300 as fb
    import synth

    fb.use_trace_library()
    fb.lib()
    dev = torch.device("cuda", 0)
    sm = torch.cuda.get_device_properties(dev).multi_processor_count
    N, K, kind = args.N, args.K, args.kind
    packs = []
    for c in range(args.copies):
        w = synth.w_f32_torch(N, K, seed=104729 * c + N + K, device=dev)
        wq, ws = fb.fp8bs_quant_weight(w, kind)
        packs.append(fb.fp8bs_prepack_weight(wq, ws, kind))
        del w, wq, ws
    units = (N // 128) * (K // 128)
    grid = min(units, sm)
    stream = torch.cuda.Stream(device=dev)
    for M in args.M:
        x = synth.x_bf16_torch(M, K, seed=31 + M, device=dev)
        y = torch.empty((M, N), dtype=torch.bfloat16, device=dev)
        wsp = fb.new_workspace(N, K, dev)
        torch.cuda.synchronize()

        def enqueue():
            for pk in packs:
                fb.fp8bs_gemm_fused(x, pk, N, K, kind, y=y, workspace=wsp, pdl=not args.no_pdl,
                                    stream=stream)

        with torch.cuda.stream(stream):
            enqueue()
        stream.synchronize()
        g = torch.cuda.CUDAGraph()
        with torch.cuda.graph(g, stream=stream):
            enqueue()
        for _ in range(args.replays):
            g.replay()
        torch.cuda.synchronize()
        rc = fb.fp8bs_check_error(wsp)
        if rc != 0:
            raise SystemExit(f"M={M}: device status {rc}")
        last_epoch = int(wsp[256:260].view(torch.int32).item()) & 0xFFFFFFFF
        epochs = list(range(last_epoch - args.copies + 1, last_epoch + 1))
        tr = fb.fp8bs_trace_read()
        calls = analyse(tr, epochs, grid)
        if calls is None:
            print(f"M={M}: incomplete trace (grid {grid})")
            continue
        print(report(M, N, K, grid, calls), flush=True)
        del g, x, y, wsp
    return 0


if __name__ == "__main__":
    sys.exit(main())
