"""Phase timeline of the split kernel from a clock-stamped build.

Builds libmla with -DMLA_TRACE into split_kv_mla_gb300/_build_trace/ (the
kernel then writes the global timer at nine points of every CTA's life), runs a
workload a few times through the public calls (L2 flushed before each launch
unless --warm), and prints, per phase, when CTAs
reach it relative to the launch's first CTA start (mean / min / max over CTAs,
microseconds), plus the span of the CTAs' lives.

    python -m split_kv_mla_gb300.trace c1q1 [c4-8 ...] [--splits N] [--tile 16|32]

Workload names are bench.py's.  The traced build is for timelines only: its
stamps cost a few global stores per CTA, and bench.py never loads it.
"""
from __future__ import annotations

import argparse
import ctypes
import os
import sys

import numpy as np

HERE = os.path.dirname(os.path.abspath(__file__))
ROOT = os.path.dirname(HERE)
TRACE_BUILD = os.path.join(HERE, "_build_trace")
SLOTS = 12          # stamps per CTA (kTraceSlots)
MAX_CTAS = 8192     # kTraceCtas
BLOCK_CTAS, BLOCKS, BLOCK_EVENTS = 4, 64, 8   # per-block events of the first CTAs
WORDS = MAX_CTAS * SLOTS + BLOCK_CTAS * BLOCKS * BLOCK_EVENTS
EVENTS = ["issue", "issued", "qk", "s_read", "p_done", "pv", "s1_read", "p1_done"]
PHASES = ["start", "waited", "gather0", "qk0", "pv_last", "o_ready", "staged", "stored", "end",
          "q_tile", "mma_go"]


def build_traced() -> str:
    from split_kv_mla_gb300 import build
    return build.build(extra=("-DMLA_TRACE",), build_dir=TRACE_BUILD)


def phase_table(stamps: np.ndarray, ctas: int):
    """Rows (phase, mean, min, max) in microseconds after the first CTA start;
    phases that no CTA stamped are left out."""
    t = stamps[:ctas].astype(np.int64)
    t0 = t[:, 0][t[:, 0] > 0].min()
    rows = []
    for i, name in enumerate(PHASES):
        v = t[:, i]
        v = v[v > 0]
        if v.size:
            rel = (v - t0) / 1e3
            rows.append((name, rel.mean(), rel.min(), rel.max()))
    return rows


def main(argv=None):
    ap = argparse.ArgumentParser(description="split-kernel phase timeline")
    ap.add_argument("workloads", nargs="*", default=["c1q1"])
    ap.add_argument("--splits", type=int, default=0)
    ap.add_argument("--tile", type=int, default=0, choices=(0, 16, 32),
                    help="query rows per CTA (default: the planner's)")
    ap.add_argument("--reps", type=int, default=5)
    ap.add_argument("--warm", action="store_true",
                    help="leave the inputs in L2 between launches (default: flush L2 first)")
    args = ap.parse_args(argv)
    sys.path.insert(0, ROOT)
    lib_path = build_traced()
    import torch
    from split_kv_mla_gb300 import mla
    import bench
    lib = mla.load(path=lib_path)
    lib.mla_trace_read.argtypes = [ctypes.c_void_p, ctypes.c_int64]
    device = torch.device("cuda", 0)
    for name in args.workloads:
        kind, inp, desc = bench.make_workload(name)
        runner = bench.Runner(kind, inp, device, 1, args.splits)
        plan = runner.plan_step()
        if args.tile:
            rows = plan.q_len * plan.num_heads
            plan.rows_per_cta = args.tile
            plan.head_blocks = plan.grid_x = -(-rows // args.tile)
        runner.plan = plan
        stream = torch.cuda.current_stream()
        spans = []
        flush = None if args.warm else torch.empty(512 << 20, dtype=torch.uint8, device=device)
        for _ in range(args.reps):
            lib.mla_trace_clear()
            if flush is not None:
                flush.fill_(1)   # evict the inputs from L2 (512 MiB > 129 MB of L2)
            runner.step(0, stream, splits_only=True, plan=plan)
            torch.cuda.synchronize()
            raw = np.zeros(WORDS, dtype=np.uint64)
            if lib.mla_trace_read(raw.ctypes.data, raw.size) != 0:
                raise RuntimeError("mla_trace_read failed")
            buf = raw[:MAX_CTAS * SLOTS].reshape(MAX_CTAS, SLOTS)
            blk = raw[MAX_CTAS * SLOTS:].reshape(BLOCK_CTAS, BLOCKS, BLOCK_EVENTS)
            ctas = runner.plan.grid_x * runner.plan.grid_y * runner.plan.grid_z
            spans.append(phase_table(buf, min(ctas, MAX_CTAS)))
        last = spans[-1]
        print(f"{name}: {desc}; {ctas} CTAs, {runner.plan.num_splits} splits "
              f"(last of {args.reps} launches, us after the first CTA start)")
        for phase, mean, lo, hi in last:
            print(f"  {phase:9s} mean {mean:8.2f}  min {lo:8.2f}  max {hi:8.2f}")
        # the block chain of CTA 0, us after its start
        t0 = int(buf[0, 0])
        print("  CTA 0 per block (us after its start): " + " ".join(f"{e:>7s}" for e in EVENTS))
        for j in range(BLOCKS):
            row = blk[0, j].astype(np.int64)
            if not row.any():
                break
            print(f"    block {j:3d}                          " +
                  " ".join(f"{(v - t0) / 1e3:7.2f}" if v else "      -" for v in row))
        del runner, flush
        torch.cuda.empty_cache()


if __name__ == "__main__":
    main()
