#!/usr/bin/env python3
"""Benchmark: split-KV absorbed-MLA decode over a paged fp8 KV cache on GB300.

A step is one full pass of the decode path (plan, split kernel over the paged
fp8 rows, online base-2 softmax partials, split-K reduce) over one batch of the
synthetic workload.  Default workload: B=8 requests, H=16 heads, S=8192 keys
each, q_len=1, 576-byte e4m3fn rows (37.7 MB of KV per call).

Timing: steps are captured into CUDA graphs (the pages' own method: "timed as
CUDA-graph replays") and replayed; the inputs are rotated over enough device
copies that the rotation is > 4x the L2 size, so every step streams its KV from
HBM.  The dominant kernel's duration comes from CUDA events recorded around
each of its launches on its own stream.  `e2e` repeats the measurement through
the public call with host buffers: per step the queries and page table go
host->device from pinned memory and o/lse come back.

Prints ONE JSON line (rank 0).  `--impl reference` times the fp64 CPU oracle on
the host's cores on the same metric instead.
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
import threading
import time

import torch

ROOT = os.path.dirname(os.path.abspath(__file__))
sys.path.insert(0, ROOT)

METRIC = ("MLA decode µs/call and achieved KV-stream HBM GB/s "
          "(fraction of GB300 peak)")
FALLBACK_HBM_GBS = 6800.0
ROW_BYTES = {"dense": 576, "sparse": 512}


# ---- workloads ------------------------------------------------------------------

def make_workload(name: str):
    from split_kv_mla_gb300 import inputs as gen
    if name == "c0":
        return "dense", gen.workload_c0(), "B=1 H=16 q_len=1 S=256"
    if name in ("c1", "c1q1"):
        return "dense", gen.workload_c1(q_len=1), "B=8 H=16 q_len=1 S=8192"
    if name == "c1q4":
        return "dense", gen.workload_c1(q_len=4), "B=8 H=16 q_len=4 S=8192"
    if name.startswith("c2-"):
        b, s = name[3:].split("x")
        return "dense", gen.workload_c2(int(b), int(s)), f"B={b} H=64 q_len=1 S={s}"
    if name == "c3":
        return "dense", gen.workload_c3(), "B=64 H=128 q_len=1 S~U[1024,32768]"
    if name.startswith("c4-"):
        t = int(name[3:])
        return "sparse", gen.workload_c4(t), f"T={t} H=64 top-k 2048 of 131072, 448+64"
    if name.startswith("c4x-"):
        t = int(name[4:])
        return ("sparse", gen.workload_c4x(t),
                f"T={t} H=64 top-k 2048 of 131072 + 512 of a 32768-row second cache, 448+64")
    if name.startswith("p-"):
        b, s = (int(x) for x in name[2:].split("-"))
        return "dense", gen.workload_c1(q_len=4, seq=s, batch=b), f"B={b} H=16 q_len=4 S={s}"
    if name.startswith("d-"):
        # any dense shape: d-B-H-Q-S (batch, heads, q_len, keys per request)
        b, h, q, s = (int(x) for x in name[2:].split("-"))
        return ("dense", gen.dense_inputs(b, q, h, [s] * b, 0),
                f"B={b} H={h} q_len={q} S={s}")
    if name.startswith("dcp") and "-" in name:
        # rank 0's share of a dense workload under decode context parallelism
        w, base = name[3:].split("-", 1)
        kind, inp, desc = make_workload(base)
        if kind != "dense" or int(w) < 2:
            raise SystemExit("DCP applies to dense workloads over 2 or more ranks")
        shard, glen = dcp_rank_inputs(inp, int(w), 0)
        shard.dcp_glen, shard.dcp_world, shard.dcp_base = glen, int(w), inp
        return "dcp", shard, f"{desc}, DCP rank 0 of {w}"
    raise SystemExit(f"unknown workload {name}")


def dcp_rank_inputs(inp, world: int, rank: int = 0):
    """(share inputs, glen): the rank's page table under DCP (positions
    p % world == rank) over the same queries and pool."""
    import dataclasses
    from split_kv_mla_gb300 import dcp
    sl, si, sp, glen = dcp.shard_page_table(inp.seq_lens, inp.kv_indices, inp.kv_indptr,
                                            rank, world)
    return dataclasses.replace(inp, seq_lens=sl, kv_indices=si, kv_indptr=sp), glen


# The pages' MI300X results for the same dense shapes (H=16, q_len=4, shuffled
# page-size-1 slots, KV bytes only): (B, S) -> TB/s ("Results -- MLA decode",
# moonmath-ai/amd-kernels README).  Context on other hardware, not the target.
PAGES_MI300X_TBS = {(1, 150000): 1.13, (2, 150000): 1.54, (8, 8192): 0.73, (8, 32768): 1.48,
                    (8, 65536): 1.67, (8, 150000): 1.75, (16, 150000): 1.70, (32, 8192): 1.45}


def pages_baseline_gbs(name: str):
    """The pages' GB/s for exactly this workload, or None."""
    if name.startswith("dcp"):
        return None
    if name == "c1q4":
        key = (8, 8192)
    elif name.startswith("p-"):
        key = tuple(int(x) for x in name[2:].split("-"))
    else:
        return None
    v = PAGES_MI300X_TBS.get(key)
    return None if v is None else v * 1000.0


def max_over_ranks(x: float, world: int, device) -> float:
    """The largest x over all ranks (every rank gets it)."""
    if world <= 1:
        return x
    t = torch.tensor([x], dtype=torch.float64, device=device)
    torch.distributed.all_reduce(t, op=torch.distributed.ReduceOp.MAX)
    return float(t.item())


def job_gbs(bytes_per_call: int, world: int, ms_per_call: float) -> float:
    """Whole-job GB/s: every rank's calls over the slowest rank's time."""
    return bytes_per_call * world / (ms_per_call * 1e-3) / 1e9


def keys_per_call(kind, inp) -> int:
    if kind in ("dense", "dcp"):
        return int(inp.seq_lens.sum())
    extra = int((inp.extra_indices >= 0).sum()) if inp.extra_topk else 0
    return int((inp.indices >= 0).sum()) + extra


def kv_bytes_per_call(kind, inp) -> int:
    return keys_per_call(kind, inp) * row_bytes(kind)


def workload_label(name, kind, desc) -> str:
    """The config's workload string, the same in both arms."""
    return (f"{name}: dense MLA decode {desc}" if kind != "sparse"
            else f"{name}: sparse top-k MLA decode {desc}")


def row_bytes(kind) -> int:
    return ROW_BYTES["sparse" if kind == "sparse" else "dense"]


def flops_per_call(kind, inp) -> int:
    # 2 * (QK width + V width) per key and query row
    if kind in ("dense", "dcp"):
        rows = inp.q_len * inp.num_heads
        return 2 * (576 + 512) * rows * keys_per_call(kind, inp)
    return 2 * (512 + 448) * inp.num_heads * keys_per_call(kind, inp)


# ---- measured peaks, clocks, traffic ----------------------------------------------

def measured_peaks():
    p = os.path.join(ROOT, "MEASURED_PEAKS.json")
    try:
        d = json.load(open(p))
        return float(d["hbm_gbs"]), "measured"
    except Exception:
        return FALLBACK_HBM_GBS, "fallback"


class ClockSampler:
    """nvidia-smi clocks and throttle reasons sampled in the background."""

    FIELDS = ("index,clocks.sm,clocks.max.sm,power.draw,clocks_event_reasons.active,"
              "clocks_event_reasons.hw_slowdown,clocks_event_reasons.hw_thermal_slowdown,"
              "clocks_event_reasons.sw_thermal_slowdown,clocks_event_reasons.sw_power_cap")

    def __init__(self, device_id: str):
        self.idx = device_id
        self.proc = None
        self.lines = []
        self.t = None

    def start(self):
        try:
            self.proc = subprocess.Popen(
                ["nvidia-smi", "-i", str(self.idx), f"--query-gpu={self.FIELDS}",
                 "--format=csv,noheader,nounits", "-lms", "50"],
                stdout=subprocess.PIPE, stderr=subprocess.DEVNULL, text=True)
        except Exception:
            self.proc = None
            return
        self.t = threading.Thread(target=self._read, daemon=True)
        self.t.start()

    def _read(self):
        for line in self.proc.stdout:
            self.lines.append(line.strip())

    def stop(self):
        if self.proc is None:
            return
        self.proc.terminate()
        try:
            self.proc.wait(timeout=5)
        except Exception:
            self.proc.kill()
        if self.t:
            self.t.join(timeout=2)

    def summary(self):
        sm, mx, reasons = [], [], set()
        names = ["hw_slowdown", "hw_thermal_slowdown", "sw_thermal_slowdown", "sw_power_cap"]
        for line in self.lines:
            parts = [x.strip() for x in line.split(",")]
            if len(parts) < 9:
                continue
            try:
                sm.append(float(parts[1]))
                mx.append(float(parts[2]))
            except ValueError:
                continue
            for n, v in zip(names, parts[5:9]):
                if v.lower() in ("active", "1", "0x1"):
                    reasons.add(n)
        if not sm:
            return {"sm_mhz": None, "sm_max_mhz": None, "reasons": [], "samples": 0}
        return {"sm_mhz": statistics.median(sm), "sm_max_mhz": max(mx),
                "reasons": sorted(reasons), "samples": len(sm)}


def split_kernel_source_hash() -> str:
    h = hashlib.sha256()
    csrc = os.path.join(ROOT, "split_kv_mla_gb300", "csrc")
    for f in sorted(os.listdir(csrc)):
        if f.startswith("mla_split") or f.endswith(".cuh"):
            h.update(open(os.path.join(csrc, f), "rb").read())
    return h.hexdigest()[:16]


def recorded_traffic(workload: str):
    """DRAM bytes per launch of the split kernel from the committed ncu summary,
    or None if it was taken on another build of the kernel."""
    p = os.path.join(ROOT, "profiles", "traffic.json")
    try:
        d = json.load(open(p))
        e = d[workload]
        if e.get("kernel_src_sha") != split_kernel_source_hash():
            return None
        return float(e["dram_bytes_per_launch"])
    except Exception:
        return None


# ---- our arm ---------------------------------------------------------------------

class Runner:
    """Device copies of one workload and the calls that run it."""

    def __init__(self, kind, inp, device, copies, force_splits=0, force_tile=0):
        from split_kv_mla_gb300 import mla
        self.mla = mla
        self.kind, self.inp, self.device = kind, inp, device
        self.force_splits, self.force_tile = force_splits, force_tile
        sms = mla.sm_count(device)
        self.sms = sms
        if kind == "dense":
            self.plan = mla.mla_decode_plan(inp.batch, inp.q_len, inp.num_heads,
                                            inp.total_keys, sms)
            base = dict(q_lat=inp.q_lat, q_pe=inp.q_pe, pool=inp.pool, seq_lens=inp.seq_lens,
                        kv_indices=inp.kv_indices, kv_indptr=inp.kv_indptr)
            rows = inp.batch * inp.q_len
            self.o = torch.empty(rows, inp.num_heads, 512, dtype=torch.bfloat16, device=device)
            self.lse = torch.empty(rows, inp.num_heads, dtype=torch.float32, device=device)
        else:
            self.plan = mla.mla_sparse_decode_plan(inp.num_tokens, inp.num_heads, inp.topk, sms,
                                                   extra_topk=inp.extra_topk)
            base = dict(q_nope=inp.q_nope, q_pe=inp.q_pe, pool=inp.pool, indices=inp.indices)
            if inp.extra_topk:
                base.update(extra_pool=inp.extra_pool, extra_indices=inp.extra_indices)
            self.o = torch.empty(inp.num_tokens, inp.num_heads, 448, dtype=torch.bfloat16,
                                 device=device)
            self.lse = torch.empty(inp.num_tokens, inp.num_heads, dtype=torch.float32,
                                   device=device)
        if force_splits or force_tile:
            self.plan = self.plan_step()
        first = {k: v.to(device) for k, v in base.items()}
        self.copies = [first] + [{k: v.clone() for k, v in first.items()}
                                 for _ in range(copies - 1)]
        self.ws = mla.workspace(self.plan, device)
        self.sms = sms

    def plan_step(self):
        mla, inp = self.mla, self.inp
        if self.kind != "sparse":
            p = mla.mla_decode_plan(inp.batch, inp.q_len, inp.num_heads, inp.total_keys,
                                    self.sms)
        else:
            p = mla.mla_sparse_decode_plan(inp.num_tokens, inp.num_heads, inp.topk, self.sms,
                                           extra_topk=inp.extra_topk)
        if self.force_tile:
            # query rows per CTA (16, or 32 above 16 rows): tile sweeps
            rows = p.q_len * p.num_heads
            p.rows_per_cta = self.force_tile
            p.head_blocks = p.grid_x = -(-rows // self.force_tile)
        return mla.mla_plan_force_splits(p, self.force_splits) if self.force_splits else p

    def call(self, d, pool, o, lse, stream, splits_only=False, plan=None):
        """One public call on the inputs `d` (pool given separately)."""
        mla, inp = self.mla, self.inp
        plan = plan or self.plan_step()
        if self.kind == "dense":
            fn = mla.mla_decode_splits if splits_only else mla.mla_decode
            fn(plan, d["q_lat"], d["q_pe"], pool, d["seq_lens"], d["kv_indices"],
               d["kv_indptr"], inp.scale, inp.kv_scale, o_lat=o, lse=lse,
               workspace_t=self.ws, stream=stream)
        elif inp.extra_topk:
            fn = mla.mla_sparse_decode_extra_splits if splits_only else mla.mla_sparse_decode_extra
            fn(plan, d["q_nope"], d["q_pe"], pool, d["indices"], d["extra_pool"],
               d["extra_indices"], inp.scale, inp.kv_scale, o=o, lse=lse, workspace_t=self.ws,
               stream=stream)
        else:
            fn = mla.mla_sparse_decode_splits if splits_only else mla.mla_sparse_decode
            fn(plan, d["q_nope"], d["q_pe"], pool, d["indices"], inp.scale, inp.kv_scale,
               o=o, lse=lse, workspace_t=self.ws, stream=stream)

    def step(self, i, stream, splits_only=False, plan=None):
        d = self.copies[i % len(self.copies)]
        self.call(d, d["pool"], self.o, self.lse, stream, splits_only, plan)

    def input_names(self):
        if self.kind == "sparse":
            return ["q_nope", "q_pe", "indices"] + (["extra_indices"] if self.inp.extra_topk
                                                    else [])
        return ["q_lat", "q_pe", "seq_lens", "kv_indices", "kv_indptr"]

    def launches_per_step(self):
        return 1 if self.plan.num_splits == 1 else 2


class DcpRunner(Runner):
    """Rank 0's step under decode context parallelism, on one GPU: its share of
    the workload (mla_decode_dcp, fp32 share) and the merge of all ranks'
    shares (mla_dcp_lse_merge_ranks).  The other ranks' shares, which an
    all-gather would deliver, are computed once beforehand and stay in place."""

    def __init__(self, shard, device, copies, force_splits=0, force_tile=0):
        super().__init__("dense", shard, device, copies, force_splits, force_tile)
        self.kind = "dcp"
        base_inp, world = shard.dcp_base, shard.dcp_world
        self.world = world
        self.glen = shard.dcp_glen.to(device)
        rows, H = shard.batch * shard.q_len, shard.num_heads
        self.parts = torch.zeros(world, rows, H, 512, dtype=torch.float32, device=device)
        self.lses = torch.full((world, rows, H), -float("inf"), dtype=torch.float32,
                               device=device)
        mla = self.mla
        for k in range(1, world):
            sk, gk = dcp_rank_inputs(base_inp, world, k)
            pk = mla.mla_decode_plan(sk.batch, sk.q_len, sk.num_heads, sk.total_keys, self.sms)
            dk = {n: getattr(sk, n).to(device) for n in
                  ("q_lat", "q_pe", "seq_lens", "kv_indices", "kv_indptr")}
            mla.mla_decode_dcp(pk, dk["q_lat"], dk["q_pe"], self.copies[0]["pool"],
                               dk["seq_lens"], dk["kv_indices"], dk["kv_indptr"], sk.scale,
                               sk.kv_scale, gk.to(device), k, world, o=self.parts[k],
                               lse=self.lses[k], workspace_t=mla.workspace(pk, device))
        torch.cuda.synchronize(device)

    def call(self, d, pool, o, lse, stream, splits_only=False, plan=None):
        mla, inp = self.mla, self.inp
        plan = plan or self.plan_step()
        fn = mla.mla_decode_dcp_splits if splits_only else mla.mla_decode_dcp
        fn(plan, d["q_lat"], d["q_pe"], pool, d["seq_lens"], d["kv_indices"], d["kv_indptr"],
           inp.scale, inp.kv_scale, self.glen, 0, self.world, o=self.parts[0],
           lse=self.lses[0], workspace_t=self.ws, stream=stream)
        if not splits_only:
            mla.mla_dcp_lse_merge_ranks(self.parts, self.lses, out=o, lse_out=lse,
                                        stream=stream)

    def launches_per_step(self):
        return (1 if self.plan.num_splits == 1 else 2) + 1

    def copy_bytes(self):
        return sum(t.numel() * t.element_size() for t in self.copies[0].values())


def capture(runner, stream, n, offset=0):
    g = torch.cuda.CUDAGraph()
    with torch.cuda.stream(stream):
        with torch.cuda.graph(g, stream=stream):
            for i in range(n):
                runner.step(offset + i, stream)
    return g


def time_steps(runner, stream, steps, copies):
    """Device time of exactly `steps` steps (graph replays), in ms."""
    full, rem = divmod(steps, copies)
    g_full = capture(runner, stream, copies) if full else None
    g_rem = capture(runner, stream, rem) if rem else None
    torch.cuda.synchronize()
    start = torch.cuda.Event(enable_timing=True)
    end = torch.cuda.Event(enable_timing=True)
    return g_full, g_rem, full, start, end


def kernel_times(runner, stream, steps, step_ms):
    """Average device duration (ms) of the split kernel, and the rest of a call
    (the split-K reduce and its launch), from CUDA events on the launching stream
    around CUDA-graph replays of split-kernel-only calls over the same rotating
    inputs; the rest is the whole call's time minus the split kernel's."""
    if runner.plan.num_splits == 1:
        return step_ms, 0.0
    copies = len(runner.copies)
    g = torch.cuda.CUDAGraph()
    with torch.cuda.stream(stream):
        with torch.cuda.graph(g, stream=stream):
            for i in range(copies):
                runner.step(i, stream, splits_only=True)
    reps = max(1, steps // copies)
    start = torch.cuda.Event(enable_timing=True)
    end = torch.cuda.Event(enable_timing=True)
    with torch.cuda.stream(stream):
        g.replay()
        start.record(stream)
        for _ in range(reps):
            g.replay()
        end.record(stream)
    torch.cuda.synchronize()
    split_ms = start.elapsed_time(end) / (reps * copies)
    return split_ms, max(0.0, step_ms - split_ms)


def _packed(tensors, device=None, pinned=False):
    """One uint8 buffer holding the tensors back to back (256-byte aligned),
    and views of it with the tensors' shapes and dtypes."""
    offs, total = [], 0
    for t in tensors:
        offs.append(total)
        total += -(-t.numel() * t.element_size() // 256) * 256
    buf = torch.empty(total, dtype=torch.uint8, device=device)
    if pinned:
        buf = buf.pin_memory()
    views = [buf[o:o + t.numel() * t.element_size()].view(t.dtype).view(t.shape)
             for o, t in zip(offs, tensors)]
    return buf, views


def e2e_measure(runner, stream, steps):
    """Same metric through the public call with host buffers: every step copies
    that step's queries and page table from pinned host memory to the device
    (one copy of a packed buffer), runs the decode, and copies o and lse back
    (one copy of a packed buffer); the KV pool is resident cache state and
    rotates over the device copies like the main arm.  As a serving loop would,
    the steps are replayed from a CUDA graph (60 or more steps per replay) and
    pipelined over two sets of buffers: step i's input copy (one copy stream)
    and step i-1's result copy (another) overlap the decode of the step in
    between, and a buffer is reused only after the step two back has finished
    with it."""
    inp = runner.inp
    names = runner.input_names()
    src = [getattr(inp, n).contiguous() for n in names]
    host_in, host_views = _packed(src, pinned=True)
    for hv, t in zip(host_views, src):
        hv.copy_(t)
    dev_in, dviews, dev_out, outs, host_out = [], [], [], [], []
    for _ in range(2):
        buf, views = _packed(src, device=runner.device)
        dev_in.append(buf)
        dviews.append(dict(zip(names, views)))
        obuf, (o, lse) = _packed([runner.o, runner.lse], device=runner.device)
        dev_out.append(obuf)
        outs.append((o, lse))
        host_out.append(_packed([runner.o, runner.lse], pinned=True)[0])
    h2d = host_in.numel()
    d2h = host_out[0].numel()
    plan = runner.plan
    copies = runner.copies
    c_in = torch.cuda.Stream(runner.device)
    c_out = torch.cuda.Stream(runner.device)
    ev_in = [torch.cuda.Event() for _ in range(2)]
    ev_done = [torch.cuda.Event() for _ in range(2)]
    ev_out = [torch.cuda.Event() for _ in range(2)]

    def one(i, first):
        k = i % 2
        d = dviews[k]
        o, lse = outs[k]
        with torch.cuda.stream(c_in):
            if not first:
                c_in.wait_event(ev_done[k])      # step i-2 has read dev_in[k]
            dev_in[k].copy_(host_in, non_blocking=True)
            ev_in[k].record(c_in)
        stream.wait_event(ev_in[k])
        if not first:
            stream.wait_event(ev_out[k])         # step i-2's result has left dev_out[k]
        if "extra_pool" in copies[0]:
            d["extra_pool"] = copies[i % len(copies)]["extra_pool"]
        runner.call(d, copies[i % len(copies)]["pool"], o, lse, stream, plan=plan)
        ev_done[k].record(stream)
        with torch.cuda.stream(c_out):
            c_out.wait_event(ev_done[k])
            host_out[k].copy_(dev_out[k], non_blocking=True)
            ev_out[k].record(c_out)

    def run(n):
        # the copy streams fork from and join back into the decode stream
        c_in.wait_stream(stream)
        c_out.wait_stream(stream)
        for i in range(n):
            one(i, i < 2)
        stream.wait_stream(c_in)
        stream.wait_stream(c_out)

    # one graph holds whole rotations of the input copies, at least 60 steps,
    # so that the pipeline's fill and drain at each replay cost little
    n = max(2, len(copies)) * max(1, -(-60 // max(2, len(copies))))
    with torch.cuda.stream(stream):
        run(3)
    torch.cuda.synchronize()
    g = torch.cuda.CUDAGraph()
    with torch.cuda.stream(stream):
        with torch.cuda.graph(g, stream=stream):
            run(n)
    reps = max(1, steps // n)
    start = torch.cuda.Event(enable_timing=True)
    end = torch.cuda.Event(enable_timing=True)
    with torch.cuda.stream(stream):
        g.replay()
        start.record(stream)
        for _ in range(reps):
            g.replay()
        end.record(stream)
    torch.cuda.synchronize()
    return start.elapsed_time(end) / (reps * n), h2d, d2h


def cpu_baseline(kind, inp, budget_s: float):
    """fp64 oracle on the host's cores over a bounded sample of the workload:
    whole requests (all heads and draft rows), repeated until about budget_s."""
    from oracle import oracle
    oracle.build()
    if kind != "sparse":
        n_req = inp.batch
        req_keys = inp.seq_lens.tolist()
        heads_rows = inp.q_len * inp.num_heads
    else:
        n_req = inp.num_tokens
        req_keys = (inp.indices >= 0).sum(1)
        if inp.extra_topk:
            req_keys = req_keys + (inp.extra_indices >= 0).sum(1)
        req_keys = req_keys.tolist()
        heads_rows = inp.num_heads
    # time one request, then size the sample
    t0 = time.perf_counter()
    items = list(range(0, heads_rows))
    _oracle_items(kind, inp, items)
    t1 = time.perf_counter() - t0
    per_req = max(t1, 1e-4)
    n = max(1, min(n_req, int(budget_s / per_req)))
    items = list(range(0, n * heads_rows))
    t0 = time.perf_counter()
    reps = 0
    while True:
        _oracle_items(kind, inp, items)
        reps += 1
        el = time.perf_counter() - t0
        if el >= budget_s or reps >= 100000:
            break
    keys = sum(req_keys[:n]) * reps
    gbs = keys * row_bytes(kind) / el / 1e9
    sample = (f"{n} of {n_req} {'tokens' if kind == 'sparse' else 'requests'} "
              f"(all {heads_rows} rows each), {reps} pass(es), {el:.1f} s")
    return {"value": gbs, "unit": "GB/s", "cores": oracle.cpu_threads(), "kind": "oracle",
            "sample": sample}


def _oracle_items(kind, inp, items):
    import numpy as np
    from oracle import oracle
    sel = np.asarray(items, dtype=np.int64)
    if kind == "dense":
        oracle.dense_decode(inp, sel)
    elif kind == "dcp":
        # items are the rows of the first n requests of rank 0's share
        import dataclasses
        n = len(items) // (inp.q_len * inp.num_heads)
        end = int(inp.kv_indptr[n])
        sub = dataclasses.replace(inp, batch=n, q_lat=inp.q_lat[:n * inp.q_len],
                                  q_pe=inp.q_pe[:n * inp.q_len], seq_lens=inp.seq_lens[:n],
                                  kv_indices=inp.kv_indices[:end], kv_indptr=inp.kv_indptr[:n + 1])
        oracle.dcp_decode(sub, inp.dcp_glen[:n], 0, inp.dcp_world)
    elif inp.extra_topk:
        # items are the rows of the first n tokens
        import dataclasses
        n = len(items) // inp.num_heads
        sub = dataclasses.replace(inp, num_tokens=n, q_nope=inp.q_nope[:n], q_pe=inp.q_pe[:n],
                                  indices=inp.indices[:n], extra_indices=inp.extra_indices[:n])
        oracle.sparse_extra_decode(sub)
    else:
        oracle.sparse_decode(inp, sel)


# Every synthetic workload timed next to the headline one in the same run (the
# five configurations of the benchmark: c0, c1 at q_len 1 and 4, the four
# split-heavy c2 points, the variable-length c3 batch and the sparse c4 token
# counts).
ALL_WORKLOADS = ["c0", "c1q1", "c1q4", "c2-1x131072", "c2-2x65536", "c2-8x131072",
                 "c2-16x131072", "c3", "c4-1", "c4-8", "c4-24", "c4-64"]


def bf16_peak_tflops():
    p = os.path.join(ROOT, "MEASURED_PEAKS.json")
    try:
        return float(json.load(open(p))["bf16_tflops"]), "measured"
    except Exception:
        return 1900.0, "fallback"


def l2_copies(kind, inp, l2):
    """(copies, bytes per copy): device copies of the inputs whose rotation
    exceeds 4x L2, so every call streams its KV from HBM."""
    dense = kind != "sparse"
    per_copy = (inp.pool.numel() + (inp.q_lat.numel() * 2 if dense else inp.q_nope.numel() * 2)
                + inp.q_pe.numel() * 2 + (inp.kv_indices.numel() * 4 if dense
                                          else inp.indices.numel() * 4))
    if not dense and inp.extra_topk:
        per_copy += inp.extra_pool.numel() + inp.extra_indices.numel() * 4
    return max(1, min(64, math.ceil(4 * l2 / max(per_copy, 1)))), per_copy


def measure_workload(name, device, world, steps, cpu_budget):
    """One workload's call time (graph replays over rotating inputs), its split
    kernel's own time, and the oracle on the host for a short sample."""
    kind, inp, desc = make_workload(name)
    props = torch.cuda.get_device_properties(device)
    l2 = getattr(props, "L2_cache_size", 0) or (126 << 20)
    copies, _ = l2_copies(kind, inp, l2)
    runner = Runner(kind, inp, device, copies)
    stream = torch.cuda.Stream(device)
    with torch.cuda.stream(stream):
        for i in range(3):
            runner.step(i, stream)
    torch.cuda.synchronize()
    g_full, g_rem, full, start, end = time_steps(runner, stream, steps, copies)
    with torch.cuda.stream(stream):
        if g_full is not None:
            g_full.replay()
        start.record(stream)
        for _ in range(full):
            g_full.replay()
        if g_rem is not None:
            g_rem.replay()
        end.record(stream)
    torch.cuda.synchronize()
    ms = max_over_ranks(start.elapsed_time(end) / steps, world, device)
    split_ms, _ = kernel_times(runner, stream, steps, ms)
    split_ms = max_over_ranks(split_ms, world, device)
    peak, _ = measured_peaks()
    tpeak, _ = bf16_peak_tflops()
    kv = kv_bytes_per_call(kind, inp)
    flops = flops_per_call(kind, inp)
    gbs = kv / (ms * 1e-3) / 1e9
    out = {"desc": desc, "us_per_call": round(ms * 1e3, 3),
           "kv_gbs": round(gbs * world, 2),
           "keys_per_s": keys_per_call(kind, inp) * world / (ms * 1e-3),
           "frac_of_measured_hbm": round(gbs / peak, 4),
           "split_kernel_us": round(split_ms * 1e3, 3),
           "split_kernel_frac_of_measured_hbm": round(kv / (split_ms * 1e-3) / 1e9 / peak, 4),
           "tflops": round(flops / (ms * 1e-3) / 1e12, 2),
           "frac_of_bf16_tensor_peak": round(flops / (ms * 1e-3) / 1e12 / tpeak, 4),
           "flop_per_kv_byte": round(flops / kv, 1),
           "bound": "tensor" if flops / kv > tpeak * 1e12 / (peak * 1e9) else "hbm",
           "num_splits": runner.plan.num_splits, "head_blocks": runner.plan.head_blocks}
    if cpu_budget > 0:
        cb = cpu_baseline(kind, inp, cpu_budget)
        out["oracle_gbs"] = round(cb["value"], 4)
        out["oracle_sample"] = cb["sample"]
    del runner, g_full, g_rem
    torch.cuda.synchronize()
    torch.cuda.empty_cache()
    return out


def run_ours(args, rank, world, local_rank):
    torch.cuda.set_device(local_rank)
    device = torch.device("cuda", local_rank)
    from split_kv_mla_gb300 import mla
    mla.load()
    kind, inp, desc = make_workload(args.workload)
    props = torch.cuda.get_device_properties(device)
    l2 = getattr(props, "L2_cache_size", 0) or (126 << 20)
    # rotation copies: total input bytes > 4x L2
    copies, per_copy = l2_copies(kind, inp, l2)
    runner = (DcpRunner(inp, device, copies, args.splits, args.tile) if kind == "dcp"
              else Runner(kind, inp, device, copies, args.splits, args.tile))
    stream = torch.cuda.Stream(device)

    # warm-up (eager) then graphs
    with torch.cuda.stream(stream):
        for i in range(max(args.warmup, 3)):
            runner.step(i, stream)
    torch.cuda.synchronize()
    g_full, g_rem, full, start, end = time_steps(runner, stream, args.steps, copies)
    with torch.cuda.stream(stream):
        for _ in range(args.warmup):  # warm the graphs too
            if g_full is not None:
                g_full.replay()
                break
    torch.cuda.synchronize()

    uuid = str(getattr(props, "uuid", "") or "")
    sampler = ClockSampler(("GPU-" + uuid) if uuid and not uuid.startswith("GPU-") else
                           (uuid or str(local_rank)))
    sampler.start()
    time.sleep(0.2)
    if world > 1:
        torch.distributed.barrier()
    torch.cuda.synchronize()
    with torch.cuda.stream(stream):
        start.record(stream)
        for _ in range(full):
            g_full.replay()
        if g_rem is not None:
            g_rem.replay()
        end.record(stream)
    torch.cuda.synchronize()
    if world > 1:
        torch.distributed.barrier()
    ms_total = start.elapsed_time(end)
    # keep the device busy until the sampler has seen load
    t_load = time.perf_counter()
    while ms_total < 1500 and time.perf_counter() - t_load < 1.5 and g_full is not None:
        with torch.cuda.stream(stream):
            for _ in range(20):
                g_full.replay()
        torch.cuda.synchronize()
    sampler.stop()
    clocks = sampler.summary()

    ms_total = max_over_ranks(ms_total, world, device)
    ms_step = ms_total / args.steps
    bytes_call = kv_bytes_per_call(kind, inp)
    value = job_gbs(bytes_call, world, ms_step)

    split_ms, reduce_ms = kernel_times(runner, stream, min(2000, max(200, args.steps)), ms_step)
    split_ms = max_over_ranks(split_ms, world, device)
    e2e_ms, h2d, d2h = e2e_measure(runner, stream, min(200, max(20, args.steps)))
    e2e_ms = max_over_ranks(e2e_ms, world, device)
    peak, peak_src = measured_peaks()
    achieved = bytes_call / (split_ms * 1e-3) / 1e9
    traffic = recorded_traffic(args.workload)

    out = {
        "metric": METRIC, "value": round(value, 2), "unit": "GB/s", "n_gpus": world,
        "steps": args.steps, "warmup": args.warmup, "ms_per_step": ms_step,
        "higher_is_better": True, "scaling": "weak",
        "vs_baseline": (round(value / pages_baseline_gbs(args.workload), 3)
                        if pages_baseline_gbs(args.workload) else None),
        "dtype": "e4m3fn-kv/bf16-q(e4m3 hi+mid[+lo])/p(e4m3 hi+lo)/fp32-acc",
        "data": "synthetic (seeded; N(0,1) bf16 queries, N(0,1)/kv_scale e4m3fn pool, shuffled page_size-1 slots)",
        "config": {"workload": workload_label(args.workload, kind, desc),
                   "kv_bytes_per_call": bytes_call, "keys_per_call": keys_per_call(kind, inp),
                   "num_splits": runner.plan.num_splits, "head_blocks": runner.plan.head_blocks,
                   "l2": f"inputs rotated over {copies} device copies "
                         f"({copies * per_copy / 2**20:.0f} MiB > 4x L2 {l2 / 2**20:.0f} MiB)",
                   "timing": "CUDA-graph replays, CUDA events on the launch stream",
                   **({"forced_splits": args.splits} if args.splits else {}),
                   **({"forced_rows_per_cta": args.tile} if args.tile else {}),
                   "rows_per_cta": runner.plan.rows_per_cta,
                   "parallelism": f"replicas x{world}"},
        "us_per_call": ms_step * 1e3,
        "keys_per_s": keys_per_call(kind, inp) * world / (ms_step * 1e-3),
        "hbm_frac_of_measured": round(value / world / peak, 4),
        "hbm_frac_of_spec_8tbs": round(value / world / 8000.0, 4),
        "gpu_launches": args.steps * runner.launches_per_step(),
        "kernels": {"split_ms": split_ms, "rest_ms": reduce_ms,
                    "split_share": split_ms / (split_ms + reduce_ms) if reduce_ms > 0 else 1.0,
                    "timing": "graph replays of split-kernel-only calls; rest = call - split"},
        "roofline": {"bound": "hbm", "achieved": round(achieved, 2), "peak": peak,
                     "unit": "GB/s", "frac": round(achieved / peak, 4), "traffic": traffic,
                     "peak_source": peak_src, "kernel": "split kernel",
                     "algorithmic_bytes": bytes_call},
        "e2e": {"value": round(job_gbs(bytes_call, world, e2e_ms), 2), "unit": "GB/s",
                "us_per_call": e2e_ms * 1e3, "h2d_bytes_per_step": h2d,
                "d2h_bytes_per_step": d2h},
        "clocks": clocks,
        "tflops": flops_per_call(kind, inp) / (ms_step * 1e-3) / 1e12,
    }
    # the oracle baseline runs on rank 0 of a single-GPU run only
    oracle_here = not args.no_cpu_baseline and rank == 0 and world == 1
    if oracle_here:
        out["cpu_baseline"] = cpu_baseline(kind, inp, args.cpu_budget)
    # every workload in single-GPU runs (multi-rank runs time the headline only,
    # unless a list is given)
    if args.workloads != "none" and not (args.workloads == "all" and world > 1):
        names = ALL_WORKLOADS if args.workloads == "all" else args.workloads.split(",")
        del runner
        torch.cuda.empty_cache()
        sweep = {}
        for name in names:
            sweep[name] = measure_workload(
                name, device, world, args.workload_steps,
                args.workload_cpu_budget if oracle_here else 0.0)
        if rank == 0:
            out["workloads"] = sweep
    return out


def run_reference(args, rank, world):
    """The oracle on the host's cores, same workload and metric."""
    if rank != 0:
        return None
    from oracle import oracle
    oracle.build()
    kind, inp, desc = make_workload(args.workload)
    # one step = a bounded sample: the first request (all rows), fixed across steps
    if kind != "sparse":
        heads_rows = inp.q_len * inp.num_heads
        n_req = max(1, min(inp.batch, args.ref_requests))
        keys = int(inp.seq_lens[:n_req].sum())
    else:
        heads_rows = inp.num_heads
        n_req = max(1, min(inp.num_tokens, args.ref_requests))
        keys = int((inp.indices[:n_req] >= 0).sum())
        if inp.extra_topk:
            keys += int((inp.extra_indices[:n_req] >= 0).sum())
    items = list(range(n_req * heads_rows))
    for _ in range(args.warmup):
        _oracle_items(kind, inp, items)
    t0 = time.perf_counter()
    for _ in range(args.steps):
        _oracle_items(kind, inp, items)
    el = time.perf_counter() - t0
    ms_step = el / args.steps * 1e3
    value = keys * row_bytes(kind) / (ms_step * 1e-3) / 1e9
    sample = (f"{n_req} {'token' if kind == 'sparse' else 'request'}(s) of the workload, "
              f"all {heads_rows} rows, per step")
    return {
        "impl": "reference", "metric": METRIC, "value": round(value, 4), "unit": "GB/s",
        "n_gpus": world, "steps": args.steps, "warmup": args.warmup, "ms_per_step": ms_step,
        "higher_is_better": True, "scaling": "weak", "vs_baseline": None, "dtype": "f64",
        "data": "synthetic (seeded, same recipe as the GPU arm)",
        "config": {"workload": workload_label(args.workload, kind, desc),
                   "kv_bytes_per_call": kv_bytes_per_call(kind, inp),
                   "keys_per_call": keys_per_call(kind, inp), "sample": sample},
        "cpu_baseline": {"value": round(value, 4), "unit": "GB/s", "cores": oracle.cpu_threads(),
                         "kind": "oracle", "sample": sample},
        "e2e": {"value": round(value, 4), "unit": "GB/s", "h2d_bytes_per_step": 0,
                "d2h_bytes_per_step": 0},
        "gpu_launches": 0,
    }


def _free_port() -> int:
    import socket
    sk = socket.socket()
    sk.bind(("127.0.0.1", 0))
    port = sk.getsockname()[1]
    sk.close()
    return port


def _rank_entry(rank, world, port, argv, target):
    os.environ.update(RANK=str(rank), LOCAL_RANK=str(rank), WORLD_SIZE=str(world),
                      LOCAL_WORLD_SIZE=str(world), MASTER_ADDR="127.0.0.1",
                      MASTER_PORT=str(port))
    target(argv)


def spawn_ranks(world: int, argv, target=None) -> None:
    """Run `target(argv)` (default: this benchmark) in `world` fresh processes,
    one rank per GPU of this node, as torchrun would: RANK, LOCAL_RANK,
    WORLD_SIZE and a 127.0.0.1 rendezvous in the environment."""
    import torch.multiprocessing as mp
    mp.start_processes(_rank_entry, args=(world, _free_port(), list(argv), target or main),
                       nprocs=world, join=True, start_method="spawn")


def main(argv=None):
    ap = argparse.ArgumentParser(description=__doc__.split("\n")[0])
    ap.add_argument("--gpus", type=int, default=1,
                    help="ranks (one per GPU); without torchrun, spawns that many processes")
    ap.add_argument("--steps", type=int, default=2000)
    ap.add_argument("--warmup", type=int, default=20)
    ap.add_argument("--impl", choices=["ours", "reference"], default="ours")
    ap.add_argument("--workload", default="c1q1")
    ap.add_argument("--cpu-budget", type=float, default=12.0)
    ap.add_argument("--no-cpu-baseline", action="store_true")
    ap.add_argument("--ref-requests", type=int, default=1)
    ap.add_argument("--splits", type=int, default=0,
                    help="force the split count instead of the planner's (split sweeps)")
    ap.add_argument("--tile", type=int, default=0, choices=(0, 16, 32),
                    help="force the query rows per CTA instead of the planner's (tile sweeps)")
    ap.add_argument("--workloads", default="all",
                    help="also time these workloads in the same run: all (single-GPU "
                         "runs), none, or a comma-separated list")
    ap.add_argument("--workload-steps", type=int, default=200)
    ap.add_argument("--workload-cpu-budget", type=float, default=1.5)
    args = ap.parse_args(argv)
    if args.warmup < 3:
        args.warmup = 3

    if "WORLD_SIZE" not in os.environ and args.gpus > 1:
        spawn_ranks(args.gpus, sys.argv[1:] if argv is None else argv)
        return
    world = int(os.environ.get("WORLD_SIZE", "1"))
    rank = int(os.environ.get("RANK", "0"))
    local_rank = int(os.environ.get("LOCAL_RANK", "0"))
    if args.impl == "reference":
        out = run_reference(args, rank, world)
    else:
        if world > 1:
            torch.cuda.set_device(local_rank)
            torch.distributed.init_process_group("nccl", device_id=torch.device("cuda", local_rank))
        out = run_ours(args, rank, world, local_rank)
        if world > 1:
            torch.distributed.destroy_process_group()
    if out is not None and rank == 0:
        print(json.dumps(out), flush=True)


if __name__ == "__main__":
    main()
