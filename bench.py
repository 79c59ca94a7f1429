#!/usr/bin/env python
"""Benchmark of the GB300 attention path (one JSON line on rank 0).

A step is one pass of the whole hot path over one batch of the dense causal
B=2 H=16 L=16384 d=128 workload (bf16 inputs resident in HBM; 537 MB of Q, K,
V and dO, larger than the 129 MB L2):
  1. causal forward                    (attn_fwd: O, LSE)
  2. split-KV forward: 8 KV chunks     (attn_fwd_splitkv: the partial states of
                                        every chunk in one launch, then
                                        attn_merge_states)
  3. block-sparse forward              (attn_fwd_blocksparse, the local + global
                                        + random list over 128 blocks)
  4. backward by recomputation         (attn_bwd: D, dQ, dK, dV)
`value` is the metric's own quantity: the causal forward's algorithmic TFLOP/s
(4d FLOPs per allowed pair) over its CUDA-event time inside the timed steps,
summed over ranks.  `step_tflops` is the whole step's algorithmic TFLOP/s
(10d per allowed pair for the backward).  Sparse pairs/s, the roofline of the
step's dominant kernel (the backward's main kernel, its own launch timed by
CUDA events the library records around it) and of the forward, and the other
workload shapes are reported beside it.

--impl reference times the fp64 CPU oracle's forward on a bounded sample of
the same workload (rows of one head) on the host cores, with the same metric
and unit.  Multi-GPU (torchrun): every rank runs its own batch (independent
heads, no data-path collective; weak scaling); time is the max over ranks.
"""
from __future__ import annotations

import argparse
import dataclasses
import json
import math
import os
import statistics
import subprocess
import sys
import time

ROOT = os.path.dirname(os.path.abspath(__file__))
if ROOT not in sys.path:
    sys.path.insert(0, ROOT)

import numpy as np  # noqa: E402
import torch  # noqa: E402

from workloads import (BWD_8K, CAUSAL_4K, CAUSAL_16K, DECODE_16K, DENSE_SMALL,  # noqa: E402
                       GQA_16K, SPARSE_16K,
                       SPLITKV_128K, Workload, chunk_bounds, local_global_random_blocklist,
                       make_inputs)

METRIC = "attention fwd TFLOP/s (bf16) and % of GB300 tensor-core peak; sparse pairs/s"
UNIT = "TFLOP/s"
L2_BYTES = 129 * 1024 * 1024


# ---------------------------------------------------------------------------
# Work accounting (logical allowed pairs and executed tiles)
# ---------------------------------------------------------------------------

def causal_pairs(Lq, Lk, q0=0, k0=0):
    """Number of (i, j), i < Lq, j < Lk with j + k0 <= i + q0."""
    i = np.arange(Lq, dtype=np.int64)
    return int(np.clip(i + q0 - k0 + 1, 0, Lk).sum())


def sparse_counts(L, row_ptr, col_idx, causal, block=128):
    """(logical pairs, executed 128x128 tiles) of a block list with set semantics."""
    n = (L + block - 1) // block
    pairs = tiles = 0
    for a in range(n):
        r0, r1 = a * block, min(L, (a + 1) * block)
        for c in set(int(x) for x in col_idx[row_ptr[a]:row_ptr[a + 1]]):
            k0, k1 = c * block, min(L, (c + 1) * block)
            if causal:
                i = np.arange(r0, r1)
                cnt = int(np.clip(np.minimum(i, k1 - 1) - k0 + 1, 0, None).sum())
            else:
                cnt = (r1 - r0) * (k1 - k0)
            if cnt:
                pairs += cnt
                tiles += 1
    return pairs, tiles


# ---------------------------------------------------------------------------
# Environment helpers
# ---------------------------------------------------------------------------

def load_peaks():
    path = os.path.join(ROOT, "MEASURED_PEAKS.json")
    if os.path.exists(path):
        with open(path) as f:
            pk = json.load(f)
        return {"bf16_burst": pk["bf16_tflops"], "bf16_sustained": pk["bf16_tflops_sustained"],
                "hbm_gbs": pk["hbm_gbs"], "source": "measured"}
    return {"bf16_burst": 1900.0, "bf16_sustained": 1700.0, "hbm_gbs": 6800.0, "source": "fallback"}


# The kernels behind each row of the step, and the sources that define the
# kernel whose DRAM traffic is reported (the traffic recorded for a kernel is
# used only while those sources are unchanged).
KERNEL_OF_ROW = {
    "fwd": "attn_fwd_wide_kernel (causal, persistent, 256-key score tiles): the whole attn_fwd call",
    "splitkv": "attn_fwd_kernel (partial, 8 key chunks in one launch) + merge_states_kernel",
    "sparse": "attn_fwd_wide_kernel (block-sparse, 256-key score tiles)",
    "bwd": "attn_bwd call: attn_bwd_preprocess_kernel + attn_bwd_main_kernel + "
           "attn_bwd_dq_convert_kernel (timed together)",
}
# The dominant row's own kernel where the row's call launches more than one:
# the backward's main kernel, timed by the CUDA events attn_bwd records around
# its launch (attn_bwd_time_main).
MAIN_KERNEL_OF_ROW = {"bwd": "attn_bwd_main_kernel: its own launch, between CUDA events the "
                             "library records around it inside attn_bwd (preprocess and dQ "
                             "conversion excluded)"}
TRAFFIC_KERNEL = {"fwd": "attn_fwd_wide_kernel", "bwd": "attn_bwd_main_kernel"}
KERNEL_SOURCES = {"attn_fwd_wide_kernel": ["fwd_wide.cu", "common.cuh", "ptx.cuh"],
                  "attn_bwd_main_kernel": ["bwd.cu", "common.cuh", "ptx.cuh"]}
STEP_WORKLOAD = CAUSAL_16K


def kernel_source_hash(kernel: str) -> str:
    import hashlib
    h = hashlib.sha256()
    for f in KERNEL_SOURCES[kernel]:
        with open(os.path.join(ROOT, "block_sparse_softmax_gb300", "csrc", f), "rb") as fh:
            h.update(fh.read())
    return h.hexdigest()


def dram_traffic(row: str):
    """DRAM bytes (read + write) per launch of the row's dominant kernel, from
    the ncu capture summarised in profiles/traffic.json, or None when there is
    none or the kernel's sources changed after it was taken."""
    kernel = TRAFFIC_KERNEL.get(row)
    path = os.path.join(ROOT, "profiles", "traffic.json")
    if kernel is None or not os.path.exists(path):
        return None, "no ncu capture of this kernel"
    with open(path) as f:
        rec = json.load(f).get(f"{kernel}@{STEP_WORKLOAD.name}")
    if rec is None:
        return None, "no ncu capture of this kernel on the step's workload"
    if rec.get("source_sha256") != kernel_source_hash(kernel):
        return None, "kernel changed since the ncu capture"
    return rec["dram_bytes_per_launch"], rec.get("capture", "")


class ClockSampler:
    """nvidia-smi samples of SM clock and throttle reasons during a timed region."""
    FIELDS = ("index,clocks.sm,clocks.max.sm,power.draw,clocks_event_reasons.active,"
              "clocks_event_reasons.hw_slowdown,clocks_event_reasons.hw_thermal_slowdown,"
              "clocks_event_reasons.sw_thermal_slowdown,clocks_event_reasons.sw_power_cap")

    def __init__(self, device_index: int):
        self.idx = device_index
        self.proc = None
        self.path = os.path.join("/tmp", f"bss_clocks_{os.getpid()}.csv")

    def start(self):
        try:
            self.fh = open(self.path, "w")
            self.proc = subprocess.Popen(
                ["nvidia-smi", f"--id={self.idx}", f"--query-gpu={self.FIELDS}",
                 "--format=csv,noheader,nounits", "-lms", "20"], stdout=self.fh,
                stderr=subprocess.DEVNULL)
        except (OSError, FileNotFoundError):
            self.proc = None
            return
        # nvidia-smi takes a while to start: wait (up to 3 s) for its first
        # sample so that the timed region is covered from its beginning
        t0 = time.time()
        while time.time() - t0 < 3.0 and self.proc.poll() is None:
            self.fh.flush()
            if os.path.getsize(self.path) > 0:
                break
            time.sleep(0.02)

    def stop(self):
        if self.proc is None:
            return {"sm_mhz": None, "sm_max_mhz": None, "reasons": ["nvidia-smi unavailable"]}
        self.proc.terminate()
        try:
            self.proc.wait(timeout=5)
        except subprocess.TimeoutExpired:
            self.proc.kill()
        self.fh.close()
        sm, smax, reasons = [], None, set()
        names = ["hw_slowdown", "hw_thermal_slowdown", "sw_thermal_slowdown", "sw_power_cap"]
        with open(self.path) as f:
            for line in f:
                parts = [p.strip() for p in line.split(",")]
                if len(parts) < 9:
                    continue
                try:
                    sm.append(float(parts[1]))
                    smax = float(parts[2])
                except ValueError:
                    continue
                for n_, v in zip(names, parts[5:9]):
                    if v.lower() == "active":
                        reasons.add(n_)
        os.remove(self.path)
        if not sm:
            return {"sm_mhz": None, "sm_max_mhz": smax, "reasons": ["no samples"]}
        busy = [x for x in sm if smax and x > 0.5 * smax] or sm
        return {"sm_mhz": statistics.median(busy), "sm_max_mhz": smax, "samples": len(sm),
                "reasons": sorted(reasons)}


def dist_setup():
    world = int(os.environ.get("WORLD_SIZE", "1"))
    rank = int(os.environ.get("RANK", "0"))
    local = int(os.environ.get("LOCAL_RANK", "0"))
    return rank, world, local


def rank_workload(w: Workload, rank: int) -> Workload:
    """This rank's share of an N-rank job: the same shape with a batch of its
    own (seed offset by the rank), so that N ranks process N independent
    batches and no data moves between them (weak scaling)."""
    return w if rank == 0 else dataclasses.replace(w, seed=w.seed + 1000 * rank)


def max_over_ranks(x: float, device) -> float:
    """The largest value of x over the ranks of the default process group."""
    import torch.distributed as dist
    t = torch.tensor([float(x)], device=device)
    dist.all_reduce(t, op=dist.ReduceOp.MAX)
    return float(t.item())


def job_throughput(flops_per_rank: float, ms_max: float, world: int) -> float:
    """Whole-job TFLOP/s: the work of every rank over the slowest rank's time."""
    return world * flops_per_rank / ms_max / 1e9


# ---------------------------------------------------------------------------
# The GPU step
# ---------------------------------------------------------------------------

class Step:
    """All rows of the hot path on one batch; buffers preallocated."""

    ROWS = ("fwd", "splitkv", "sparse", "bwd")

    def __init__(self, bss, w: Workload, dev, cpu=None):
        self.bss = bss
        self.w = w
        B, H, L, d = w.B, w.H, w.L, w.d
        if cpu is None:
            cpu = make_inputs(Workload(w.name, B, H, L, d, True, w.seed, backward=True))
        self.cpu = cpu
        self.dev = {k: v.to(dev) for k, v in cpu.items()}
        self.o = torch.empty_like(self.dev["q"])
        self.lse = torch.empty((B, H, L), device=dev)
        self.n_chunks = 8
        self.ws_split = torch.empty(bss.attn_fwd_splitkv_workspace_bytes(B, H, L, L, d, self.n_chunks),
                                    device=dev, dtype=torch.uint8)
        self.o_split = torch.empty_like(self.o)
        self.lse_split = torch.empty_like(self.lse)
        nblk = (L + 127) // 128
        self.row_ptr, self.col_idx = local_global_random_blocklist(nblk, seed=2)
        self.rp_dev = torch.from_numpy(self.row_ptr).to(dev)
        self.ci_dev = torch.from_numpy(self.col_idx).to(dev)
        self.o_sparse = torch.empty_like(self.o)
        self.lse_sparse = torch.empty_like(self.lse)
        self.dq = torch.empty_like(self.o)
        self.dk = torch.empty_like(self.o)
        self.dv = torch.empty_like(self.o)
        self.delta = torch.empty_like(self.lse)
        self.ws = torch.empty(bss.attn_bwd_workspace_bytes(B, H, L, d), device=dev, dtype=torch.uint8)
        # work per step
        heads = B * H
        self.pairs_causal = heads * causal_pairs(L, L)
        sp, st = sparse_counts(L, self.row_ptr, self.col_idx, True)
        self.pairs_sparse, self.tiles_sparse = heads * sp, heads * st
        self.flops = {
            "fwd": 4 * d * self.pairs_causal,
            "splitkv": 4 * d * self.pairs_causal,
            "sparse": 4 * d * self.pairs_sparse,
            "bwd": 10 * d * self.pairs_causal,
        }
        self.total_flops = sum(self.flops.values())
        self.launches = {"fwd": 1, "splitkv": 2, "sparse": 1, "bwd": 3}
        self.launches_per_step = sum(self.launches.values())
        self.events = None

    def run_fwd(self):
        d, w = self.dev, self.w
        self.bss.attn_fwd(d["q"], d["k"], d["v"], causal=True, scale=w.scale, out=self.o,
                          lse=self.lse)

    def run(self, timed_rows=False):
        bss, d, w = self.bss, self.dev, self.w
        ev = self.events if timed_rows else None
        if ev is not None:
            ev["fwd"][0].record()
        self.run_fwd()
        if ev is not None:
            ev["fwd"][1].record()
            ev["splitkv"][0].record()
        bss.attn_fwd_splitkv(d["q"], d["k"], d["v"], self.n_chunks, causal=True, scale=w.scale,
                             workspace=self.ws_split, out=self.o_split, lse=self.lse_split)
        if ev is not None:
            ev["splitkv"][1].record()
            ev["sparse"][0].record()
        bss.attn_fwd_blocksparse(d["q"], d["k"], d["v"], self.rp_dev, self.ci_dev, causal=True,
                                 scale=w.scale, out=self.o_sparse, lse=self.lse_sparse)
        if ev is not None:
            ev["sparse"][1].record()
            ev["bwd"][0].record()
            # the backward's main kernel alone: events the library records
            # around its launch inside attn_bwd
            bss.attn_bwd_time_main(*self.main_events)
        bss.attn_bwd(d["q"], d["k"], d["v"], self.o, self.lse, d["do"], causal=True,
                     scale=w.scale, workspace=self.ws, dq=self.dq, dk=self.dk, dv=self.dv,
                     delta=self.delta)
        if ev is not None:
            bss.attn_bwd_time_main()
            ev["bwd"][1].record()

    def new_events(self):
        self.events = {k: (torch.cuda.Event(enable_timing=True), torch.cuda.Event(enable_timing=True))
                       for k in self.flops}
        self.main_events = (torch.cuda.Event(enable_timing=True),
                            torch.cuda.Event(enable_timing=True))


def time_loop(fn, steps, warmup, sync_all):
    for _ in range(warmup):
        fn(False)
    torch.cuda.synchronize()
    sync_all()
    start = torch.cuda.Event(enable_timing=True)
    end = torch.cuda.Event(enable_timing=True)
    start.record()
    for _ in range(steps):
        fn(True)
    end.record()
    torch.cuda.synchronize()
    sync_all()
    return start.elapsed_time(end) / steps


def e2e_pipelined_ms(sets, host_in, host_outs, out_names, compute_fn, steps, warmup, sync_all):
    """Milliseconds per step end to end through the public API: every step
    uploads its inputs from pinned host memory and downloads its results to
    pinned host memory, all inside the timed region.  The copies run on one
    stream per direction and overlap the neighbouring steps' compute: step k+1
    uploads into one of two device buffer sets while step k computes on the
    other and step k-1's results come down.  ``compute_fn(set)`` runs a step's
    calls on a buffer set; ``out_names`` are the set's result attributes."""
    comp = torch.cuda.current_stream()
    up, down = torch.cuda.Stream(), torch.cuda.Stream()
    ev_up = [torch.cuda.Event() for _ in range(2)]      # set s: inputs uploaded
    ev_comp = [torch.cuda.Event() for _ in range(2)]    # set s: step computed
    ev_down = [torch.cuda.Event() for _ in range(2)]    # set s: results downloaded

    def upload(k):
        s = k % 2
        with torch.cuda.stream(up):
            if k >= 2:
                up.wait_event(ev_comp[s])               # set s's inputs no longer read
            for n, t in host_in.items():
                sets[s].dev[n].copy_(t, non_blocking=True)
            ev_up[s].record(up)

    def compute(k):
        s = k % 2
        comp.wait_event(ev_up[s])
        if k >= 2:
            comp.wait_event(ev_down[s])                 # set s's results already copied out
        compute_fn(sets[s])
        ev_comp[s].record(comp)

    def download(k):
        s = k % 2
        st, ho = sets[s], host_outs[s]
        with torch.cuda.stream(down):
            down.wait_event(ev_comp[s])
            for n in out_names:
                ho[n].copy_(getattr(st, n), non_blocking=True)
            ev_down[s].record(down)

    def run(n, start=None, end=None):
        if start is not None:
            start.record(comp)
        up.wait_stream(comp)
        down.wait_stream(comp)
        upload(0)
        for k in range(n):
            if k + 1 < n:
                upload(k + 1)
            compute(k)
            download(k)
        comp.wait_stream(up)
        comp.wait_stream(down)
        if end is not None:
            end.record(comp)

    run(max(2, warmup))
    torch.cuda.synchronize()
    sync_all()
    start = torch.cuda.Event(enable_timing=True)
    end = torch.cuda.Event(enable_timing=True)
    run(steps, start, end)
    torch.cuda.synchronize()
    sync_all()
    return start.elapsed_time(end) / steps


def bench_kernel(fn, reps=10, warmup=3):
    """Median device time of fn() between CUDA events on the current stream.
    A ~1 ms device sleep queued ahead of each start event keeps the GPU busy
    while the host enqueues the call, so the events bracket device work only
    (not the binding's host time)."""
    for _ in range(warmup):
        fn()
    torch.cuda.synchronize()
    s, e = torch.cuda.Event(enable_timing=True), torch.cuda.Event(enable_timing=True)
    times = []
    for _ in range(reps):
        torch.cuda._sleep(2_000_000)
        s.record()
        fn()
        e.record()
        torch.cuda.synchronize()
        times.append(s.elapsed_time(e))
    return statistics.median(times)


def measure_configs(bss, dev, peaks):
    """Each workload shape of the study, timed on its own (not part of `value`)."""
    out = {}
    pk = peaks["bf16_burst"]
    # the exponential unit: the forward takes one ex2 per pair, a second
    # ceiling beside the tensor core's (4 d FLOPs per pair at the ex2 rate)
    sms = torch.cuda.get_device_properties(dev).multi_processor_count
    blocks, iters = sms * 8, 2048
    sink = torch.zeros(1, device=dev)
    n_ex2 = blocks * 256 * 8 * iters
    ms_x = bench_kernel(lambda: bss.attn_probe_ex2_rate(blocks, iters, sink=sink), reps=10)
    ex2_rate = n_ex2 / (ms_x * 1e-3)
    out["ex2_rate"] = {"ex2_per_s": float(f"{ex2_rate:.4g}"),
                       "per_sm_per_clock_at_2070mhz": round(ex2_rate / (sms * 2070e6), 2),
                       "fwd_tflops_ceiling": {"d64": round(4 * 64 * ex2_rate / 1e12, 1),
                                              "d128": round(4 * 128 * ex2_rate / 1e12, 1)}}
    # dense L=256 d=64: latency
    w = DENSE_SMALL
    x = {k: t.to(dev) for k, t in make_inputs(w).items()}
    ms = bench_kernel(lambda: bss.attn_fwd(x["q"], x["k"], x["v"], scale=w.scale), reps=50)
    out[w.name] = {"us": round(ms * 1e3, 2)}
    # dense causal target at L=16384, timed alone (the step times it in place)
    w = CAUSAL_16K
    x = {k: t.to(dev) for k, t in make_inputs(w).items()}
    o = torch.empty_like(x["q"])
    lse = torch.empty(w.B, w.H, w.L, device=dev)
    ms = bench_kernel(lambda: bss.attn_fwd(x["q"], x["k"], x["v"], causal=True, scale=w.scale,
                                           out=o, lse=lse), reps=20)
    fl = 4 * w.d * w.B * w.H * causal_pairs(w.L, w.L)
    tf = fl / ms / 1e9
    out[w.name] = {"ms": round(ms, 4), "tflops": round(tf, 1), "frac_burst": round(tf / pk, 4),
                   "frac_sustained": round(tf / peaks["bf16_sustained"], 4),
                   "frac_ex2_ceiling": round(tf / (4 * w.d * ex2_rate / 1e12), 4),
                   "target_frac": 0.6}
    del x, o, lse
    # causal B=4 H=16 L=4096 d=128: forward, 8-chunk split-KV, backward
    w = CAUSAL_4K
    x = {k: t.to(dev) for k, t in make_inputs(
        Workload(w.name, w.B, w.H, w.L, w.d, True, w.seed, backward=True)).items()}
    o = torch.empty_like(x["q"])
    lse = torch.empty(w.B, w.H, w.L, device=dev)
    ms_f = bench_kernel(lambda: bss.attn_fwd(x["q"], x["k"], x["v"], causal=True, scale=w.scale,
                                             out=o, lse=lse), reps=20)
    ws = torch.empty(bss.attn_fwd_splitkv_workspace_bytes(w.B, w.H, w.L, w.L, w.d, 8),
                     device=dev, dtype=torch.uint8)
    o2, lse2 = torch.empty_like(o), torch.empty_like(lse)
    ms_s = bench_kernel(lambda: bss.attn_fwd_splitkv(x["q"], x["k"], x["v"], 8, causal=True,
                                                     scale=w.scale, workspace=ws, out=o2,
                                                     lse=lse2), reps=20)
    wsb = torch.empty(bss.attn_bwd_workspace_bytes(w.B, w.H, w.L, w.d), device=dev,
                      dtype=torch.uint8)
    g = [torch.empty_like(x["q"]) for _ in range(3)]
    dl = torch.empty_like(lse)
    ms_b = bench_kernel(lambda: bss.attn_bwd(x["q"], x["k"], x["v"], o, lse, x["do"], causal=True,
                                             scale=w.scale, workspace=wsb, dq=g[0], dk=g[1],
                                             dv=g[2], delta=dl), reps=20)
    pairs = w.B * w.H * causal_pairs(w.L, w.L)
    out[w.name] = {"fwd_ms": round(ms_f, 4), "fwd_tflops": round(4 * w.d * pairs / ms_f / 1e9, 1),
                   "fwd_frac_burst": round(4 * w.d * pairs / ms_f / 1e9 / pk, 4),
                   "splitkv8_ms": round(ms_s, 4),
                   "splitkv8_tflops": round(4 * w.d * pairs / ms_s / 1e9, 1),
                   "bwd_ms": round(ms_b, 4), "bwd_tflops": round(10 * w.d * pairs / ms_b / 1e9, 1),
                   "bwd_frac_burst": round(10 * w.d * pairs / ms_b / 1e9 / pk, 4)}
    del x, o, lse, ws, o2, lse2, wsb, g, dl
    # block-sparse L'=16320
    w = SPARSE_16K
    x = {k: t.to(dev) for k, t in make_inputs(w).items()}
    rp, ci = local_global_random_blocklist(w.n_blocks, seed=w.seed)
    rpd, cid = torch.from_numpy(rp).to(dev), torch.from_numpy(ci).to(dev)
    o = torch.empty_like(x["q"])
    lse = torch.empty(w.B, w.H, w.L, device=dev)
    ms = bench_kernel(lambda: bss.attn_fwd_blocksparse(x["q"], x["k"], x["v"], rpd, cid,
                                                       causal=True, scale=w.scale, out=o, lse=lse))
    pairs, tiles = sparse_counts(w.L, rp, ci, True)
    pairs *= w.B * w.H
    tiles *= w.B * w.H
    # its backward (attn_bwd_blocksparse), from the forward's O and LSE
    do = make_inputs(Workload(w.name, w.B, w.H, w.L, w.d, True, w.seed, backward=True))["do"].to(dev)
    ws = torch.empty(bss.attn_bwd_blocksparse_workspace_bytes(w.B, w.H, w.L, w.d), device=dev,
                     dtype=torch.uint8)
    g = [torch.empty_like(x["q"]) for _ in range(3)]
    dl = torch.empty_like(lse)
    ms_b = bench_kernel(lambda: bss.attn_bwd_blocksparse(
        x["q"], x["k"], x["v"], o, lse, do, rpd, cid, causal=True, scale=w.scale, workspace=ws,
        dq=g[0], dk=g[1], dv=g[2], delta=dl))
    out[w.name] = {"ms": round(ms, 4), "logical_pairs": pairs, "executed_tiles": tiles,
                   "pairs_per_s": pairs / ms * 1e3,
                   "tflops_logical": round(4 * w.d * pairs / ms / 1e9, 1),
                   "tflops_executed": round(4 * w.d * tiles * 128 * 128 / ms / 1e9, 1),
                   "bwd_ms": round(ms_b, 4),
                   "bwd_tflops_logical": round(10 * w.d * pairs / ms_b / 1e9, 1)}
    del do, ws, g, dl
    # the same inputs with long lists (16 local and 8 random blocks a row,
    # about 24 raw entries): at d=128 the kernel with 256-key score tiles
    lrp, lci = local_global_random_blocklist(w.n_blocks, seed=w.seed, n_local=16, n_random=8)
    lrpd, lcid = torch.from_numpy(lrp).to(dev), torch.from_numpy(lci).to(dev)
    ms_l = bench_kernel(lambda: bss.attn_fwd_blocksparse(x["q"], x["k"], x["v"], lrpd, lcid,
                                                         causal=True, scale=w.scale, out=o,
                                                         lse=lse))
    lpairs, ltiles = sparse_counts(w.L, lrp, lci, True)
    lpairs *= w.B * w.H
    ltiles *= w.B * w.H
    out[w.name]["long_lists"] = {
        "entries_per_row": round(len(lci) / w.n_blocks, 1), "ms": round(ms_l, 4),
        "logical_pairs": lpairs, "executed_tiles": ltiles, "pairs_per_s": lpairs / ms_l * 1e3,
        "tflops_logical": round(4 * w.d * lpairs / ms_l / 1e9, 1),
        "tflops_executed": round(4 * w.d * ltiles * 128 * 128 / ms_l / 1e9, 1)}
    del lrpd, lcid
    # mean-pooled selector on the same inputs: one list per head of the 4 local
    # and 4 best-scoring blocks; HBM-bound (Q and K read once for the block
    # means), then the block-sparse forward on the lists it chose
    n_lists = w.B * w.H
    sel_ws = torch.empty(bss.attn_select_blocks_workspace_bytes(w.B, w.H, w.L, w.d), device=dev,
                         dtype=torch.uint8)
    ms_sel = bench_kernel(lambda: bss.attn_select_blocks(
        x["q"], x["k"], 4, local_blocks=4, causal=True, n_lists=n_lists, scale=w.scale,
        workspace=sel_ws), reps=20)
    srp, sci = bss.attn_select_blocks(x["q"], x["k"], 4, local_blocks=4, causal=True,
                                      n_lists=n_lists, scale=w.scale, workspace=sel_ws)
    ms_sf = bench_kernel(lambda: bss.attn_fwd_blocksparse(x["q"], x["k"], x["v"], srp, sci,
                                                          causal=True, scale=w.scale, out=o,
                                                          lse=lse))
    sel_bytes = 2 * w.B * w.H * w.L * w.d * 2
    sel_tiles = int(sci.numel())
    out["selector_" + w.name] = {
        "select_ms": round(ms_sel, 4), "select_gbs": round(sel_bytes / ms_sel / 1e6, 1),
        "select_frac_hbm": round(sel_bytes / ms_sel / 1e6 / peaks["hbm_gbs"], 4),
        "lists": n_lists, "entries": sel_tiles, "sparse_fwd_ms": round(ms_sf, 4),
        "sparse_fwd_tflops_executed": round(4 * w.d * sel_tiles * 128 * 128 / ms_sf / 1e9, 1),
        "select_share": round(ms_sel / (ms_sel + ms_sf), 4)}
    del x, o, lse, sel_ws, srp, sci
    # split-KV L=131072, 8 chunks + merge
    w = SPLITKV_128K
    x = {k: t.to(dev) for k, t in make_inputs(w).items()}
    bounds = chunk_bounds(w.L, w.chunks)
    kc = [x["k"][:, :, s:e].contiguous() for s, e in bounds]
    vc = [x["v"][:, :, s:e].contiguous() for s, e in bounds]
    C = len(bounds)
    m = torch.empty(C, w.B, w.H, w.L, device=dev)
    l_ = torch.empty_like(m)
    acc = torch.empty(C, w.B, w.H, w.L, w.d, device=dev)
    o = torch.empty_like(x["q"])
    lse = torch.empty(w.B, w.H, w.L, device=dev)

    def partials():
        for c, (s, _) in enumerate(bounds):
            bss.attn_fwd_partial(x["q"], kc[c], vc[c], causal=True, scale=w.scale, k_offset=s,
                                 m=m[c], l=l_[c], acc=acc[c])

    ms_p = bench_kernel(partials, reps=5, warmup=1)
    ms_m = bench_kernel(lambda: bss.attn_merge_states(m, l_, acc, out=o, lse=lse), reps=10)
    del m, l_, acc, kc, vc
    # the same in one split-KV launch (chunks read in place) + merge
    ws = torch.empty(bss.attn_fwd_splitkv_workspace_bytes(w.B, w.H, w.L, w.L, w.d, w.chunks),
                     device=dev, dtype=torch.uint8)
    ms_s = bench_kernel(lambda: bss.attn_fwd_splitkv(x["q"], x["k"], x["v"], w.chunks, causal=True,
                                                     scale=w.scale, workspace=ws, out=o, lse=lse),
                        reps=5, warmup=1)
    fl = 4 * w.d * w.B * w.H * causal_pairs(w.L, w.L)
    rows = w.B * w.H * w.L
    nonempty = sum(w.B * w.H * max(0, w.L - s) for s, _ in bounds)
    merge_bytes = C * rows * 8 + nonempty * w.d * 4 + rows * (w.d * 2 + 4)
    out[w.name] = {"splitkv_ms": round(ms_s, 3), "tflops": round(fl / ms_s / 1e9, 1),
                   "per_chunk_launches_ms": round(ms_p + ms_m, 3),
                   "merge_ms": round(ms_m, 4),
                   "merge_gbs": round(merge_bytes / ms_m / 1e6, 1),
                   "merge_frac_hbm": round(merge_bytes / ms_m / 1e6 / peaks["hbm_gbs"], 4)}
    del x, o, lse, ws
    # decode-shaped: 16 queries at the end of a 16384-key causal cache, 16 chunks
    w = DECODE_16K
    x = {k: t.to(dev) for k, t in make_inputs(w).items()}
    o = torch.empty_like(x["q"])
    lse = torch.empty(w.B, w.H, w.Lq, device=dev)
    ws = torch.empty(bss.attn_fwd_splitkv_workspace_bytes(w.B, w.H, w.Lq, w.L, w.d, w.chunks),
                     device=dev, dtype=torch.uint8)
    qo = w.L - w.Lq
    ms_d = bench_kernel(lambda: bss.attn_fwd_splitkv(x["q"], x["k"], x["v"], w.chunks, causal=True,
                                                     scale=w.scale, q_offset=qo, workspace=ws,
                                                     out=o, lse=lse), reps=20)
    ms_1 = bench_kernel(lambda: bss.attn_fwd(x["q"], x["k"], x["v"], causal=True, scale=w.scale,
                                             q_offset=qo, out=o, lse=lse), reps=10)
    pairs = w.B * w.H * causal_pairs(w.Lq, w.L, q0=qo)
    kv_bytes = 2 * w.B * w.H * w.L * w.d * 2
    out[w.name] = {"ms": round(ms_d, 4), "unsplit_ms": round(ms_1, 4),
                   "tflops": round(4 * w.d * pairs / ms_d / 1e9, 2),
                   "kv_gbs": round(kv_bytes / ms_d / 1e6, 1),
                   "kv_frac_hbm": round(kv_bytes / ms_d / 1e6 / peaks["hbm_gbs"], 4)}
    del x, o, lse, ws
    # fwd + bwd L=8192 d=64
    w = BWD_8K
    x = {k: t.to(dev) for k, t in make_inputs(w).items()}
    o = torch.empty_like(x["q"])
    lse = torch.empty(w.B, w.H, w.L, device=dev)
    ws = torch.empty(bss.attn_bwd_workspace_bytes(w.B, w.H, w.L, w.d), device=dev, dtype=torch.uint8)
    g = [torch.empty_like(x["q"]) for _ in range(3)]
    dl = torch.empty_like(lse)
    ms_f = bench_kernel(lambda: bss.attn_fwd(x["q"], x["k"], x["v"], causal=True, scale=w.scale,
                                             out=o, lse=lse))
    ms_b = bench_kernel(lambda: bss.attn_bwd(x["q"], x["k"], x["v"], o, lse, x["do"], causal=True,
                                             scale=w.scale, workspace=ws, dq=g[0], dk=g[1],
                                             dv=g[2], delta=dl))
    pairs = w.B * w.H * causal_pairs(w.L, w.L)
    out[w.name] = {"fwd_ms": round(ms_f, 4), "bwd_ms": round(ms_b, 4),
                   "fwd_tflops": round(4 * w.d * pairs / ms_f / 1e9, 1),
                   "bwd_tflops": round(10 * w.d * pairs / ms_b / 1e9, 1),
                   "fwd_frac_ex2_ceiling": round(pairs / (ms_f * 1e-3) / ex2_rate, 4)}
    del x, o, lse, ws, g, dl
    # grouped key/value heads: 16 query heads over 4 shared K/V heads, L=16384
    w = GQA_16K
    x = {k: t.to(dev) for k, t in make_inputs(w).items()}
    o = torch.empty_like(x["q"])
    lse = torch.empty(w.B, w.H, w.L, device=dev)
    ws = torch.empty(bss.attn_bwd_workspace_bytes(w.B, w.H, w.L, w.d), device=dev, dtype=torch.uint8)
    g = [torch.empty_like(x["q"]), torch.empty_like(x["k"]), torch.empty_like(x["v"])]
    dl = torch.empty_like(lse)
    ms_f = bench_kernel(lambda: bss.attn_fwd(x["q"], x["k"], x["v"], causal=True, scale=w.scale,
                                             out=o, lse=lse), reps=10)
    ms_b = bench_kernel(lambda: bss.attn_bwd(x["q"], x["k"], x["v"], o, lse, x["do"], causal=True,
                                             scale=w.scale, workspace=ws, dq=g[0], dk=g[1],
                                             dv=g[2], delta=dl), reps=10)
    pairs = w.B * w.H * causal_pairs(w.L, w.L)
    out[w.name] = {"fwd_ms": round(ms_f, 4), "bwd_ms": round(ms_b, 4),
                   "fwd_tflops": round(4 * w.d * pairs / ms_f / 1e9, 1),
                   "bwd_tflops": round(10 * w.d * pairs / ms_b / 1e9, 1),
                   "fwd_frac_burst": round(4 * w.d * pairs / ms_f / 1e9 / pk, 4),
                   "fwd_frac_ex2_ceiling": round(pairs / (ms_f * 1e-3) / ex2_rate, 4)}
    return out


def run_gpu(args):
    rank, world, local = dist_setup()
    torch.cuda.set_device(local)
    dev = torch.device("cuda", local)
    if world > 1:
        import torch.distributed as dist
        dist.init_process_group("nccl", device_id=dev)

        def sync_all():
            dist.barrier()
    else:
        def sync_all():
            pass
    import block_sparse_softmax_gb300 as bss
    bss.library()
    peaks = load_peaks()
    w = rank_workload(STEP_WORKLOAD, rank)
    step = Step(bss, w, dev)
    # warm-up, then the timed region (device-resident inputs); every row of
    # every step is bracketed by CUDA events on the launching stream
    clocks = ClockSampler(local)
    for _ in range(args.warmup):
        step.run()
    torch.cuda.synchronize()
    sync_all()
    events, main_events = [], []
    for _ in range(args.steps):
        step.new_events()
        events.append(step.events)
        main_events.append(step.main_events)
    clocks.start()
    t0 = time.time()
    start = torch.cuda.Event(enable_timing=True)
    end = torch.cuda.Event(enable_timing=True)
    start.record()
    for i in range(args.steps):
        step.events = events[i]
        step.main_events = main_events[i]
        step.run(timed_rows=True)
    end.record()
    torch.cuda.synchronize()
    sync_all()
    wall = time.time() - t0
    clock_info = clocks.stop()
    ms_step = start.elapsed_time(end) / args.steps
    row_avg = {k: statistics.mean(ev[k][0].elapsed_time(ev[k][1]) for ev in events)
               for k in step.flops}
    ms_bwd_main = statistics.mean(a.elapsed_time(b) for a, b in main_events)
    ms_fwd = row_avg["fwd"]
    if world > 1:
        ms_step = max_over_ranks(ms_step, dev)
        ms_fwd = max_over_ranks(ms_fwd, dev)

    # end to end through the public API, pinned host buffers in and out, copies
    # overlapping the neighbouring steps (a second device buffer set):
    #   the metric's own operation: upload Q, K, V; attn_fwd; download O, LSE
    #   the whole step: upload Q, K, V, dO; every row; download O, LSE, dQ, dK, dV
    sets = [step, Step(bss, w, dev, cpu=step.cpu)]
    fwd_in = {n: step.cpu[n].pin_memory() for n in ("q", "k", "v")}
    step_in = {**fwd_in, "do": step.cpu["do"].pin_memory()}

    def host_like(names):
        return [{n: torch.empty(getattr(step, n).shape, dtype=getattr(step, n).dtype).pin_memory()
                 for n in names} for _ in range(2)]

    fwd_out_names, step_out_names = ("o", "lse"), ("o", "lse", "dq", "dk", "dv")
    fwd_outs, step_outs = host_like(fwd_out_names), host_like(step_out_names)
    nbytes = lambda d: sum(t.numel() * t.element_size() for t in d.values())
    n_e2e = max(3, args.steps // 2)
    ms_e2e = e2e_pipelined_ms(sets, fwd_in, fwd_outs, fwd_out_names, Step.run_fwd, n_e2e, 2,
                              sync_all)
    ms_e2e_step = e2e_pipelined_ms(sets, step_in, step_outs, step_out_names, Step.run, n_e2e, 2,
                                   sync_all)

    # the forward with no overlap: upload, attn_fwd, download on one stream
    def e2e_serial(_timed):
        for n, t in fwd_in.items():
            step.dev[n].copy_(t, non_blocking=True)
        step.run_fwd()
        for n in fwd_out_names:
            fwd_outs[0][n].copy_(getattr(step, n), non_blocking=True)

    ms_e2e_serial = time_loop(e2e_serial, n_e2e, 2, sync_all)
    del sets
    if world > 1:
        ms_e2e = max_over_ranks(ms_e2e, dev)
        ms_e2e_step = max_over_ranks(ms_e2e_step, dev)
        ms_e2e_serial = max_over_ranks(ms_e2e_serial, dev)
    status = bss.attn_poll_status()
    # the step's block list as the library counts it (listed, executed,
    # causal-future blocks, allowed pairs), beside the host accounting
    list_stats = bss.attn_blocklist_stats(step.rp_dev, step.ci_dev, w.L, causal=True).cpu().tolist()[0]

    pk_b, pk_s = peaks["bf16_burst"], peaks["bf16_sustained"]
    value = job_throughput(step.flops["fwd"], ms_fwd, world)
    step_tf = job_throughput(step.total_flops, ms_step, world)
    row_tf = {k: step.flops[k] / row_avg[k] / 1e9 for k in step.flops}
    # dominant kernel: the largest share of the step's time; for the backward
    # row its main kernel, timed by itself
    dom = max(row_avg, key=row_avg.get)
    dom_ms = ms_bwd_main if dom == "bwd" else row_avg[dom]
    dom_tf = step.flops[dom] / dom_ms / 1e9
    traffic, traffic_note = dram_traffic(dom)
    traffic_f, traffic_note_f = dram_traffic("fwd")
    timed_s = ms_step * args.steps / 1e3
    # the per-workload table is one GPU's measurement: rank 0 alone takes it
    extra = {} if (args.quick or rank != 0) else measure_configs(bss, dev, peaks)
    peak_kind = (f"bf16 burst ({peaks['source']}): the timed region lasts {timed_s:.2f} s, "
                 f"not a seconds-long run at the power cap")
    out = {
        "metric": METRIC,
        "value": round(value, 2),
        "unit": UNIT,
        "n_gpus": world,
        "steps": args.steps,
        "warmup": args.warmup,
        "ms_per_step": round(ms_step, 4),
        "higher_is_better": True,
        "scaling": "weak",
        "vs_baseline": None,
        "dtype": "bf16",
        "data": "synthetic: torch.randn seeded, rounded to bf16 (no dataset)",
        "config": {"workload": w.name, "B": w.B, "H": w.H, "L": w.L, "d": w.d, "causal": True,
                   "value": "causal forward (attn_fwd): 4d FLOPs per allowed pair over its mean "
                            "CUDA-event time inside the timed steps, summed over ranks",
                   "step": "causal fwd + 8-chunk split-KV fwd and merge + block-sparse fwd "
                           "(local+global+random, 128-blocks) + recompute bwd",
                   "l2": "inputs 537 MB per step > 129 MB L2; no flush",
                   "parallelism": f"replicas x{world} (independent heads per GPU)"},
        "fwd_ms": round(ms_fwd, 4),
        "fwd_frac_of_burst_peak": round(value / world / pk_b, 4),
        "step_tflops": round(step_tf, 2),
        "row_tflops": {k: round(v, 1) for k, v in row_tf.items()},
        "row_ms": {k: round(v, 4) for k, v in row_avg.items()},
        "sparse_pairs_per_s": step.pairs_sparse / row_avg["sparse"] * 1e3,
        "sparse_executed_tiles": step.tiles_sparse,
        "sparse_list_stats": dict(zip(("listed", "executed", "future", "pairs"), list_stats)),
        "roofline": {"kernel": MAIN_KERNEL_OF_ROW.get(dom, KERNEL_OF_ROW[dom]),
                     "share_of_step": round(row_avg[dom] / sum(row_avg.values()), 4),
                     "bound": "tensor", "achieved": round(dom_tf, 1),
                     "peak": pk_b, "unit": "TFLOP/s",
                     "frac": round(dom_tf / pk_b, 4),
                     "frac_of_sustained": round(dom_tf / pk_s, 4),
                     "peak_kind": peak_kind,
                     "flops_per_launch": step.flops[dom],
                     "ms_per_launch": round(dom_ms, 4),
                     "call": {"what": KERNEL_OF_ROW[dom], "ms": round(row_avg[dom], 4),
                              "achieved": round(row_tf[dom], 1),
                              "frac": round(row_tf[dom] / pk_b, 4)},
                     "traffic": traffic, "traffic_note": traffic_note},
        "roofline_fwd": {"kernel": KERNEL_OF_ROW["fwd"], "bound": "tensor",
                         "achieved": round(row_tf["fwd"], 1), "peak": pk_b, "unit": "TFLOP/s",
                         "frac": round(row_tf["fwd"] / pk_b, 4),
                         "frac_of_sustained": round(row_tf["fwd"] / pk_s, 4),
                         "flops_per_launch": step.flops["fwd"], "target_frac": 0.6,
                         "traffic": traffic_f, "traffic_note": traffic_note_f},
        "clocks": clock_info,
        "e2e": {"value": round(job_throughput(step.flops["fwd"], ms_e2e, world), 2), "unit": UNIT,
                "h2d_bytes_per_step": nbytes(fwd_in), "d2h_bytes_per_step": nbytes(fwd_outs[0]),
                "ms_per_step": round(ms_e2e, 4),
                "what": "attn_fwd through the public API: Q, K, V uploaded from pinned host "
                        "memory, O and LSE downloaded, every step",
                "copies": "one stream per direction, overlapping the neighbouring steps",
                "serial_value": round(job_throughput(step.flops["fwd"], ms_e2e_serial, world), 2),
                "serial_ms_per_step": round(ms_e2e_serial, 4),
                "step": {"tflops": round(job_throughput(step.total_flops, ms_e2e_step, world), 2),
                         "ms_per_step": round(ms_e2e_step, 4),
                         "h2d_bytes_per_step": nbytes(step_in),
                         "d2h_bytes_per_step": nbytes(step_outs[0])}},
        "gpu_launches": step.launches_per_step * args.steps,
        "device_status": status,
        "wall_s_timed": round(wall, 3),
        "configs_measured": extra,
    }
    if rank == 0 and not args.no_cpu_baseline:
        out["cpu_baseline"] = cpu_baseline(sample_seconds=args.cpu_seconds)
    if rank == 0:
        print(json.dumps(out), flush=True)
    if world > 1:
        import torch.distributed as dist
        dist.destroy_process_group()


# ---------------------------------------------------------------------------
# CPU oracle timing (the baseline arm)
# ---------------------------------------------------------------------------

def oracle_forward_sample(cpu, w, stride=16, offset=0):
    """The oracle's causal forward on every ``stride``-th query row of one head
    (rows offset, offset+stride, ...) of the step's workload; returns the
    algorithmic FLOPs of those rows (4d per allowed pair)."""
    import oracle
    from workloads import to_f64
    q, k, v = (to_f64(cpu[n][0:1, 0:1]) for n in ("q", "k", "v"))
    rows = np.arange(offset % stride, w.L, stride)
    oracle.attention_forward(q, k, v, w.scale, causal=True, rows=rows)
    return 4 * w.d * int((rows + 1).sum())


def _oracle_inputs(w):
    return make_inputs(Workload(w.name, 1, 1, w.L, w.d, True, w.seed))


def cpu_baseline(sample_seconds=15.0):
    w = STEP_WORKLOAD
    cpu = _oracle_inputs(w)
    t0 = time.time()
    flops = 0
    n = 0
    while True:
        flops += oracle_forward_sample(cpu, w, offset=n)
        n += 1
        if time.time() - t0 >= sample_seconds or n >= 16:
            break
    dt = time.time() - t0
    return {"value": round(flops / dt / 1e12, 6), "unit": UNIT,
            "cores": len(os.sched_getaffinity(0)), "kind": "oracle",
            "sample": f"{n} x every 16th query row (1024 rows) of one head (B=1, H=1) of the "
                      f"step's workload L={w.L} d={w.d}: causal forward, fp64 numpy, {dt:.1f} s"}


def run_reference(args):
    rank, world, _ = dist_setup()
    if rank != 0:
        return
    w = STEP_WORKLOAD
    cpu = _oracle_inputs(w)
    for i in range(args.warmup):
        oracle_forward_sample(cpu, w, offset=i)
    t0 = time.time()
    flops = 0
    for i in range(args.steps):
        flops += oracle_forward_sample(cpu, w, offset=i)
    dt = time.time() - t0
    value = flops / dt / 1e12
    out = {
        "impl": "reference",
        "metric": METRIC,
        "value": round(value, 6),
        "unit": UNIT,
        "n_gpus": world,
        "steps": args.steps,
        "warmup": args.warmup,
        "ms_per_step": round(dt / args.steps * 1e3, 2),
        "higher_is_better": True,
        "scaling": "weak",
        "vs_baseline": None,
        "dtype": "f64",
        "data": "synthetic: torch.randn seeded, rounded to bf16, upcast to fp64",
        "config": {"workload": w.name, "B": w.B, "H": w.H, "L": w.L, "d": w.d, "causal": True,
                   "sample_per_step": "every 16th query row (1024 rows) of one head (B=1, H=1) "
                                      "drawn like the workload; causal forward",
                   "parallelism": "host cores"},
        "cpu_baseline": {"value": round(value, 6), "unit": UNIT,
                         "cores": len(os.sched_getaffinity(0)), "kind": "oracle",
                         "sample": "per step, every 16th query row of one L=16384 d=128 head: "
                                   "the oracle's causal forward (fp64 numpy)"},
        "e2e": {"value": round(value, 6), "unit": UNIT, "h2d_bytes_per_step": 0,
                "d2h_bytes_per_step": 0},
    }
    print(json.dumps(out), flush=True)


PROFILE_CASES = ("fwd", "fwd16k", "sparse", "sparse16k", "sparse_bwd", "bwd", "bwd16k", "fwd64",
                 "bwd64", "partial", "merge", "splitkv", "splitkv16k", "select", "decode")


def run_profile_case(kind: str):
    """One kernel on one workload, for ncu: two launches (a warm-up and a
    measured one).  Unsuffixed cases use the causal B=4 H=16 L=4096 d=128
    workload (inputs 268 MB > L2); "16k" cases the bench step's B=2 H=16
    L=16384 d=128 workload; "sparse_bwd" the block-sparse L'=16320 workload;
    "fwd64"/"bwd64" the B=8 H=16 L=8192 d=64 workload."""
    import block_sparse_softmax_gb300 as bss
    bss.library()
    dev = torch.device("cuda", 0)
    if kind == "decode":
        # 16 queries at the end of a 16384-key causal cache, split as the bench row splits it
        w = DECODE_16K
        x = {k: t.to(dev) for k, t in make_inputs(w).items()}
        ws = torch.empty(bss.attn_fwd_splitkv_workspace_bytes(w.B, w.H, w.Lq, w.L, w.d, w.chunks),
                         device=dev, dtype=torch.uint8)
        fn = lambda: bss.attn_fwd_splitkv(x["q"], x["k"], x["v"], w.chunks, causal=True,
                                          scale=w.scale, q_offset=w.L - w.Lq, workspace=ws)
        return _run_profile_fn(kind, fn)
    if kind == "select":
        # the selector on the block-sparse workload: one list per head,
        # 4 local blocks + the 4 best-scoring earlier blocks per query block
        w = SPARSE_16K
        x = {k: t.to(dev) for k, t in make_inputs(w).items()}
        fn = lambda: bss.attn_select_blocks(x["q"], x["k"], 4, local_blocks=4, causal=True,
                                            n_lists=w.B * w.H, scale=w.scale)
        return _run_profile_fn(kind, fn)
    if kind in ("fwd16k", "sparse16k", "bwd16k", "splitkv16k"):
        w = CAUSAL_16K
    elif kind == "sparse_bwd":
        w = SPARSE_16K
    elif kind in ("fwd64", "bwd64"):
        w = BWD_8K
    else:
        w = CAUSAL_4K
    w = Workload(w.name, w.B, w.H, w.L, w.d, True, w.seed, backward=True)
    x = {k: t.to(dev) for k, t in make_inputs(w).items()}
    base = kind.replace("16k", "").replace("64", "")
    if base == "fwd":
        fn = lambda: bss.attn_fwd(x["q"], x["k"], x["v"], causal=True, scale=w.scale)
    elif base in ("sparse", "sparse_bwd"):
        rp, ci = local_global_random_blocklist(w.n_blocks, seed=2)
        rpd, cid = torch.from_numpy(rp).to(dev), torch.from_numpy(ci).to(dev)
        fn = lambda: bss.attn_fwd_blocksparse(x["q"], x["k"], x["v"], rpd, cid, causal=True,
                                              scale=w.scale)
        if base == "sparse_bwd":
            o, lse = fn()
            ws = torch.empty(bss.attn_bwd_blocksparse_workspace_bytes(w.B, w.H, w.L, w.d),
                             device=dev, dtype=torch.uint8)
            fn = lambda: bss.attn_bwd_blocksparse(x["q"], x["k"], x["v"], o, lse, x["do"], rpd,
                                                  cid, causal=True, scale=w.scale, workspace=ws)
    elif base == "bwd":
        o, lse = bss.attn_fwd(x["q"], x["k"], x["v"], causal=True, scale=w.scale)
        fn = lambda: bss.attn_bwd(x["q"], x["k"], x["v"], o, lse, x["do"], causal=True,
                                  scale=w.scale)
    elif base == "splitkv":
        ws = torch.empty(bss.attn_fwd_splitkv_workspace_bytes(w.B, w.H, w.L, w.L, w.d, 8),
                         device=dev, dtype=torch.uint8)
        fn = lambda: bss.attn_fwd_splitkv(x["q"], x["k"], x["v"], 8, causal=True,
                                          scale=w.scale, workspace=ws)
    elif base in ("partial", "merge"):
        bounds = chunk_bounds(w.L, 8)
        kc = [x["k"][:, :, s:e].contiguous() for s, e in bounds]
        vc = [x["v"][:, :, s:e].contiguous() for s, e in bounds]
        C = len(bounds)
        m = torch.empty(C, w.B, w.H, w.L, device=dev)
        l_ = torch.empty_like(m)
        acc = torch.empty(C, w.B, w.H, w.L, w.d, device=dev)

        def partials():
            for c, (s, _) in enumerate(bounds):
                bss.attn_fwd_partial(x["q"], kc[c], vc[c], causal=True, scale=w.scale,
                                     k_offset=s, m=m[c], l=l_[c], acc=acc[c])
        if base == "partial":
            fn = partials
        else:
            partials()
            fn = lambda: bss.attn_merge_states(m, l_, acc)
    else:
        raise SystemExit(f"unknown profile case {kind}")
    _run_profile_fn(kind, fn)


def _run_profile_fn(kind: str, fn):
    import block_sparse_softmax_gb300 as bss
    for _ in range(2):
        fn()
    torch.cuda.synchronize()
    status = bss.attn_poll_status()
    print(json.dumps({"profile_case": kind, "status": status}))
    if status != 0:
        raise SystemExit(1)


def main():
    ap = argparse.ArgumentParser()
    ap.add_argument("--profile", choices=PROFILE_CASES, default=None,
                    help="run one small case of one kernel (for ncu) and exit")
    ap.add_argument("--gpus", type=int, default=1)
    ap.add_argument("--steps", type=int, default=100)
    ap.add_argument("--warmup", type=int, default=5)
    ap.add_argument("--impl", choices=["native", "reference"], default="native")
    ap.add_argument("--quick", action="store_true", help="skip the per-workload measurements")
    ap.add_argument("--no-cpu-baseline", action="store_true")
    ap.add_argument("--cpu-seconds", type=float, default=12.0)
    args = ap.parse_args()
    if args.warmup < 3:
        args.warmup = 3
    if args.profile:
        run_profile_case(args.profile)
    elif args.impl == "reference":
        run_reference(args)
    else:
        run_gpu(args)


if __name__ == "__main__":
    main()
