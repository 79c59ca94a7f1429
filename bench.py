#!/usr/bin/env python
"""Benchmark of the GB300 attention path (one JSON line on rank 0).

A step is one pass of the whole hot path over one batch of the causal
B=4 H=16 L=4096 d=128 workload (bf16 inputs resident in HBM):
  1. causal forward                    (attn_fwd: O, LSE)
  2. split-KV forward: 8 KV chunks     (attn_fwd_partial x 8, attn_merge_states)
  3. block-sparse forward              (attn_fwd_blocksparse, local+global+random list)
  4. backward by recomputation         (attn_bwd: D, dQ, dK, dV)
`value` is the algorithmic TFLOP/s of the step (4d FLOPs per allowed pair for
each forward, 10d per allowed pair for the backward).  The forward alone
(the metric's own operation), sparse pairs/s, the L=16384 dense causal
target and the other workload shapes are reported beside it.

--impl reference times the fp64 CPU oracle on a bounded sample of the same
step (one head) on the host cores, with the same metric and unit.
Multi-GPU (torchrun): every rank runs its own batch (independent heads, no
data-path collective; weak scaling); time is the max over ranks.
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


# The kernel behind each row of the step, and the sources that define it (the
# DRAM traffic recorded for a kernel is used only while they are unchanged).
KERNEL_OF_ROW = {
    "fwd": "attn_fwd_kernel (causal, persistent)",
    "splitkv": "attn_fwd_kernel (partial, 8 key chunks in one launch) + merge_states_kernel",
    "sparse": "attn_fwd_kernel (block-sparse)",
    "bwd": "attn_bwd_main_kernel (+ preprocess and dq_convert in the same call)",
}
TRAFFIC_KERNEL = {"fwd": "attn_fwd_kernel", "bwd": "attn_bwd_main_kernel"}
KERNEL_SOURCES = {"attn_fwd_kernel": ["fwd.cu", "common.cuh", "ptx.cuh"],
                  "attn_bwd_main_kernel": ["bwd.cu", "common.cuh", "ptx.cuh"]}


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
        rec = json.load(f).get(kernel)
    if rec is None:
        return None, "no ncu capture of this kernel"
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
                 "--format=csv,noheader,nounits", "-lms", "50"], stdout=self.fh,
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

    def __init__(self, bss, w: Workload, dev):
        self.bss = bss
        self.w = w
        B, H, L, d = w.B, w.H, w.L, w.d
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
        self.launches_per_step = 1 + 2 + 1 + 3
        self.events = None

    def run(self, timed_rows=False):
        bss, d, w = self.bss, self.dev, self.w
        ev = self.events if timed_rows else None
        if ev is not None:
            ev["fwd"][0].record()
        bss.attn_fwd(d["q"], d["k"], d["v"], causal=True, scale=w.scale, out=self.o, lse=self.lse)
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
        bss.attn_bwd(d["q"], d["k"], d["v"], self.o, self.lse, d["do"], causal=True,
                     scale=w.scale, workspace=self.ws, dq=self.dq, dk=self.dk, dv=self.dv,
                     delta=self.delta)
        if ev is not None:
            ev["bwd"][1].record()

    def new_events(self):
        self.events = {k: (torch.cuda.Event(enable_timing=True), torch.cuda.Event(enable_timing=True))
                       for k in self.flops}


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


def e2e_pipelined_ms(sets, host_in, host_outs, steps, warmup, sync_all):
    """Milliseconds per step end to end through the public API: every step
    uploads its inputs from pinned host memory and downloads its results
    (O, LSE, dQ, dK, dV) to pinned host memory, all inside the timed region.
    The copies run on one stream per direction and overlap the neighbouring
    steps' compute: step k+1 uploads into one of two device buffer sets while
    step k computes on the other and step k-1's results come down."""
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
        sets[s].run()
        ev_comp[s].record(comp)

    def download(k):
        s = k % 2
        st, ho = sets[s], host_outs[s]
        with torch.cuda.stream(down):
            down.wait_event(ev_comp[s])
            ho["o"].copy_(st.o, non_blocking=True)
            ho["lse"].copy_(st.lse, non_blocking=True)
            ho["dq"].copy_(st.dq, non_blocking=True)
            ho["dk"].copy_(st.dk, non_blocking=True)
            ho["dv"].copy_(st.dv, non_blocking=True)
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
    # dense causal target at L=16384
    w = CAUSAL_16K
    x = {k: t.to(dev) for k, t in make_inputs(w).items()}
    o = torch.empty_like(x["q"])
    lse = torch.empty(w.B, w.H, w.L, device=dev)
    ms = bench_kernel(lambda: bss.attn_fwd(x["q"], x["k"], x["v"], causal=True, scale=w.scale,
                                           out=o, lse=lse))
    fl = 4 * w.d * w.B * w.H * causal_pairs(w.L, w.L)
    tf = fl / ms / 1e9
    out[w.name] = {"ms": round(ms, 4), "tflops": round(tf, 1), "frac_burst": round(tf / pk, 4),
                   "frac_sustained": round(tf / peaks["bf16_sustained"], 4),
                   "frac_ex2_ceiling": round(tf / (4 * w.d * ex2_rate / 1e12), 4),
                   "target_frac": 0.6}
    del x, o, lse
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

    ms_p = bench_kernel(partials, reps=2, warmup=1)
    ms_m = bench_kernel(lambda: bss.attn_merge_states(m, l_, acc, out=o, lse=lse), reps=10)
    del m, l_, acc, kc, vc
    # the same in one split-KV launch (chunks read in place) + merge
    ws = torch.empty(bss.attn_fwd_splitkv_workspace_bytes(w.B, w.H, w.L, w.L, w.d, w.chunks),
                     device=dev, dtype=torch.uint8)
    ms_s = bench_kernel(lambda: bss.attn_fwd_splitkv(x["q"], x["k"], x["v"], w.chunks, causal=True,
                                                     scale=w.scale, workspace=ws, out=o, lse=lse),
                        reps=3, warmup=1)
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
    w = rank_workload(CAUSAL_4K, rank)
    step = Step(bss, w, dev)
    # warm-up, then the timed region (device-resident inputs); every row of
    # every step is bracketed by CUDA events on the launching stream
    clocks = ClockSampler(local)
    for _ in range(args.warmup):
        step.run()
    torch.cuda.synchronize()
    sync_all()
    events = []
    for _ in range(args.steps):
        step.new_events()
        events.append(step.events)
    clocks.start()
    t0 = time.time()
    start = torch.cuda.Event(enable_timing=True)
    end = torch.cuda.Event(enable_timing=True)
    start.record()
    for i in range(args.steps):
        step.events = events[i]
        step.run(timed_rows=True)
    end.record()
    torch.cuda.synchronize()
    sync_all()
    wall = time.time() - t0
    clock_info = clocks.stop()
    ms_step = start.elapsed_time(end) / args.steps
    row_avg = {k: statistics.mean(ev[k][0].elapsed_time(ev[k][1]) for ev in events)
               for k in step.flops}
    if world > 1:
        ms_step = max_over_ranks(ms_step, dev)

    # end to end through the public API: pinned host inputs in, results out,
    # copies overlapping the neighbouring steps (a second device buffer set)
    names_in = ["q", "k", "v", "do"]
    host_in = {n: step.cpu[n].pin_memory() for n in names_in}
    host_outs = [{**{n: torch.empty(step.o.shape, dtype=torch.bfloat16).pin_memory()
                     for n in ("o", "dq", "dk", "dv")},
                  "lse": torch.empty(step.lse.shape).pin_memory()} for _ in range(2)]
    h2d = sum(t.numel() * t.element_size() for t in host_in.values())
    d2h = sum(t.numel() * t.element_size() for t in host_outs[0].values())
    sets = [step, Step(bss, w, dev)]
    ms_e2e = e2e_pipelined_ms(sets, host_in, host_outs, max(3, args.steps // 2), 2, sync_all)
    del sets

    # the same with no overlap: upload, step, download on one stream
    def e2e_serial(_timed):
        for n in names_in:
            step.dev[n].copy_(host_in[n], non_blocking=True)
        step.run()
        for n, t in (("o", step.o), ("lse", step.lse), ("dq", step.dq), ("dk", step.dk),
                     ("dv", step.dv)):
            host_outs[0][n].copy_(t, non_blocking=True)

    ms_e2e_serial = time_loop(e2e_serial, max(3, args.steps // 2), 2, sync_all)
    if world > 1:
        ms_e2e = max_over_ranks(ms_e2e, dev)
        ms_e2e_serial = max_over_ranks(ms_e2e_serial, dev)
    status = bss.attn_poll_status()

    fwd_tf = step.flops["fwd"] / row_avg["fwd"] / 1e9
    bwd_tf = step.flops["bwd"] / row_avg["bwd"] / 1e9
    value = job_throughput(step.total_flops, ms_step, world)
    # dominant kernel: the largest share of the step's time
    dom = max(row_avg, key=row_avg.get)
    dom_tf = step.flops[dom] / row_avg[dom] / 1e9
    traffic, traffic_note = dram_traffic(dom)
    # the per-workload table is one GPU's measurement: rank 0 alone takes it
    extra = {} if (args.quick or rank != 0) else measure_configs(bss, dev, peaks)
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
                   "step": "causal fwd + 8-chunk split-KV fwd and merge + block-sparse fwd "
                           "(local+global+random, 128-blocks) + recompute bwd",
                   "l2": "inputs 268 MB per step > 129 MB L2; no flush",
                   "parallelism": f"replicas x{world} (independent heads per GPU)"},
        "fwd_tflops": round(fwd_tf, 1),
        "fwd_frac_of_burst_peak": round(fwd_tf / peaks["bf16_burst"], 4),
        "bwd_tflops": round(bwd_tf, 1),
        "sparse_pairs_per_s": step.pairs_sparse / row_avg["sparse"] * 1e3,
        "sparse_executed_tiles": step.tiles_sparse,
        "row_ms": {k: round(v, 4) for k, v in row_avg.items()},
        "roofline": {"kernel": KERNEL_OF_ROW[dom],
                     "share_of_step": round(row_avg[dom] / sum(row_avg.values()), 4),
                     "bound": "tensor", "achieved": round(dom_tf, 1),
                     "peak": peaks["bf16_sustained"], "unit": "TFLOP/s",
                     "frac": round(dom_tf / peaks["bf16_sustained"], 4),
                     "peak_kind": f"bf16 sustained ({peaks['source']})",
                     "traffic": traffic, "traffic_note": traffic_note},
        "clocks": clock_info,
        "e2e": {"value": round(job_throughput(step.total_flops, ms_e2e, world), 2), "unit": UNIT,
                "h2d_bytes_per_step": h2d, "d2h_bytes_per_step": d2h,
                "ms_per_step": round(ms_e2e, 4),
                "copies": "one stream per direction, overlapping the neighbouring steps",
                "serial_value": round(job_throughput(step.total_flops, ms_e2e_serial, world), 2),
                "serial_ms_per_step": round(ms_e2e_serial, 4)},
        "gpu_launches": step.launches_per_step * args.steps,
        "device_status": status,
        "wall_s_timed": round(wall, 3),
        "configs_measured": extra,
    }
    if rank == 0 and not args.no_cpu_baseline:
        out["cpu_baseline"] = cpu_baseline(step_sample_seconds=args.cpu_seconds)
    if rank == 0:
        print(json.dumps(out), flush=True)
    if world > 1:
        import torch.distributed as dist
        dist.destroy_process_group()


# ---------------------------------------------------------------------------
# CPU oracle timing (the baseline arm)
# ---------------------------------------------------------------------------

def oracle_step_one_head(cpu, w, head=(0, 0)):
    """The oracle on one (b, h) head of the step: returns its algorithmic FLOPs."""
    import oracle
    from workloads import to_f64
    b, h = head
    q, k, v, do = (to_f64(cpu[n][b:b + 1, h:h + 1]) for n in ("q", "k", "v", "do"))
    L, d = w.L, w.d
    oracle.attention_forward(q, k, v, w.scale, causal=True)
    states = []
    for s, e in chunk_bounds(L, 8):
        M = oracle.allowed_rows(np.arange(L), e - s, causal=True, k_offset=s)
        states.append(oracle.partial_state(q[0, 0], k[0, 0, s:e], v[0, 0, s:e], w.scale, M))
    oracle.merge_states(np.stack([x[0] for x in states]), np.stack([x[1] for x in states]),
                        np.stack([x[2] for x in states]))
    rp, ci = local_global_random_blocklist((L + 127) // 128, seed=2)
    oracle.attention_forward(q, k, v, w.scale, causal=True, block=128, row_ptr=rp, col_idx=ci)
    oracle.attention_backward(q, k, v, do, w.scale, causal=True)
    pairs = causal_pairs(L, L)
    sp, _ = sparse_counts(L, rp, ci, True)
    return 4 * d * pairs * 2 + 4 * d * sp + 10 * d * pairs


def cpu_baseline(step_sample_seconds=20.0):
    w = CAUSAL_4K
    cpu = make_inputs(Workload(w.name, 1, 1, w.L, w.d, True, w.seed, backward=True))
    t0 = time.time()
    flops = 0
    n = 0
    while True:
        flops += oracle_step_one_head(cpu, w)
        n += 1
        if time.time() - t0 >= step_sample_seconds or n >= 8:
            break
    dt = time.time() - t0
    return {"value": round(flops / dt / 1e12, 6), "unit": UNIT,
            "cores": len(os.sched_getaffinity(0)), "kind": "oracle",
            "sample": f"{n} x one head (B=1,H=1) of the step workload L={w.L} d={w.d}: causal fwd, "
                      f"8-chunk partial+merge, block-sparse fwd, bwd; fp64 numpy, {dt:.1f} s"}


def run_reference(args):
    rank, world, _ = dist_setup()
    if rank != 0:
        return
    w = CAUSAL_4K
    cpu = make_inputs(Workload(w.name, 1, 1, w.L, w.d, True, w.seed, backward=True))
    for _ in range(args.warmup):
        oracle_step_one_head(cpu, w)
    t0 = time.time()
    flops = 0
    for _ in range(args.steps):
        flops += oracle_step_one_head(cpu, w)
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
                   "sample_per_step": "one head (b=0, h=0) of the workload through every row",
                   "parallelism": "host cores"},
        "cpu_baseline": {"value": round(value, 6), "unit": UNIT,
                         "cores": len(os.sched_getaffinity(0)), "kind": "oracle",
                         "sample": "one head per step of the L=4096 d=128 causal workload: fwd, "
                                   "8-chunk partial+merge, block-sparse fwd, bwd (fp64 numpy)"},
        "e2e": {"value": round(value, 6), "unit": UNIT, "h2d_bytes_per_step": 0,
                "d2h_bytes_per_step": 0},
    }
    print(json.dumps(out), flush=True)


def run_profile_case(kind: str):
    """One kernel of the bench step on the step's own workload (causal B=4 H=16
    L=4096 d=128, inputs 268 MB > L2), or the L=16384 target shape, for ncu:
    one warm-up launch and one measured launch."""
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
    w = CAUSAL_16K if kind == "fwd16k" else CAUSAL_4K
    w = Workload(w.name, w.B, w.H, w.L, w.d, True, w.seed, backward=True)
    x = {k: t.to(dev) for k, t in make_inputs(w).items()}
    if kind in ("fwd", "fwd16k"):
        fn = lambda: bss.attn_fwd(x["q"], x["k"], x["v"], causal=True, scale=w.scale)
    elif kind == "sparse":
        rp, ci = local_global_random_blocklist(w.n_blocks, seed=2)
        rpd, cid = torch.from_numpy(rp).to(dev), torch.from_numpy(ci).to(dev)
        fn = lambda: bss.attn_fwd_blocksparse(x["q"], x["k"], x["v"], rpd, cid, causal=True,
                                              scale=w.scale)
    elif kind == "bwd":
        o, lse = bss.attn_fwd(x["q"], x["k"], x["v"], causal=True, scale=w.scale)
        fn = lambda: bss.attn_bwd(x["q"], x["k"], x["v"], o, lse, x["do"], causal=True,
                                  scale=w.scale)
    elif kind == "splitkv":
        ws = torch.empty(bss.attn_fwd_splitkv_workspace_bytes(w.B, w.H, w.L, w.L, w.d, 8),
                         device=dev, dtype=torch.uint8)
        fn = lambda: bss.attn_fwd_splitkv(x["q"], x["k"], x["v"], 8, causal=True,
                                          scale=w.scale, workspace=ws)
    elif kind in ("partial", "merge"):
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
        if kind == "partial":
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
    ap.add_argument("--profile", choices=["fwd", "fwd16k", "sparse", "bwd", "partial", "merge",
                                            "splitkv", "select", "decode"],
                    default=None,
                    help="run one small case of one kernel (for ncu) and exit")
    ap.add_argument("--gpus", type=int, default=1)
    ap.add_argument("--steps", type=int, default=100)
    ap.add_argument("--warmup", type=int, default=5)
    ap.add_argument("--impl", choices=["native", "reference"], default="native")
    ap.add_argument("--quick", action="store_true", help="skip the per-workload measurements")
    ap.add_argument("--no-cpu-baseline", action="store_true")
    ap.add_argument("--cpu-seconds", type=float, default=15.0)
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
