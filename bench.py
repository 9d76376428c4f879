#!/usr/bin/env python3
"""Benchmark: sparse-MLA paged decode on GB300, microseconds per call.

One step = one decode call (split kernel + merge when nsplit > 1) over one
batch of synthetic inputs already resident in HBM.  Calls cycle through R
independent input sets (q, top-k, block table) over one large cache, with
R * bytes-per-call >= 4 x L2, so every timed call reads rows that are not in
L2.  Timed on the device with CUDA events around CUDA-graph replays.

  python bench.py [--gpus N] [--steps K] [--warmup W] [--workload NAME]
                  [--impl ours|reference] [--no-per-config] [--no-cpu-baseline]

Prints one JSON line (rank 0).  --impl reference times the float64 CPU
oracle on the host cores (a bounded sample of the same workload, scaled to
a full call).
"""
from __future__ import annotations

import argparse
import hashlib
import glob
import json
import math
import os
import statistics
import subprocess
import sys
import threading
import time

ROOT = os.path.dirname(os.path.abspath(__file__))
sys.path.insert(0, ROOT)

METRIC = "µs/call and achieved HBM GB/s (% roofline) for sparse-MLA decode, B=1..96"
UNIT = "us/call"
HEADLINE = "b32_ctx32k"
ALL_CONFIGS = ["tiny", "bs1_ctx8k", "b32_ctx32k", "b80_ctx128k", "b96_ragged_h64", "b96_ragged_h16"]
MIN_POOL_PAGES = 65536          # cache pages for rotations of small configs (2.75 GB)
FALLBACK_HBM_GBS = 6800.0


# ----------------------------------------------------------------------------- rank / env helpers

def dist_env():
    return int(os.environ.get("RANK", 0)), int(os.environ.get("WORLD_SIZE", 1)), int(os.environ.get("LOCAL_RANK", 0))


def reduce_max(value: float, world: int) -> float:
    """Max of a float over ranks (identity when world == 1)."""
    if world == 1:
        return value
    import torch
    import torch.distributed as dist
    dev = "cuda" if dist.get_backend() == "nccl" else "cpu"
    t = torch.tensor([value], dtype=torch.float64, device=dev)
    dist.all_reduce(t, op=dist.ReduceOp.MAX)
    return float(t.item())


def barrier(world: int):
    if world > 1:
        import torch.distributed as dist
        dist.barrier()


def aggregate_us_per_call(max_elapsed_s: float, steps: int, world: int) -> float:
    """Whole-job microseconds per call: every rank ran `steps` calls in at most max_elapsed_s."""
    return max_elapsed_s * 1e6 / (steps * world)


def replica_spec(name: str, rank: int):
    """The workload recipe a replica runs: the named configuration with a seed of its own per rank
    (rank 0 keeps the configuration's seed), so replicas read different rows of their caches."""
    import dataclasses
    from sparse_mla_decode_paged_gb300 import workloads as wl
    spec = wl.CONFIGS[name]
    return dataclasses.replace(spec, seed=spec.seed + 7777 * rank) if rank else spec


def measured_peaks():
    p = os.path.join(ROOT, "MEASURED_PEAKS.json")
    if os.path.exists(p):
        with open(p) as f:
            d = json.load(f)
        return float(d["hbm_gbs"]), "measured"
    return FALLBACK_HBM_GBS, "fallback"


SPLIT_KERNEL_SOURCES = ("smla_split.cu", "smla_split_layout.cuh", "smla_ptx.cuh", "smla_device.cuh")


def kernel_source_hash() -> str:
    """Hash of the split kernel's own sources (its translation unit and device headers)."""
    h = hashlib.sha256()
    for name in SPLIT_KERNEL_SOURCES:
        with open(os.path.join(ROOT, "sparse_mla_decode_paged_gb300", "csrc", name), "rb") as fh:
            h.update(fh.read())
    return h.hexdigest()[:16]


def recorded_traffic(workload: str):
    """DRAM bytes per launch of the split kernel from the committed ncu summary, if it was taken
    on the current kernel sources (else None)."""
    p = os.path.join(ROOT, "profiles", "split_kernel_dram_traffic.json")
    if not os.path.exists(p):
        return None
    with open(p) as f:
        d = json.load(f)
    if d.get("kernel_source_hash") != kernel_source_hash():
        return None
    return d.get("traffic_bytes_per_launch", {}).get(workload)


# ----------------------------------------------------------------------------- clocks

class ClockSampler:
    """nvidia-smi samples (200 ms) of SM clock and throttle reasons while running.  The GPU is named
    by the entry of CUDA_VISIBLE_DEVICES (an index or a UUID, both of which nvidia-smi -i takes) or by
    its index when that variable is unset."""
    FIELDS = "clocks.sm,clocks.max.sm,power.draw,clocks_event_reasons.active,clocks_event_reasons.hw_slowdown," \
             "clocks_event_reasons.hw_thermal_slowdown,clocks_event_reasons.sw_thermal_slowdown," \
             "clocks_event_reasons.sw_power_cap"

    def __init__(self, gpu_index):
        self.gpu = gpu_index
        self.proc = None
        self.lines = []
        self.error = None

    def __enter__(self):
        try:
            self.proc = subprocess.Popen(["nvidia-smi", "-i", str(self.gpu), f"--query-gpu={self.FIELDS}",
                                          "--format=csv,noheader,nounits", "-lms", "200"],
                                         stdout=subprocess.PIPE, stderr=subprocess.PIPE, text=True)
            self._t = threading.Thread(target=self._read, daemon=True)
            self._t.start()
        except OSError as e:
            self.proc = None
            self.error = repr(e)
        return self

    def _read(self):
        for line in self.proc.stdout:
            self.lines.append(line.strip())

    def wait_first(self, timeout_s: float = 10.0) -> bool:
        """Block until nvidia-smi has printed its first sample (its start-up takes about a second)."""
        t0 = time.time()
        while self.proc is not None and not self.lines and time.time() - t0 < timeout_s:
            if self.proc.poll() is not None:
                break
            time.sleep(0.02)
        return bool(self.lines)

    def __exit__(self, *a):
        if self.proc:
            self.proc.terminate()
            try:
                self.proc.wait(timeout=5)
            except subprocess.TimeoutExpired:
                self.proc.kill()

    def mark(self):
        """Samples printed from here on are the ones summary() reports (the load window)."""
        self.start = len(self.lines)

    def summary(self):
        sm, smax, reasons = [], None, set()
        names = ["hw_slowdown", "hw_thermal_slowdown", "sw_thermal_slowdown", "sw_power_cap"]
        for ln in self.lines[getattr(self, "start", 0):]:
            parts = [x.strip() for x in ln.split(",")]
            try:
                sm.append(float(parts[0]))
            except (ValueError, IndexError):
                continue
            try:
                smax = float(parts[1])
            except (ValueError, IndexError):
                pass
            for n, v in zip(names, parts[4:8]):
                if v.lower() == "active":
                    reasons.add(n)
        out = {"sm_mhz": statistics.median(sm) if sm else None, "sm_max_mhz": smax,
               "reasons": sorted(reasons), "samples": len(sm), "gpu": str(self.gpu)}
        if not sm:
            err = self.error
            if err is None and self.proc is not None and self.proc.stderr is not None:
                try:
                    err = self.proc.stderr.read()[-300:].strip() or None
                except Exception:
                    err = None
            out["error"] = err or "nvidia-smi printed no sample"
            sys.stderr.write(f"bench: no clock sample from nvidia-smi -i {self.gpu}: {out['error']}\n")
        return out


# ----------------------------------------------------------------------------- our arm

class Bench:
    def __init__(self, name: str, device, seed_offset: int = 0, nsplit: int = 0, merge: int = 0,
                 heads_per_cta: int = 0):
        import torch
        from sparse_mla_decode_paged_gb300 import api
        from sparse_mla_decode_paged_gb300 import workloads as wl
        self.torch, self.api, self.wl = torch, api, wl
        self.name = name
        spec = replica_spec(name, seed_offset)
        self.spec = spec
        self.device = device
        w0 = wl.make_workload(spec, device=device, pool_pages=MIN_POOL_PAGES)
        self.cache = w0.kv_cache
        self.w0 = w0
        self.bytes_per_call = wl.algorithmic_bytes(w0.topk_idx, w0.seq_lens, w0.block_table, w0.H, w0.num_pages)
        self.flops_per_call = wl.algorithmic_flops(w0.topk_idx, w0.seq_lens, w0.H)
        l2 = torch.cuda.get_device_properties(device).L2_cache_size
        self.l2 = l2
        self.R = int(min(2048, max(8, math.ceil(4 * l2 / self.bytes_per_call))))
        self.sets = [w0] + [wl.make_workload(spec, device=device, rotation=r, kv_cache=self.cache)
                            for r in range(1, self.R)]
        self.dims = api.dims_of(w0.q, w0.kv_cache, w0.block_table, w0.topk_idx, nsplit, heads_per_cta, merge)
        self.plan = api.plan(self.dims, device.index if hasattr(device, "index") else None)
        self.nsplit = self.plan.nsplit
        self.dims.nsplit = self.nsplit
        self.ws = api.alloc_workspace(self.dims, self.nsplit, device)
        B, H = w0.B, w0.H
        self.out = torch.empty((B, H, 512), dtype=torch.bfloat16, device=device)
        self.lse = torch.empty((B, H), dtype=torch.float32, device=device)
        self.o_part = torch.empty((B, self.nsplit, H, 512), dtype=torch.float32, device=device)
        self.lse_part = torch.empty((B, self.nsplit, H), dtype=torch.float32, device=device)

    def call(self, i: int):
        w = self.sets[i % self.R]
        self.api.sparse_mla_decode(w.q, self.cache, w.block_table, w.topk_idx, w.seq_lens, w.sm_scale,
                                   out=self.out, lse=self.lse, workspace=self.ws, nsplit=self.nsplit,
                                   heads_per_cta=self.plan.heads_per_cta, merge=self.dims.merge)

    def split_only(self, i: int):
        """The split kernel as the call launches it: the call itself when that is one launch (one partition,
        or the partitions merged inside the kernel), else the split kernel writing its partials."""
        if self.nsplit == 1 or self.plan.fused:
            return self.call(i)
        w = self.sets[i % self.R]
        d = self.dims
        lib = self.api._lib()
        import ctypes as C
        st = lib.sparse_mla_split(C.byref(d), self.nsplit, self.api._ptr(w.q), self.api._ptr(self.cache),
                                  self.api._ptr(w.block_table), self.api._ptr(w.topk_idx), self.api._ptr(w.seq_lens),
                                  C.c_float(w.sm_scale), self.api._ptr(self.o_part), self.api._ptr(self.lse_part),
                                  self.api._ptr(self.ws), self.api._stream())
        if st != 0:
            raise RuntimeError(f"sparse_mla_split failed: {st}")

    def append_setup(self, sets: int = 8):
        """Inputs of the KV append step at this batch: one new token per request, written into a cache
        of its own (one page per request), latent/rope drawn per rotation."""
        torch = self.torch
        B = self.w0.B
        g = torch.Generator(device="cpu").manual_seed(12345)
        self.app_sets = [((torch.randn(B, 512, generator=g)).to(torch.bfloat16).to(self.device),
                          torch.randn(B, 64, generator=g).to(torch.bfloat16).to(self.device),
                          torch.full((B,), r % 64, dtype=torch.int32).to(self.device)) for r in range(sets)]
        self.app_cache = torch.zeros((B, 64, 656), dtype=torch.uint8, device=self.device)
        self.app_bt = torch.arange(B, dtype=torch.int32, device=self.device).reshape(B, 1)
        # bytes per token: latent 1024 + rope 128 read, record 656 written, position + table entry 8
        self.app_bytes = B * (1024 + 128 + 656 + 8)

    def append_only(self, i: int):
        lat, rope, pos = self.app_sets[i % len(self.app_sets)]
        self.api.sparse_mla_kv_append(lat, rope, self.app_bt, pos, self.app_cache)

    def topk_setup(self):
        """Inputs of the top-k selection step at this workload: indexer-score stand-ins (standard
        normal, float32) over each query's context, the workload's lengths and top-k count; enough
        rotating score sets that they exceed 4 x L2."""
        torch = self.torch
        from sparse_mla_decode_paged_gb300 import workloads as wl
        w = self.w0
        self.tk_lens = w.seq_lens
        self.tk_cols = int(w.seq_lens.max().item())
        set_bytes = w.B * self.tk_cols * 4
        n_sets = int(min(256, max(4, math.ceil(4 * self.l2 / set_bytes))))
        self.tk_sets = [wl.make_indexer_scores(w.B, self.tk_cols, seed=5000 + r, device=self.device)
                        for r in range(n_sets)]
        self.tk_out = torch.empty((w.B, w.topk_idx.shape[1]), dtype=torch.int32, device=self.device)
        # scores read below each length, kept positions written, lengths read
        self.tk_bytes = int(w.seq_lens.sum().item()) * 4 + w.B * w.topk_idx.shape[1] * 4 + w.B * 4

    def topk_only(self, i: int):
        s = self.tk_sets[i % len(self.tk_sets)]
        self.api.sparse_mla_topk_select(s, self.tk_lens, self.tk_out.shape[1])

    def topk_then_decode(self, i: int):
        """A decode step's attention: the top-k selection over rotating score rows, then the decode of
        rotating inputs reading the lists it just produced (a programmatic dependent of the selection)."""
        s = self.tk_sets[i % len(self.tk_sets)]
        w = self.sets[i % self.R]
        tk = self.api.sparse_mla_topk_select(s, self.tk_lens, self.tk_out.shape[1])
        self.api.sparse_mla_decode(w.q, self.cache, w.block_table, tk, w.seq_lens, w.sm_scale,
                                   out=self.out, lse=self.lse, workspace=self.ws, nsplit=self.nsplit,
                                   heads_per_cta=self.plan.heads_per_cta, merge=self.dims.merge)

    def launches_per_call(self) -> int:
        return 1 + (1 if self.nsplit > 1 and not self.plan.fused else 0)

    def _graph(self, fn, start: int, n: int):
        torch = self.torch
        g = torch.cuda.CUDAGraph()
        s = torch.cuda.Stream()
        s.wait_stream(torch.cuda.current_stream())
        with torch.cuda.stream(s):
            fn(start)          # warm the path on the capture stream
        torch.cuda.current_stream().wait_stream(s)
        torch.cuda.synchronize()
        with torch.cuda.graph(g):
            for i in range(n):
                fn(start + i)
        return g

    def timed(self, fn, steps: int, warmup: int, world: int = 1, preroll_s: float = 0.0):
        """Run warmup calls, then exactly `steps` calls as graph replays; returns max-over-ranks seconds.
        preroll_s > 0 replays the same graph untimed for that long right before the timed region (a load
        window long enough for the clock sampler to see the GPU busy however short the timed region)."""
        torch = self.torch
        for i in range(warmup):
            fn(i)
        torch.cuda.synchronize()
        G = min(self.R, steps)
        start = warmup % self.R
        g_full = self._graph(fn, start, G)
        reps, tail = divmod(steps, G)
        g_tail = self._graph(fn, start, tail) if tail else None
        g_full.replay()                 # one untimed replay: graph upload
        torch.cuda.synchronize()
        if preroll_s > 0:
            t_end = time.time() + preroll_s
            while time.time() < t_end:
                for _ in range(max(1, 2000 // G)):
                    g_full.replay()
                torch.cuda.synchronize()
        stream = torch.cuda.current_stream()
        e0, e1 = torch.cuda.Event(enable_timing=True), torch.cuda.Event(enable_timing=True)
        barrier(world)
        torch.cuda.synchronize()
        e0.record(stream)
        for _ in range(reps):
            g_full.replay()
        if g_tail is not None:
            g_tail.replay()
        e1.record(stream)
        torch.cuda.synchronize()
        barrier(world)
        return reduce_max(e0.elapsed_time(e1) / 1e3, world)

    def replay_stats(self, fn, n_replays: int = 24, calls: int = 0):
        """Per-call time of each of n_replays replays of one graph of `calls` calls (default: one call per
        rotating input set, at most 64), each replay bracketed by its own events: (median, min, max) us."""
        torch = self.torch
        G = calls or min(self.R, 64)
        g = self._graph(fn, 0, G)
        g.replay()
        torch.cuda.synchronize()
        ts = []
        for _ in range(n_replays):
            e0, e1 = torch.cuda.Event(enable_timing=True), torch.cuda.Event(enable_timing=True)
            e0.record()
            g.replay()
            e1.record()
            torch.cuda.synchronize()
            ts.append(e0.elapsed_time(e1) * 1e3 / G)
        return statistics.median(ts), min(ts), max(ts)

    def single_calls(self, fn, n: int = 24):
        """Eager calls (host launch included), each timed alone with events after the previous one
        finished: median us."""
        torch = self.torch
        for i in range(3):
            fn(i)
        torch.cuda.synchronize()
        ts = []
        for i in range(n):
            e0, e1 = torch.cuda.Event(enable_timing=True), torch.cuda.Event(enable_timing=True)
            e0.record()
            fn(i)
            e1.record()
            torch.cuda.synchronize()
            ts.append(e0.elapsed_time(e1) * 1e3)
        return statistics.median(ts)

    def e2e(self, steps: int, warmup: int):
        """End to end through the public API with host buffers: every step copies its inputs from pinned
        host memory to the device, runs the decode call and reads out + lse back to pinned host memory.
        The steps are pipelined as a serving loop runs them: copies in on one stream, the decode on a
        second, copies out on a third, with two device buffer sets (each direction one copy of a slab
        holding the step's tensors), so step i + 1's inputs and step
        i - 1's results move while step i computes (events order each step's copy in -> decode -> copy
        out and keep a buffer set from being overwritten before it is read).  The loop of G steps is
        captured once as a CUDA graph (copies and launches) and replayed, as a serving loop does to keep
        the host's launch cost (about 15 us per decode call, measured separately) off the critical
        path."""
        torch = self.torch
        w0 = self.w0
        # a step's inputs sit in one pinned host slab and its results in another (views at 256-byte
        # offsets), so that each direction is one copy per step
        ins = (w0.q, w0.block_table, w0.topk_idx, w0.seq_lens)
        in_bytes = [t.numel() * t.element_size() for t in ins]
        in_off = [0]
        for nb in in_bytes:
            in_off.append(in_off[-1] + (nb + 255) // 256 * 256)

        def in_views(buf):
            return tuple(buf[in_off[i]:in_off[i] + in_bytes[i]].view(ins[i].dtype).view(ins[i].shape)
                         for i in range(len(ins)))

        out_bytes = self.out.numel() * self.out.element_size()
        out_off = (out_bytes + 255) // 256 * 256
        out_total = out_off + self.lse.numel() * self.lse.element_size()

        def out_views(buf):
            return (buf[:out_bytes].view(self.out.dtype).view(self.out.shape),
                    buf[out_off:out_total].view(self.lse.dtype).view(self.lse.shape))

        hosts = []
        for w in self.sets[:min(self.R, 16)]:
            hb = torch.empty(in_off[-1], dtype=torch.uint8).pin_memory()
            for v, t in zip(in_views(hb), (w.q, w.block_table, w.topk_idx, w.seq_lens)):
                v.copy_(t.cpu())
            hosts.append(hb)
        dev_in = [torch.empty(in_off[-1], dtype=torch.uint8, device=self.device) for _ in range(2)]
        dev_out = [torch.empty(out_total, dtype=torch.uint8, device=self.device) for _ in range(2)]
        host_out = [torch.empty(out_total, dtype=torch.uint8).pin_memory() for _ in range(2)]
        wss = [self.ws, self.api.alloc_workspace(self.dims, self.nsplit, self.device)]
        h2d = sum(in_bytes)
        d2h = out_bytes + self.lse.numel() * self.lse.element_size()
        s_in, s_comp, s_out = torch.cuda.Stream(), torch.cuda.Stream(), torch.cuda.Stream()
        ev = lambda: torch.cuda.Event()
        copied = [ev(), ev()]                       # inputs of buffer set k on the device
        computed = [ev(), ev()]                     # decode of buffer set k done (its inputs are free)
        read = [ev(), ev()]                         # results of buffer set k on the host (its outputs are free)

        def step(i, first):
            k = i & 1
            dq, dbt, dtk, dsl = in_views(dev_in[k])
            out, lse = out_views(dev_out[k])
            with torch.cuda.stream(s_in):
                if not first:
                    s_in.wait_event(computed[k])
                dev_in[k].copy_(hosts[i % len(hosts)], non_blocking=True)
                copied[k].record(s_in)
            with torch.cuda.stream(s_comp):
                s_comp.wait_event(copied[k])
                if not first:
                    s_comp.wait_event(read[k])
                self.api.sparse_mla_decode(dq, self.cache, dbt, dtk, dsl, w0.sm_scale, out=out, lse=lse,
                                           workspace=wss[k], nsplit=self.nsplit, stream=s_comp,
                                           heads_per_cta=self.plan.heads_per_cta, merge=self.dims.merge)
                computed[k].record(s_comp)
            with torch.cuda.stream(s_out):
                s_out.wait_event(computed[k])
                host_out[k].copy_(dev_out[k], non_blocking=True)
                read[k].record(s_out)

        def loop(n, start):
            cur = torch.cuda.current_stream()
            fork = ev()
            fork.record(cur)
            for s in (s_in, s_comp, s_out):
                s.wait_event(fork)
            for i in range(n):
                step(start + i, first=i < 2)
            for s in (s_in, s_comp, s_out):
                cur.wait_stream(s)

        loop(max(2, warmup), 0)                     # eager warm-up (and a check that the path runs)
        torch.cuda.synchronize()
        G = min(64, steps)
        reps, tail = divmod(steps, G)
        graphs = []
        for n in ([G] + ([tail] if tail else [])):
            g = torch.cuda.CUDAGraph()
            cap = torch.cuda.Stream()
            cap.wait_stream(torch.cuda.current_stream())
            with torch.cuda.graph(g, stream=cap):
                loop(n, 0)
            graphs.append(g)
        torch.cuda.synchronize()
        graphs[0].replay()                          # upload
        torch.cuda.synchronize()
        e0, e1 = torch.cuda.Event(enable_timing=True), torch.cuda.Event(enable_timing=True)
        e0.record()
        for _ in range(reps):
            graphs[0].replay()
        if tail:
            graphs[1].replay()
        e1.record()
        torch.cuda.synchronize()
        return e0.elapsed_time(e1) * 1e3 / steps, h2d, d2h


def measure_config(name: str, device, steps: int, warmup: int, peak_gbs: float):
    b = Bench(name, device)
    t = b.timed(b.call, steps, warmup)
    us = t * 1e6 / steps
    ts = b.timed(b.split_only, steps, warmup)
    us_split = ts * 1e6 / steps
    # other views of the same call: the median over graph replays (rotating inputs), the same with one
    # input set replayed (warm L2: labelled, not the metric), and eager single calls (host launch included)
    med, lo, hi = b.replay_stats(b.call)
    warm, _, _ = b.replay_stats(lambda i: b.call(0), calls=16)
    single = b.single_calls(b.call)
    gbs = b.bytes_per_call / (us * 1e-6) / 1e9
    b.append_setup()
    ta = b.timed(b.append_only, steps, warmup)
    us_app = ta * 1e6 / steps
    try:
        b.topk_setup()
        tt = b.timed(b.topk_only, steps, warmup)
        us_tk = tt * 1e6 / steps
        tp = b.timed(b.topk_then_decode, steps, warmup)
        us_pipe = tp * 1e6 / steps
        topk = {"queries": b.w0.B, "positions": b.tk_cols, "k": b.tk_out.shape[1],
                "scores": "standard normal float32", "rotating_sets": len(b.tk_sets),
                "us_per_call": round(us_tk, 3), "algorithmic_bytes": b.tk_bytes,
                "gbs": round(b.tk_bytes / (us_tk * 1e-6) / 1e9, 1),
                "roofline_frac": round(b.tk_bytes / (us_tk * 1e-6) / 1e9 / peak_gbs, 4),
                "then_decode_us_per_call": round(us_pipe, 3)}
    except Exception as e:  # a side measurement: keep the decode's numbers
        topk = {"error": repr(e)}
    res = {"us_per_call": round(us, 3), "split_kernel_us": round(us_split, 3), "nsplit": b.nsplit,
           "heads_per_cta": b.plan.heads_per_cta,
           "ctas": b.plan.ctas, "algorithmic_bytes": b.bytes_per_call, "gbs": round(gbs, 1),
           "roofline_frac_call": round(gbs / peak_gbs, 4),
           "roofline_frac_split_kernel": round(b.bytes_per_call / (us_split * 1e-6) / 1e9 / peak_gbs, 4),
           "rotations": b.R,
           "graph_replays": {"replays": 24, "calls_per_replay": min(b.R, 64), "median_us_per_call": round(med, 3),
                             "min": round(lo, 3), "max": round(hi, 3)},
           "warm_l2_us_per_call": round(warm, 3),
           "single_call_us": round(single, 3),
           "kv_append": {"tokens": b.w0.B, "us_per_call": round(us_app, 3), "algorithmic_bytes": b.app_bytes,
                         "gbs": round(b.app_bytes / (us_app * 1e-6) / 1e9, 1)},
           "topk_select": topk}
    del b
    import torch
    torch.cuda.empty_cache()
    return res


def cpu_oracle_sample(name: str, target_s: float = 15.0, max_queries: int = None):
    """Time the float64 oracle on a bounded sample of the workload on this host; returns
    (us per full call, queries timed, threads)."""
    import numpy as np
    import torch
    import oracle
    from sparse_mla_decode_paged_gb300 import workloads as wl
    import dataclasses
    spec = wl.CONFIGS[name]
    # the same recipe for a few queries on the host: per-query oracle work does not depend on the others
    small = dataclasses.replace(spec, B=min(spec.B, 4), pool_pages=None)
    w = wl.make_workload(small, device="cpu")
    q = w.q.view(torch.int16).numpy().view(np.uint16)
    kv, bt, tk, sl = w.kv_cache.numpy(), w.block_table.numpy(), w.topk_idx.numpy(), w.seq_lens.numpy()
    done, t0 = 0, time.perf_counter()
    order = list(range(w.B))
    while True:
        b = order[done % w.B]
        oracle.sparse_mla_decode(q[b:b + 1], kv, bt[b:b + 1], tk[b:b + 1], sl[b:b + 1], w.sm_scale)
        done += 1
        el = time.perf_counter() - t0
        if el >= target_s or (max_queries and done >= max_queries):
            break
    per_query = el / done
    return per_query * spec.B * 1e6, done, w.B


_WORKER_DATA = {}


def _oracle_worker(args):
    """One worker of the all-cores oracle baseline: runs single-query oracle calls over the saved host
    sample for target_s seconds (timed from after its own data load) and returns (calls, seconds)."""
    path, target_s, wid = args
    import numpy as np
    import oracle
    if path not in _WORKER_DATA:
        d = np.load(path)
        _WORKER_DATA[path] = {k: d[k] for k in d.files}
    d = _WORKER_DATA[path]
    B = d["q"].shape[0]
    sm_scale = float(d["sm_scale"])
    n, t0 = 0, time.perf_counter()
    while True:
        b = (wid + n) % B
        oracle.sparse_mla_decode(d["q"][b:b + 1], d["kv"], d["bt"][b:b + 1], d["tk"][b:b + 1], d["sl"][b:b + 1],
                                 sm_scale)
        n += 1
        el = time.perf_counter() - t0
        if el >= target_s:
            return n, el


class OraclePool:
    """The float64 oracle on every host core: a spawned process pool (one BLAS thread per process)
    over single-query calls on a host sample of the workload (per-query oracle work does not depend on
    the other queries).  Spawned, so it is safe after CUDA was initialised in this process."""

    def __init__(self, name: str, procs: int = 0):
        import multiprocessing as mp
        import tempfile
        import dataclasses
        import numpy as np
        import torch
        from sparse_mla_decode_paged_gb300 import workloads as wl
        spec = wl.CONFIGS[name]
        self.B_full = spec.B
        self.procs = procs or len(os.sched_getaffinity(0))
        small = dataclasses.replace(spec, B=min(spec.B, 8), pool_pages=None)
        w = wl.make_workload(small, device="cpu")
        d = "/dev/shm" if os.path.isdir("/dev/shm") else None
        fd, self.path = tempfile.mkstemp(suffix=".npz", dir=d)
        os.close(fd)
        np.savez(self.path, q=w.q.view(torch.int16).numpy().view(np.uint16), kv=w.kv_cache.numpy(),
                 bt=w.block_table.numpy(), tk=w.topk_idx.numpy(), sl=w.seq_lens.numpy(),
                 sm_scale=np.float64(w.sm_scale))
        self.drawn = w.B
        for v in ("OMP_NUM_THREADS", "OPENBLAS_NUM_THREADS", "MKL_NUM_THREADS"):
            os.environ[v] = "1"      # inherited by the spawned workers
        self.pool = mp.get_context("spawn").Pool(self.procs)
        self.pool.map(_oracle_worker, [(self.path, 0.05, i) for i in range(self.procs)], chunksize=1)   # load

    def us_per_call(self, target_s: float):
        """Microseconds per full call of the workload, all workers running for ~target_s."""
        res = self.pool.map(_oracle_worker, [(self.path, target_s, i) for i in range(self.procs)], chunksize=1)
        rate = sum(n / el for n, el in res)              # queries per second over all workers
        return self.B_full / rate * 1e6, sum(n for n, _ in res)

    def close(self):
        self.pool.terminate()
        self.pool.join()
        try:
            os.remove(self.path)
        except OSError:
            pass


def cpu_baselines(name: str, target_s: float):
    """The oracle as it stands on one host core and on every host core (the latter the line's value)."""
    one_us, n1, drawn = cpu_oracle_sample(name, target_s)
    pool = OraclePool(name)
    try:
        all_us, n_all = pool.us_per_call(target_s)
    finally:
        pool.close()
    return {"value": round(all_us, 1), "unit": UNIT, "cores": pool.procs, "kind": "oracle",
            "sample": f"{n_all} single-query float64 oracle runs over {pool.drawn} queries drawn with the {name} "
                      f"recipe, {pool.procs} spawned processes (one BLAS thread each) for ~{target_s:.0f} s, "
                      f"scaled to a full call of {pool.B_full} queries",
            "single_core": {"value": round(one_us, 1), "unit": UNIT, "cores": 1,
                            "sample": f"{n1} single-query oracle runs cycling over {drawn} queries, one thread, "
                                      f"~{target_s:.0f} s, scaled to a full call"}}


def run_cpu_baseline_subprocess(name: str, target_s: float):
    """Run the oracle timings in a child with BLAS pinned to one thread per process (so `cores` is exact)
    and no GPU visible."""
    env = dict(os.environ, OMP_NUM_THREADS="1", OPENBLAS_NUM_THREADS="1", MKL_NUM_THREADS="1",
               CUDA_VISIBLE_DEVICES="")
    code = ("import json,sys; sys.path.insert(0, %r); import bench; "
            "print(json.dumps(bench.cpu_baselines(%r, %f)))" % (ROOT, name, target_s))
    r = subprocess.run([sys.executable, "-c", code], capture_output=True, text=True, env=env, timeout=900)
    if r.returncode != 0:
        return {"error": r.stderr[-300:]}
    return json.loads(r.stdout.strip().splitlines()[-1])


def main_ours(args):
    import torch
    rank, world, local = dist_env()
    if world > 1:
        import torch.distributed as dist
        torch.cuda.set_device(local)
        dist.init_process_group("nccl")
    dev = torch.device("cuda", local if world > 1 else torch.cuda.current_device())
    torch.cuda.set_device(dev)
    peak, peak_kind = measured_peaks()
    name = args.workload
    b = Bench(name, dev, seed_offset=rank)
    if args.steps:
        steps = args.steps
    else:
        # about one second of timed calls (enough for clock samples), at least one rotation cycle
        probe = b.timed(b.call, b.R, 3, world)
        steps = int(min(200000, max(b.R, 1.0 / max(probe / b.R, 1e-7))))
    visible = [x.strip() for x in os.environ.get("CUDA_VISIBLE_DEVICES", "").split(",") if x.strip()]
    gpu_index = visible[local] if local < len(visible) else str(dev.index)
    with ClockSampler(gpu_index) as clk:
        clk.wait_first()
        clk.mark()
        # the sampler sees the GPU under load: 1.2 s of the same replays run right before each timed region
        t = b.timed(b.call, steps, args.warmup, world, preroll_s=1.2)
        ts = b.timed(b.split_only, steps, args.warmup, 1, preroll_s=0.4)
    clocks = clk.summary()
    clocks["window"] = "nvidia-smi every 200 ms over the timed regions and the 1.2 s / 0.4 s of identical " \
                       "untimed replays that precede them"
    us = aggregate_us_per_call(t, steps, world)
    us_rank = t * 1e6 / steps
    us_split = ts * 1e6 / steps
    e2e_us, h2d, d2h = b.e2e(min(steps, 2000), max(3, args.warmup))
    e2e_us = reduce_max(e2e_us, world) / world
    achieved = b.bytes_per_call / (us_split * 1e-6) / 1e9
    achieved_call = b.bytes_per_call / (us_rank * 1e-6) / 1e9
    line = {
        "metric": METRIC, "value": round(us, 3), "unit": UNIT, "n_gpus": world, "steps": steps,
        "warmup": args.warmup, "ms_per_step": round(us_rank / 1e3, 6), "higher_is_better": False,
        "scaling": "weak", "vs_baseline": None, "dtype": "fp16", "data": "synthetic",
        "config": {"workload": name, "B": b.w0.B, "H": b.w0.H, "topk": b.w0.topk,
                   "ctx": b.spec.ctx if b.spec.ctx else "log-uniform 64..524288",
                   "cache_pages": b.cache.shape[0], "nsplit": b.nsplit, "ctas": b.plan.ctas,
                   "timing": "CUDA graph replays, events on the launching stream",
                   "l2": f"inputs larger than L2: {b.R} rotating input sets x {b.bytes_per_call} B "
                         f">= 4 x L2 ({b.l2} B)",
                   "parallelism": f"replica per GPU x{world}"},
        "gbs": round(b.bytes_per_call / (us_rank * 1e-6) / 1e9, 1),
        "roofline": {"bound": "hbm", "achieved": round(achieved, 1), "peak": peak, "unit": "GB/s",
                     "frac": round(achieved / peak, 4), "traffic": recorded_traffic(name),
                     "kernel": "split kernel alone (the dominant kernel): the call's algorithmic bytes over "
                               "its own event-timed duration",
                     "kernel_us": round(us_split, 3),
                     "algorithmic_bytes_per_launch": b.bytes_per_call, "peak_source": peak_kind,
                     "call": {"achieved": round(achieved_call, 1), "frac": round(achieved_call / peak, 4),
                              "us": round(us_rank, 3),
                              "what": "whole decode call (split kernel + merge when nsplit > 1)"}},
        "e2e": {"value": round(e2e_us, 3), "unit": UNIT, "h2d_bytes_per_step": h2d, "d2h_bytes_per_step": d2h},
        "gpu_launches": steps * b.launches_per_call(),
        "clocks": clocks,
    }
    del b
    torch.cuda.empty_cache()
    if rank == 0 and world == 1 and not args.no_per_config:
        per = {}
        for n in ALL_CONFIGS:
            try:
                per[n] = measure_config(n, dev, 600 if n in ("tiny", "bs1_ctx8k") else 200, 10, peak)
            except Exception as e:  # a config that does not fit must not hide the headline line
                per[n] = {"error": repr(e)[:200]}
        line["per_config"] = per
    if rank == 0 and world == 1 and not args.no_cpu_baseline:
        line["cpu_baseline"] = run_cpu_baseline_subprocess(name, 15.0)
    if rank == 0:
        print(json.dumps(line), flush=True)
    if world > 1:
        import torch.distributed as dist
        dist.destroy_process_group()


def main_reference(args):
    rank, world, _ = dist_env()
    if rank != 0:
        return
    for v in ("OMP_NUM_THREADS", "OPENBLAS_NUM_THREADS", "MKL_NUM_THREADS"):
        os.environ[v] = "1"          # before numpy loads: one BLAS thread per oracle process
    name = args.workload
    steps, warmup = args.steps or 5, args.warmup
    per_step_target = max(0.5, 120.0 / max(1, steps + warmup))
    pool = OraclePool(name)
    try:
        for _ in range(warmup):
            pool.us_per_call(min(0.5, per_step_target / 4))
        vals, done = [], 0
        t0 = time.perf_counter()
        for _ in range(steps):
            us, n = pool.us_per_call(per_step_target)
            vals.append(us)
            done += n
        el = time.perf_counter() - t0
    finally:
        pool.close()
    value = statistics.mean(vals)
    line = {"impl": "reference", "metric": METRIC, "value": round(value, 1), "unit": UNIT, "n_gpus": world,
            "steps": steps, "warmup": warmup, "ms_per_step": round(value / 1e3, 3), "higher_is_better": False,
            "scaling": "weak", "vs_baseline": None, "dtype": "f64", "data": "synthetic",
            "config": {"workload": name, "what": "float64 CPU oracle on every host core (a spawned process per "
                                                 "core over single-query calls); each step times a bounded "
                                                 "sample of queries and scales to a full call"},
            "cpu_baseline": {"value": round(value, 1), "unit": UNIT, "cores": pool.procs, "kind": "oracle",
                             "sample": f"per step ~{per_step_target:.1f} s of oracle work on {pool.procs} processes "
                                       f"over {pool.drawn} queries of {name} ({done} single-query runs in all), "
                                       f"scaled to all {pool.B_full} queries"},
            "e2e": {"value": round(value, 1), "unit": UNIT, "h2d_bytes_per_step": 0, "d2h_bytes_per_step": 0},
            "wall_s": round(el, 1)}
    print(json.dumps(line), flush=True)


def main():
    ap = argparse.ArgumentParser()
    ap.add_argument("--gpus", type=int, default=1)
    ap.add_argument("--steps", type=int, default=0)
    ap.add_argument("--warmup", type=int, default=10)
    ap.add_argument("--workload", default=HEADLINE, choices=ALL_CONFIGS)
    ap.add_argument("--impl", default="ours", choices=["ours", "reference"])
    ap.add_argument("--no-per-config", action="store_true")
    ap.add_argument("--no-cpu-baseline", action="store_true")
    ap.add_argument("--single", type=int, default=0,
                    help="profiling driver: run this many eager calls of --workload (optionally --nsplit) and exit")
    ap.add_argument("--nsplit", type=int, default=0)
    ap.add_argument("--ctx", type=int, default=0,
                    help="with --single: context length per query instead of the workload's (ragged: the upper end)")
    ap.add_argument("--single-op", choices=("decode", "topk"), default="decode",
                    help="with --single: the decode call, or the top-k selection over the workload's contexts")
    args = ap.parse_args()
    if args.single and args.single_op == "topk":
        import torch
        from sparse_mla_decode_paged_gb300 import api
        from sparse_mla_decode_paged_gb300 import workloads as wl
        # the workload's lengths (the same draw as its decode inputs) and score rows; no cache
        spec = wl.CONFIGS[args.workload]
        lens = torch.tensor(wl.draw_context_lengths(spec, wl._gen("cuda", spec.seed), "cuda"),
                            dtype=torch.int32, device="cuda")
        scores = wl.make_indexer_scores(spec.B, int(lens.max().item()), seed=5000, device="cuda")
        for _ in range(args.single):
            api.sparse_mla_topk_select(scores, lens, spec.topk)
        torch.cuda.synchronize()
        return
    if args.single:
        import dataclasses
        import torch
        from sparse_mla_decode_paged_gb300 import api
        from sparse_mla_decode_paged_gb300 import workloads as wl
        spec = wl.CONFIGS[args.workload]
        if args.ctx:
            # the same batch, heads and top-k list length over shorter contexts: the kernels do the same work
            # per query, the cache holds only the pages used (a few GB at most, for profiling)
            spec = (dataclasses.replace(spec, ragged_hi=args.ctx, pool_pages=None) if spec.ctx is None
                    else dataclasses.replace(spec, ctx=args.ctx, pool_pages=None))
        w = wl.make_workload(spec, device="cuda")
        for _ in range(args.single):
            api.sparse_mla_decode(w.q, w.kv_cache, w.block_table, w.topk_idx, w.seq_lens, w.sm_scale,
                                  nsplit=args.nsplit)
        torch.cuda.synchronize()
        print("ok")
        return
    if args.warmup < 3:
        args.warmup = 3
    if args.impl == "reference":
        main_reference(args)
    else:
        main_ours(args)


if __name__ == "__main__":
    main()
