#!/usr/bin/env python3
"""Benchmark of the SwiAttn routed-attention hot path on GB300.

Headline: routed prefill (swiattn_prefill: gate scheduling + tensor-core
attention) on the long-context workload B=1, H=16, d=128, N=32768, W=1024,
gates in runs at routed fraction 0.13, reported as useful TFLOP/s (4*d per
visited query-key pair).  The same run also measures decode KV-read GB/s
(16 sequences x 32768 cached tokens), the 'easy' 0.05 prefill, the router
GEMV and the dual-branch training forward, each on its own workload.

    python bench.py [--gpus N] [--steps K] [--warmup W] [--impl ours|reference]

One JSON line is printed by rank 0.  Under torchrun every rank runs its own
independent sequence (weak scaling, no collective on the data path).
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
import tempfile
import time
import datetime

import numpy as np
import torch

ROOT = os.path.dirname(os.path.abspath(__file__))
sys.path.insert(0, ROOT)

import swiattn_inputs as inp  # noqa: E402

METRIC = "prefill useful TFLOP/s at N=32K (% of bf16 peak); decode KV-read GB/s"
FALLBACK_PEAKS = {"hbm_gbs": 6800.0, "bf16_tflops": 1900.0, "bf16_tflops_sustained": 1700.0}
L2_FLUSH_BYTES = 256 << 20

# DRAM traffic per launch of the dominant kernels (dram__bytes_read.sum +
# dram__bytes_write.sum from ncu on the default workloads), keyed by the
# SHA-256 of the kernel's source files at capture time; a kernel whose source
# has changed since reports null.
MEASURED_TRAFFIC = {
    # prefill_kernel, long-context prefill N=32768 f=0.13 (far items head by head):
    # 727 854 336 read + 121 214 976 written
    ("prefill", "532909cf403d4c6c"): 727854336 + 121214976,
    # decode_split2_kernel (persistent CTAs), 16 x 32768 decode: 654 431 488 read + 4 102 656 written
    ("decode", "97db57687c228419"): 654431488 + 4102656,
    # dual_kernel, dual-branch workload B=2 N=8192 GQA 16/4: 144 400 384 read + 270 856 192 written
    ("dual", "0d140f1582e3c2ea"): 144400384 + 270856192,
    # dkdv_kernel + dq_kernel, backward on the dual workload: (315 288 064 + 22 582 016)
    # + (254 839 296 + 48 433 152)
    ("backward", "789f57cbf56f040a"): 315288064 + 22582016 + 254839296 + 48433152,
    # route_kernel, 32768 tokens x 2048: 134 248 192 read + 2 795 520 written
    ("route", "4a5c0b7bf6e2d8ed"): 134248192 + 2795520,
    # route_bwd_logit + dh + reduce kernels, 16384 tokens: (201 534 208 + 3 031 552)
    # + (67 196 672 + 17 656 064) + (2 171 904 + 0); most dh rows are still in L2 at the end
    ("route_backward", "8a50a8de2fb87f90"): 201534208 + 3031552 + 67196672 + 17656064 + 2171904,
}
# Source text each stored count depends on: whole files, or a file up to a
# marker (the device code of a kernel file, before its host launcher; the
# decode split kernel, before the combine).  The prefill's count also depends
# on the order of its work list (schedule.cu, up to the fused router kernel).
KERNEL_SOURCES = {"prefill": (("attn_prefill.cu", "cudaError_t launch_prefill_tc("), "ptx.cuh",
                              ("schedule.cu", "// Router GEMV fused with the schedule")),
                  "decode": (("decode.cu", "// Log-sum-exp merge of the chunk partials"),),
                  "dual": (("attn_dual.cu", "cudaError_t launch_dual_tc("), "ptx.cuh"),
                  "backward": (("attn_bwd.cu", "cudaError_t launch_bwd_dkdv("), "ptx.cuh"),
                  "route": ("route.cu", "route_gemv.cuh"),
                  "route_backward": ("bwd_simt.cu",)}


def kernel_source_hash(kernel: str) -> str:
    h = hashlib.sha256()
    for entry in KERNEL_SOURCES[kernel]:
        name, marker = (entry, None) if isinstance(entry, str) else entry
        path = os.path.join(ROOT, "sliding_window_attention_router_gb300", "csrc", name)
        with open(path, "rb") as f:
            data = f.read()
        if marker is not None:
            data = data[:data.index(marker.encode())]
        h.update(data)
    return h.hexdigest()[:16]


def measured_traffic(kernel: str):
    return MEASURED_TRAFFIC.get((kernel, kernel_source_hash(kernel)))


def load_peaks():
    path = os.path.join(ROOT, "MEASURED_PEAKS.json")
    if os.path.exists(path):
        with open(path) as f:
            return json.load(f), "measured"
    return dict(FALLBACK_PEAKS), "fallback"


def useful_pairs(gate: np.ndarray, W: int, S: int = 0) -> int:
    """Visited (query, key) pairs per head: routed rows i+1, window rows
    min(i+1, W) plus their global anchors below the window, min(S, i-W+1)."""
    B, N = gate.shape
    i = np.arange(N, dtype=np.int64)[None, :]
    window = np.minimum(i + 1, W) + np.clip(np.minimum(S, i - W + 1), 0, None)
    n = np.where(gate != 0, i + 1, window)
    return int(n.sum())


# ------------------------------------------------------------------ dist --
class Dist:
    def __init__(self):
        self.world = int(os.environ.get("WORLD_SIZE", "1"))
        self.rank = int(os.environ.get("RANK", "0"))
        self.local_rank = int(os.environ.get("LOCAL_RANK", "0"))
        self.pg = None
        if self.world > 1:
            import torch.distributed as dist
            backend = "nccl" if torch.cuda.is_available() else "gloo"
            dist.init_process_group(backend=backend)
            self.pg = dist

    def barrier(self):
        if self.pg:
            if torch.cuda.is_available():
                self.pg.barrier(device_ids=[self.local_rank])
            else:
                self.pg.barrier()

    def max(self, x: float) -> float:
        return self._reduce(x, "max")

    def sum(self, x: float) -> float:
        return self._reduce(x, "sum")

    def _reduce(self, x: float, op: str) -> float:
        if not self.pg:
            return float(x)
        dev = torch.device("cuda", self.local_rank) if torch.cuda.is_available() else "cpu"
        t = torch.tensor([float(x)], dtype=torch.float64, device=dev)
        self.pg.all_reduce(t, op=self.pg.ReduceOp.MAX if op == "max" else self.pg.ReduceOp.SUM)
        return float(t.item())

    def close(self):
        if self.pg:
            self.pg.destroy_process_group()


def aggregate(units_per_rank: float, seconds_per_rank: float, dist: Dist):
    """Whole-job throughput: units summed over ranks / slowest rank's time."""
    total = dist.sum(units_per_rank)
    slowest = dist.max(seconds_per_rank)
    return total / slowest, slowest


# ---------------------------------------------------------------- clocks --
class ClockSampler:
    FIELDS = ("clocks.sm,clocks.max.sm,power.draw,clocks_event_reasons.hw_slowdown,"
              "clocks_event_reasons.hw_thermal_slowdown,clocks_event_reasons.sw_thermal_slowdown,"
              "clocks_event_reasons.sw_power_cap")

    def __init__(self, gpu_index: int):
        self.proc = None
        self.path = None
        try:
            fd, self.path = tempfile.mkstemp(prefix="swiattn_clocks_", suffix=".csv")
            os.close(fd)
            self.fh = open(self.path, "w")
            self.proc = subprocess.Popen(
                ["nvidia-smi", "-i", str(gpu_index), f"--query-gpu=timestamp,{self.FIELDS}",
                 "--format=csv,noheader,nounits", "-lms", "100"],
                stdout=self.fh, stderr=subprocess.DEVNULL)
        except (OSError, FileNotFoundError):
            self.proc = None

    def stop(self, t_from=None, t_to=None):
        """Stop sampling; summarise the samples taken between the host times
        t_from and t_to (datetime, local clock) when given."""
        if not self.proc:
            return None
        self.proc.terminate()
        try:
            self.proc.wait(timeout=5)
        except subprocess.TimeoutExpired:
            self.proc.kill()
        self.fh.close()
        rows = []
        with open(self.path) as f:
            for line in f:
                parts = [p.strip() for p in line.split(",")]
                if len(parts) != 8:
                    continue
                if t_from is not None:
                    try:
                        ts = datetime.datetime.strptime(parts[0], "%Y/%m/%d %H:%M:%S.%f")
                    except ValueError:
                        continue
                    if ts < t_from or ts > t_to:
                        continue
                rows.append(parts)
        os.unlink(self.path)
        if not rows:
            return {"sm_mhz": None, "sm_max_mhz": None, "reasons": [], "samples": 0}

        def num(x):
            try:
                return float(x)
            except ValueError:
                return None

        sm = [num(r[1]) for r in rows if num(r[1]) is not None]
        power = [num(r[3]) for r in rows if num(r[3]) is not None]
        names = ["hw_slowdown", "hw_thermal_slowdown", "sw_thermal_slowdown", "sw_power_cap"]
        reasons = sorted({names[k] for r in rows for k in range(4) if r[4 + k] == "Active"})
        return {"sm_mhz": statistics.median(sm) if sm else None,
                "sm_max_mhz": num(rows[0][2]), "reasons": reasons, "samples": len(rows),
                "power_w_max": max(power) if power else None}


# ----------------------------------------------------------------- timing --
class Timer:
    """Per-step CUDA-event timing with an L2 flush before every step."""

    def __init__(self, device):
        self.flush = torch.empty(L2_FLUSH_BYTES, dtype=torch.uint8, device=device)
        self.sink = torch.zeros((), dtype=torch.float32, device=device)

    def flush_l2(self):
        """Write a buffer twice the size of L2, then read it back.  The write
        evicts every line the previous step left; the read makes the flush's
        own dirty lines (up to the size of L2) go back to HBM here, before the
        timer starts, instead of inside the timed kernel, where their
        write-back would add up to 129 MB of traffic that is not the kernel's."""
        self.flush.zero_()
        torch.sum(self.flush.view(torch.float32), dim=0, out=self.sink)

    def hold(self, fn, seconds: float):
        """Keep running fn (untimed) for about `seconds`, so clock sampling sees
        the kernel under sustained load."""
        t0 = time.perf_counter()
        while time.perf_counter() - t0 < seconds:
            for _ in range(8):
                fn()
            torch.cuda.synchronize()

    def run(self, fn, steps: int, warmup: int, kernel_events: bool = False):
        """Warm up, then time `steps` calls (L2 flushed before each).  With
        kernel_events, a second loop of `steps` calls times the library's
        dominant kernel alone through its event hook; the step times come from
        the first loop, which records nothing between the library's launches
        (a recorded event there would serialise a programmatic dependent
        launch)."""
        import sliding_window_attention_router_gb300 as swa
        for _ in range(warmup):
            self.flush_l2()
            fn()
        torch.cuda.synchronize()
        starts = [torch.cuda.Event(enable_timing=True) for _ in range(steps)]
        stops = [torch.cuda.Event(enable_timing=True) for _ in range(steps)]
        for s in range(steps):
            self.flush_l2()
            starts[s].record()
            fn()
            stops[s].record()
        torch.cuda.synchronize()
        step_ms = [a.elapsed_time(b) for a, b in zip(starts, stops)]
        if not kernel_events:
            return step_ms, None
        ks = [torch.cuda.Event(enable_timing=True) for _ in range(steps)]
        ke = [torch.cuda.Event(enable_timing=True) for _ in range(steps)]
        # torch creates events lazily: record once so the handles exist
        # before the library records them around its kernel.
        for e in ks + ke:
            e.record()
        torch.cuda.synchronize()
        for s in range(steps):
            self.flush_l2()
            swa.set_profile_events(ks[s], ke[s])
            fn()
        swa.set_profile_events(None, None)
        torch.cuda.synchronize()
        kern_ms = [a.elapsed_time(b) for a, b in zip(ks, ke)]
        return step_ms, kern_ms


# ------------------------------------------------------------ workloads --
def prefill_section(swa, timer, dev, frac, steps, warmup, seed, with_e2e, N=32768, hold_s=0.0):
    d = inp.prefill_32k(frac=frac, seed=seed, N=N)
    B, N, H, D, W = d["B"], d["N"], d["Hq"], d["d"], d["W"]
    pairs = useful_pairs(d["gate"].numpy(), W)
    flops = 4.0 * D * H * pairs
    host = {k: d[k].pin_memory() for k in ("q", "k", "v", "gate")}
    q, k, v, gate = (host[n].to(dev, non_blocking=True) for n in ("q", "k", "v", "gate"))
    o = torch.empty_like(q)
    ws = torch.empty(swa.prefill_workspace(B, N, H, H, D, W, torch.bfloat16), dtype=torch.uint8,
                     device=dev)
    scale = 1.0 / math.sqrt(D)

    def step():
        swa.prefill(q, k, v, gate, W, scale, out=o, workspace=ws)

    t_from = datetime.datetime.now()
    step_ms, kern_ms = timer.run(step, steps, warmup, kernel_events=True)
    if hold_s > 0:
        timer.hold(step, hold_s)
    t_to = datetime.datetime.now()
    assert swa.get_device_error() == 0, "device-side wait timed out"
    res = dict(d=d, flops=flops, pairs=pairs, step_ms=step_ms, kern_ms=kern_ms,
               realised_frac=float(d["gate"].float().mean()), t_from=t_from, t_to=t_to)
    if with_e2e:
        # End to end through the host-buffer entry point: every step copies
        # q, k, v, gate from pinned host memory, runs the prefill and copies o
        # back, all enqueued by swiattn_prefill_host on the current stream.
        o_host = torch.empty(o.shape, dtype=o.dtype, pin_memory=True)
        ws_host = torch.empty(swa.prefill_host_workspace(B, N, H, H, D, W, torch.bfloat16),
                              dtype=torch.uint8, device=dev)

        def e2e_step():
            swa.prefill_host(host["q"], host["k"], host["v"], host["gate"], W, scale, out=o_host,
                             workspace=ws_host, device=dev)

        e2e_ms, _ = timer.run(e2e_step, max(3, steps // 2), 2)
        h2d = sum(host[n].numel() * host[n].element_size() for n in host)
        d2h = o_host.numel() * o_host.element_size()
        # The same calls issued as a stream of requests: consecutive calls
        # alternate between two streams (each with its own workspace and host
        # output), so one call's upload can overlap the previous call's
        # attention and download; timed from the first upload to the last
        # download.  Every call still copies its inputs in and its output out.
        pipe = [(torch.cuda.Stream(dev), ws_host, o_host),
                (torch.cuda.Stream(dev),
                 torch.empty_like(ws_host), torch.empty(o.shape, dtype=o.dtype, pin_memory=True))]

        def e2e_pipelined(n):
            main_s = torch.cuda.current_stream(dev)
            t0, t1 = torch.cuda.Event(enable_timing=True), torch.cuda.Event(enable_timing=True)
            t0.record(main_s)
            for st, _, _ in pipe:
                st.wait_stream(main_s)
            for i in range(n):
                st, ws_i, o_i = pipe[i % 2]
                with torch.cuda.stream(st):
                    swa.prefill_host(host["q"], host["k"], host["v"], host["gate"], W, scale,
                                     out=o_i, workspace=ws_i, device=dev)
            for st, _, _ in pipe:
                main_s.wait_stream(st)
            t1.record(main_s)
            torch.cuda.synchronize()
            return t0.elapsed_time(t1)

        n_pipe = max(4, steps)
        e2e_pipelined(2)
        pipe_ms = e2e_pipelined(n_pipe)
        res.update(e2e_ms=e2e_ms, h2d=h2d, d2h=d2h, e2e_pipe_ms=pipe_ms, e2e_pipe_n=n_pipe)
    return res


def decode_section(swa, timer, dev, steps, warmup, seed, S=0, sweep_routed=()):
    B, L, H, D, W = 16, 32768, 16, 128, 1024
    g = torch.Generator(device=dev)
    g.manual_seed(seed)
    kc = torch.randn(B, L, H, D, generator=g, device=dev, dtype=torch.float32).to(torch.bfloat16)
    vc = torch.randn(B, L, H, D, generator=g, device=dev, dtype=torch.float32).to(torch.bfloat16)
    q = torch.randn(B, H, D, generator=g, device=dev, dtype=torch.float32).to(torch.bfloat16)
    gcpu = inp._gen(seed)
    gate = inp.bernoulli_gates((B,), 0.13, gcpu).to(dev)
    sl = torch.full((B,), L, dtype=torch.int32, device=dev)
    o = torch.empty_like(q)
    ws = torch.empty(swa.decode_workspace(B, L, H, H, D, W, torch.bfloat16), dtype=torch.uint8,
                     device=dev)
    n_routed = int(gate.sum())
    entries = n_routed * L + (B - n_routed) * (W + min(S, L - W))
    kv_bytes = entries * H * D * 2 * 2
    qo_bytes = 2 * B * H * D * 2
    if S:
        ws = torch.empty(swa.decode_anchored_workspace(B, L, H, H, D, W, S, torch.bfloat16),
                         dtype=torch.uint8, device=dev)

    def step():
        if S:
            swa.decode_anchored(q, kc, vc, sl, gate, W, S, out=o, workspace=ws)
        else:
            swa.decode(q, kc, vc, sl, gate, W, out=o, workspace=ws)

    step_ms, kern_ms = timer.run(step, steps, warmup, kernel_events=True)
    assert swa.get_device_error() == 0
    sweep = []
    if sweep_routed:
        # The same caches with the first n sequences routed, n = 0 .. B.
        for n in sweep_routed:
            gate.zero_()
            gate[:n] = 1
            sbytes = (n * L + (B - n) * W) * H * D * 2 * 2 + qo_bytes
            sm, km = timer.run(step, max(3, steps // 2), 2, kernel_events=True)
            sweep.append({"n_routed": n, "gbs": sbytes / (statistics.mean(sm) / 1e3) / 1e9,
                          "kernel_gbs": sbytes / (statistics.mean(km) / 1e3) / 1e9,
                          "ms_per_step": statistics.mean(sm)})
        assert swa.get_device_error() == 0
    del kc, vc
    return dict(step_ms=step_ms, kern_ms=kern_ms, bytes=kv_bytes + qo_bytes, n_routed=n_routed,
                sweep=sweep)


def anchored_prefill_section(swa, timer, dev, steps, warmup, seed, S=256):
    """The long-context prefill workload with S global anchors per window row
    (the SWA glossary's 256-token anchor set)."""
    d = inp.prefill_32k(frac=0.13, seed=seed)
    B, N, H, D, W = d["B"], d["N"], d["Hq"], d["d"], d["W"]
    q, k, v, gate = (d[n].to(dev) for n in ("q", "k", "v", "gate"))
    o = torch.empty_like(q)
    ws = torch.empty(swa.prefill_workspace(B, N, H, H, D, W, torch.bfloat16), dtype=torch.uint8,
                     device=dev)

    def step():
        swa.prefill(q, k, v, gate, W, out=o, workspace=ws, n_anchor=S)

    step_ms, kern_ms = timer.run(step, steps, warmup, kernel_events=True)
    assert swa.get_device_error() == 0
    flops = 4.0 * D * H * useful_pairs(d["gate"].numpy(), W, S)
    return dict(step_ms=step_ms, kern_ms=kern_ms, flops=flops)


def static_hybrid_section(swa, timer, dev, steps, warmup, seed):
    """Comparator: the static 3:1 hybrid (SWA blog, Mellum 2: three window layers
    then one full-attention layer, W = 1024) on the long-context prefill
    workload.  A step is one group of four layers (the same Q/K/V per layer);
    per-layer time compares with one routed layer at the report's average
    routed fraction."""
    d = inp.prefill_32k(frac=0.13, seed=seed)
    B, N, H, D, W = d["B"], d["N"], d["Hq"], d["d"], d["W"]
    q, k, v = (d[n].to(dev) for n in ("q", "k", "v"))
    zeros = torch.zeros((B, N), dtype=torch.uint8, device=dev)
    ones = torch.ones((B, N), dtype=torch.uint8, device=dev)
    o = torch.empty_like(q)
    ws = torch.empty(swa.prefill_workspace(B, N, H, H, D, W, torch.bfloat16), dtype=torch.uint8,
                     device=dev)

    def step():
        for g in (zeros, zeros, zeros, ones):
            swa.prefill(q, k, v, g, W, out=o, workspace=ws)

    step_ms, _ = timer.run(step, steps, warmup)
    assert swa.get_device_error() == 0
    zc, oc = np.zeros((B, N), np.uint8), np.ones((B, N), np.uint8)
    flops = 4.0 * D * H * (3 * useful_pairs(zc, W) + useful_pairs(oc, W))
    return dict(step_ms=step_ms, flops=flops)


def decode_paged_section(swa, timer, dev, steps, warmup, seed, page_size=64):
    """The decode workload on a paged cache: the same 16 x 32768 tokens, pages
    of page_size tokens placed in a shuffled pool."""
    B, L, H, D, W = 16, 32768, 16, 128, 1024
    g = torch.Generator(device=dev)
    g.manual_seed(seed)
    max_pages = L // page_size
    num_pages = B * max_pages
    kp = torch.randn(num_pages, page_size, H, D, generator=g, device=dev,
                     dtype=torch.float32).to(torch.bfloat16)
    vp = torch.randn(num_pages, page_size, H, D, generator=g, device=dev,
                     dtype=torch.float32).to(torch.bfloat16)
    q = torch.randn(B, H, D, generator=g, device=dev, dtype=torch.float32).to(torch.bfloat16)
    table = torch.randperm(num_pages, generator=inp._gen(seed)).to(torch.int32).view(B, max_pages)
    table = table.to(dev)
    gate = inp.bernoulli_gates((B,), 0.13, inp._gen(seed)).to(dev)
    sl = torch.full((B,), L, dtype=torch.int32, device=dev)
    o = torch.empty_like(q)
    ws = torch.empty(swa.decode_paged_workspace(B, max_pages, page_size, H, H, D, W, torch.bfloat16),
                     dtype=torch.uint8, device=dev)
    n_routed = int(gate.sum())
    entries = n_routed * L + (B - n_routed) * W
    nbytes = entries * H * D * 2 * 2 + 2 * B * H * D * 2

    def step():
        swa.decode_paged(q, kp, vp, table, sl, gate, W, out=o, workspace=ws)

    step_ms, kern_ms = timer.run(step, steps, warmup, kernel_events=True)
    assert swa.get_device_error() == 0
    del kp, vp
    return dict(step_ms=step_ms, kern_ms=kern_ms, bytes=nbytes, n_routed=n_routed)


def route_section(swa, timer, dev, steps, warmup, seed):
    T, Dm = 32768, 2048
    r = inp.router_inputs(T, Dm, torch.bfloat16, seed)
    h, w = r["h"].to(dev), r["w"].to(dev)
    logits = torch.empty(T, dtype=torch.float32, device=dev)
    gate = torch.empty(T, dtype=torch.uint8, device=dev)

    def step():
        swa.route(h, w, r["bias"], logits=logits, gate=gate)

    step_ms, kern_ms = timer.run(step, steps, warmup, kernel_events=True)
    nbytes = T * Dm * 2 + Dm * 2 + T * 5
    return dict(step_ms=step_ms, kern_ms=kern_ms, bytes=nbytes)


def layer_4k_section(swa, timer, dev, steps, warmup, seed):
    """Single-layer prefill: router GEMV + gate, then routed prefill on its gates,
    timed as the fused call (route_prefill) and as the two separate calls."""
    d = inp.prefill_4k(seed=seed)
    B, N, H, D, W = d["B"], d["N"], d["Hq"], d["d"], d["W"]
    h, w = d["h"].to(dev), d["w"].to(dev)
    q, k, v = (d[n].to(dev) for n in ("q", "k", "v"))
    logits = torch.empty(B * N, dtype=torch.float32, device=dev)
    gate = torch.empty(B * N, dtype=torch.uint8, device=dev)
    o = torch.empty_like(q)
    ws = torch.empty(swa.prefill_workspace(B, N, H, H, D, W, torch.bfloat16), dtype=torch.uint8,
                     device=dev)

    wsf = torch.empty(swa.route_prefill_workspace(B, N, H, H, D, W, torch.bfloat16),
                      dtype=torch.uint8, device=dev)
    logits_f = torch.empty((B, N), dtype=torch.float32, device=dev)
    gate_f = torch.empty((B, N), dtype=torch.uint8, device=dev)
    o_f = torch.empty_like(q)

    def separate():
        swa.route(h, w, d["bias"], logits=logits, gate=gate)
        swa.prefill(q, k, v, gate.view(B, N), W, out=o, workspace=ws)

    def fused():
        swa.route_prefill(h, w, d["bias"], q, k, v, W, out=o_f, logits=logits_f, gate=gate_f,
                          workspace=wsf)

    sep_ms, _ = timer.run(separate, steps, warmup)
    step_ms, _ = timer.run(fused, steps, warmup)
    assert swa.get_device_error() == 0
    assert torch.equal(gate_f.view(-1), gate)
    pairs = useful_pairs(gate.view(B, N).cpu().numpy(), W)
    return dict(step_ms=step_ms, separate_ms=sep_ms, flops=4.0 * D * H * pairs,
                routed_frac=float(gate.float().mean()))


def dual_section(swa, timer, dev, steps, warmup, seed):
    d = inp.dual_8k(seed=seed)
    B, N, Hq, Hkv, D, W = d["B"], d["N"], d["Hq"], d["Hkv"], d["d"], d["W"]
    q, k, v, lg, nll = (d[n].to(dev) for n in ("q", "k", "v", "logits", "nll"))
    outs = dict(o_full=torch.empty_like(q), o_swa=torch.empty_like(q), o_gated=torch.empty_like(q),
                mse=torch.empty(B, N, device=dev), gamma=torch.empty(B, N, device=dev),
                reg_loss=torch.empty(B, N, device=dev))
    ws = torch.empty(max(256, swa.dual_branch_workspace(B, N, Hq, Hkv, D, W, torch.bfloat16)),
                     dtype=torch.uint8, device=dev)

    def step():
        swa.dual_branch(q, k, v, lg, nll, W, outs=outs, workspace=ws)

    step_ms, kern_ms = timer.run(step, steps, warmup, kernel_events=True)
    assert swa.get_device_error() == 0
    pairs_full = N * (N + 1) // 2
    flops = 4.0 * D * Hq * B * pairs_full
    return dict(step_ms=step_ms, kern_ms=kern_ms, flops=flops)


def backward_section(swa, timer, dev, steps, warmup, seed, workload):
    """Training backward (swiattn_prefill_backward): forward output and lse are
    computed once, untimed; a step is one backward call (schedule, dK/dV and dQ
    kernels).  Useful work: 10*d FLOP per visited (query, key) pair and query
    head, the five d-long products of the attention backward (recomputed
    scores, dP, dV, dK, dQ)."""
    if workload == "dual_8k":
        d = inp.dual_8k(seed=seed)
        gate_cpu = (d["logits"] > 0).to(torch.uint8)
    else:
        d = inp.prefill_32k(frac=0.13, seed=seed)
        gate_cpu = d["gate"]
    B, N, Hq, Hkv, D, W = d["B"], d["N"], d["Hq"], d["Hkv"], d["d"], d["W"]
    q, k, v = (d[n].to(dev) for n in ("q", "k", "v"))
    gate = gate_cpu.to(dev)
    do = inp.output_grad(d["q"].shape, torch.bfloat16, seed + 1).to(dev)
    o, lse = swa.prefill(q, k, v, gate, W, want_lse=True)
    outs = (torch.empty_like(q), torch.empty_like(k), torch.empty_like(v))
    ws = torch.empty(swa.prefill_backward_workspace(B, N, Hq, Hkv, D, W, torch.bfloat16),
                     dtype=torch.uint8, device=dev)

    def step():
        swa.prefill_backward(q, k, v, gate, o, lse, do, W, outs=outs, workspace=ws)

    step_ms, kern_ms = timer.run(step, steps, warmup, kernel_events=True)
    assert swa.get_device_error() == 0
    pairs = useful_pairs(gate_cpu.numpy(), W)
    return dict(step_ms=step_ms, kern_ms=kern_ms, flops=10.0 * D * Hq * pairs,
                routed_frac=float(gate_cpu.float().mean()))


def route_backward_section(swa, timer, dev, steps, warmup, seed):
    """Router backward on the dual-branch workload's shapes: 16384 tokens,
    hd = 16*128 attention outputs per token, d_model 2048 (HBM-bound: reads
    o_full, o_swa, dO and h, writes dh)."""
    T, HD, Dm = 2 * 8192, 16 * 128, 2048
    g = inp._gen(seed)
    of, os_, do = (inp.randn((T, HD), torch.bfloat16, g).to(dev) for _ in range(3))
    r = inp.router_inputs(T, Dm, torch.bfloat16, seed)
    h, w = r["h"].to(dev), r["w"].to(dev)
    logits = inp.logits_with_margin((T,), g).to(dev)
    gamma = torch.full((T,), 1e-3, device=dev)
    d_reg = torch.ones(T, device=dev)
    ws = torch.empty(swa.route_backward_workspace(T, Dm, torch.bfloat16), dtype=torch.uint8,
                     device=dev)

    def step():
        swa.route_backward(logits, of, os_, do, gamma, d_reg, h, w, workspace=ws)

    step_ms, kern_ms = timer.run(step, steps, warmup, kernel_events=True)
    nbytes = 3 * T * HD * 2 + 2 * T * Dm * 2 + T * 16 + Dm * 4
    return dict(step_ms=step_ms, kern_ms=kern_ms, bytes=nbytes)


# ------------------------------------------------------------ CPU oracle --
def oracle_sample(d, budget_s: float, seed: int = 0):
    """Time the fp64 oracle on a random sample of (row, head) outputs of the
    workload sized to about budget_s seconds; returns useful FLOP/s, cores,
    description."""
    import oracle
    N, H, D, W = d["N"], d["Hq"], d["d"], d["W"]
    gate = d["gate"].numpy()
    q64, k64, v64 = (d[n].to(torch.float64).numpy() for n in ("q", "k", "v"))
    rng = np.random.default_rng(seed)

    def run(nrows):
        sel = np.stack([np.zeros(nrows, np.int64), rng.integers(0, N, nrows),
                        rng.integers(0, H, nrows)], 1)
        i = sel[:, 1]
        n = np.where(gate[0, i] != 0, i + 1, np.minimum(i + 1, W))
        t0 = time.perf_counter()
        oracle.prefill_rows(q64, k64, v64, gate, W, 1.0 / math.sqrt(D), sel)
        return time.perf_counter() - t0, 4.0 * D * float(n.sum())

    t, f = run(64)
    per_row = max(t / 64, 1e-6)
    nrows = int(min(max(budget_s / per_row, 64), 200000))
    t, f = run(nrows)
    return dict(flops_per_s=f / t, seconds=t, rows=nrows, cores=oracle.num_threads())


def oracle_single_core_4k(budget_s: float = 3.0):
    """The oracle on one host core, on a sample of the single-layer 4K
    workload (gates from the oracle's own router): a per-core reference point
    beside the all-core baseline."""
    import oracle
    d = inp.prefill_4k(seed=0)
    _, gate = oracle.route(d["h"].to(torch.float64).numpy(), d["w"].to(torch.float64).numpy(),
                           d["bias"])
    dd = dict(d, gate=torch.from_numpy(np.ascontiguousarray(gate.reshape(1, -1))))
    prev = oracle.num_threads()
    oracle.set_num_threads(1)
    try:
        return oracle_sample(dd, budget_s)
    finally:
        oracle.set_num_threads(prev)


# ------------------------------------------------------------------ arms --
def run_reference(args, dist: Dist):
    if dist.rank != 0:
        return
    d = inp.prefill_32k(frac=0.13, seed=0)
    import oracle
    oracle.build()
    per_step = []
    flops = []
    cores = oracle.num_threads()
    for s in range(args.warmup + args.steps):
        r = oracle_sample(d, budget_s=args.ref_step_budget, seed=s)
        if s >= args.warmup:
            per_step.append(r["seconds"])
            flops.append(r["flops_per_s"] * r["seconds"])
    value = sum(flops) / sum(per_step) / 1e12
    line = {
        "impl": "reference", "metric": METRIC, "value": value, "unit": "TFLOP/s",
        "n_gpus": args.gpus, "steps": args.steps, "warmup": args.warmup,
        "ms_per_step": 1e3 * statistics.mean(per_step), "higher_is_better": True,
        "scaling": "weak", "vs_baseline": None, "dtype": "f64", "data": "synthetic",
        "config": {"workload": "long-context routed prefill, B=1 H=16 d=128 N=32768 W=1024, "
                               "gate runs at routed fraction 0.13", "routed_fraction": 0.13},
        "cpu_baseline": {"value": value, "unit": "TFLOP/s", "cores": cores, "kind": "oracle",
                         "sample": "each step: random (row, head) outputs of the workload, "
                                   f"about {args.ref_step_budget:g} s of fp64 oracle work"},
        "e2e": {"value": value, "unit": "TFLOP/s", "h2d_bytes_per_step": 0,
                "d2h_bytes_per_step": 0},
    }
    print(json.dumps(line), flush=True)


def run_ours(args, dist: Dist):
    if not torch.cuda.is_available():
        raise RuntimeError("bench.py needs a CUDA GPU")
    dev = torch.device("cuda", dist.local_rank)
    torch.cuda.set_device(dev)
    import sliding_window_attention_router_gb300 as swa
    swa._load()   # fails loudly if the library is missing
    peaks, peaks_src = load_peaks()
    timer = Timer(dev)
    gpu_index = int(os.environ.get("CUDA_VISIBLE_DEVICES", str(dist.local_rank)).split(",")[0]) \
        if os.environ.get("CUDA_VISIBLE_DEVICES", "").split(",")[0].isdigit() else dist.local_rank

    clocks = ClockSampler(gpu_index)
    dist.barrier()
    torch.cuda.synchronize()
    t_wall0 = time.perf_counter()
    main = prefill_section(swa, timer, dev, 0.13, args.steps, args.warmup, seed=dist.rank,
                           with_e2e=not args.no_e2e, N=args.n, hold_s=0.6)
    torch.cuda.synchronize()
    dist.barrier()
    wall = time.perf_counter() - t_wall0
    clk = clocks.stop(main["t_from"], main["t_to"])
    if clk is not None:
        clk["window"] = "timed headline steps plus 0.6 s of the same step under load"

    step_s = sum(main["step_ms"]) / 1e3
    value, slowest = aggregate(main["flops"] * args.steps, step_s, dist)
    e2e = None
    if "e2e_ms" in main:
        e2e_s = sum(main["e2e_ms"]) / 1e3
        serial_value, _ = aggregate(main["flops"] * len(main["e2e_ms"]), e2e_s, dist)
        e2e_value, _ = aggregate(main["flops"] * main["e2e_pipe_n"], main["e2e_pipe_ms"] / 1e3, dist)
        e2e = {"value": e2e_value / 1e12, "unit": "TFLOP/s",
               "h2d_bytes_per_step": main["h2d"], "d2h_bytes_per_step": main["d2h"],
               "steps": main["e2e_pipe_n"],
               "issue": "swiattn_prefill_host calls back to back, alternating two streams",
               "serial": {"value": serial_value / 1e12,
                          "issue": "one call per timed step, the stream idle between steps"}}
    kern_s = statistics.mean(main["kern_ms"]) / 1e3
    achieved = main["flops"] / kern_s / 1e12
    peak = float(peaks["bf16_tflops"])
    traffic = measured_traffic("prefill") if args.n == 32768 else None

    extra = {}
    if not args.headline_only:
        ks, kw = max(3, args.steps), max(3, args.warmup)
        easy = prefill_section(swa, timer, dev, 0.05, ks, kw, seed=dist.rank, with_e2e=False)
        extra["prefill_easy"] = {
            "tflops": easy["flops"] / (sum(easy["step_ms"]) / 1e3 / ks) / 1e12,
            "kernel_tflops": easy["flops"] / (statistics.mean(easy["kern_ms"]) / 1e3) / 1e12,
            "ms_per_step": statistics.mean(easy["step_ms"]),
            "realised_frac": easy["realised_frac"], "useful_tflop": easy["flops"] / 1e12}
        dec = decode_section(swa, timer, dev, ks, kw, seed=dist.rank,
                             sweep_routed=(0, 1, 2, 4, 8, 12, 16))
        dk = statistics.mean(dec["kern_ms"]) / 1e3
        ds = statistics.mean(dec["step_ms"]) / 1e3
        hbm = float(peaks["hbm_gbs"])
        decode_entry = {
            "gbs": round(dec["bytes"] / ds / 1e9, 1), "ms_per_step": round(ds * 1e3, 4),
            "n_routed": dec["n_routed"], "bytes_per_step": dec["bytes"],
            "roofline": {"bound": "hbm", "achieved": round(dec["bytes"] / dk / 1e9, 1),
                         "peak": hbm, "unit": "GB/s",
                         "frac": round(dec["bytes"] / dk / 1e9 / hbm, 4),
                         "traffic": measured_traffic("decode"),
                         "kernel": "decode_split2_kernel"},
            "workload": "decode bf16: 16 sequences x 32768 cached tokens, H=16, d=128, W=1024, "
                        "gate Bernoulli(0.13)",
            "sweep": {"columns": ["n_routed", "step GB/s", "kernel GB/s", "kernel frac of HBM"],
                      "rows": [[r["n_routed"], round(r["gbs"], 1), round(r["kernel_gbs"], 1),
                                round(r["kernel_gbs"] / hbm, 4)] for r in dec["sweep"]]}}
        da = decode_section(swa, timer, dev, ks, kw, seed=dist.rank, S=256)
        das = statistics.mean(da["step_ms"]) / 1e3
        extra["decode_anchored"] = {
            "gbs": da["bytes"] / das / 1e9, "ms_per_step": das * 1e3,
            "kernel_gbs": da["bytes"] / (statistics.mean(da["kern_ms"]) / 1e3) / 1e9,
            "workload": "decode bf16, 16 x 32768 cached tokens, window queries also read the "
                        "first 256 entries"}
        dp = decode_paged_section(swa, timer, dev, ks, kw, seed=dist.rank)
        dpk = statistics.mean(dp["kern_ms"]) / 1e3
        dps = statistics.mean(dp["step_ms"]) / 1e3
        extra["decode_paged"] = {
            "gbs": dp["bytes"] / dps / 1e9, "ms_per_step": dps * 1e3, "n_routed": dp["n_routed"],
            "kernel_gbs": dp["bytes"] / dpk / 1e9, "kernel_frac_of_hbm": dp["bytes"] / dpk / 1e9 / hbm,
            "workload": "decode bf16 on a paged cache: 16 sequences x 32768 tokens in 64-token "
                        "pages of a shuffled pool, H=16, d=128, W=1024, gate Bernoulli(0.13)"}
        an = anchored_prefill_section(swa, timer, dev, ks, kw, seed=dist.rank)
        ans = statistics.mean(an["step_ms"]) / 1e3
        extra["prefill_anchored"] = {
            "tflops": an["flops"] / ans / 1e12, "ms_per_step": ans * 1e3,
            "kernel_tflops": an["flops"] / (statistics.mean(an["kern_ms"]) / 1e3) / 1e12,
            "useful_tflop": an["flops"] / 1e12,
            "workload": "long-context routed prefill (N=32768, f=0.13) with 256 global anchors "
                        "per window row"}
        sh = static_hybrid_section(swa, timer, dev, ks, kw, seed=dist.rank)
        shs = statistics.mean(sh["step_ms"]) / 1e3
        extra["static_hybrid_3to1"] = {
            "ms_per_layer": shs * 1e3 / 4, "routed_ms_per_layer": 1e3 * slowest / args.steps,
            "tflops": sh["flops"] / shs / 1e12,
            "workload": "comparator: three window layers and one full layer (W=1024) per group "
                        "of four, N=32768, H=16, d=128; per-layer time beside one routed layer "
                        "at routed fraction 0.13"}
        rt = route_section(swa, timer, dev, ks, kw, seed=dist.rank)
        rs = statistics.mean(rt["step_ms"]) / 1e3
        rk = statistics.mean(rt["kern_ms"]) / 1e3
        extra["route"] = {"gbs": rt["bytes"] / rs / 1e9, "ms_per_step": rs * 1e3,
                          "roofline": {"bound": "hbm", "achieved": rt["bytes"] / rk / 1e9,
                                       "peak": hbm, "unit": "GB/s",
                                       "frac": rt["bytes"] / rk / 1e9 / hbm,
                                       "traffic": measured_traffic("route"),
                                       "kernel": "route_kernel"},
                          "workload": "router GEMV, 32768 tokens x d_model 2048, bf16"}
        l4 = layer_4k_section(swa, timer, dev, ks, kw, seed=dist.rank)
        l4s = statistics.mean(l4["step_ms"]) / 1e3
        extra["layer_4k"] = {"tflops": l4["flops"] / l4s / 1e12, "ms_per_step": l4s * 1e3,
                             "separate_calls_ms_per_step": statistics.mean(l4["separate_ms"]),
                             "routed_frac": l4["routed_frac"],
                             "workload": "single-layer prefill bf16: router GEMV over h [4096, 2048] "
                                         "then routed prefill B=1 H=16 d=128 N=4096 W=1024 on its "
                                         "gates, as one fused call (route_prefill)"}
        du = dual_section(swa, timer, dev, ks, kw, seed=dist.rank)
        dm = statistics.mean(du["step_ms"]) / 1e3
        dk_t = du["flops"] / (statistics.mean(du["kern_ms"]) / 1e3) / 1e12
        extra["dual"] = {"tflops": du["flops"] / dm / 1e12, "ms_per_step": dm * 1e3,
                         "kernel_tflops": dk_t,
                         "roofline": {"bound": "tensor", "achieved": dk_t, "peak": peak,
                                      "unit": "TFLOP/s", "frac": dk_t / peak,
                                      "traffic": measured_traffic("dual"), "kernel": "dual_kernel"},
                         "workload": "dual-branch forward bf16, B=2 Hq=16 Hkv=4 d=128 N=8192 W=1024"}
        for wl, desc in (("dual_8k", "training backward bf16 on the dual-branch workload: B=2 "
                                     "Hq=16 Hkv=4 d=128 N=8192 W=1024, gates = logits > 0"),
                         ("prefill_32k", "training backward bf16 on the long-context prefill "
                                         "workload: B=1 H=16 d=128 N=32768 W=1024, f=0.13")):
            bw = backward_section(swa, timer, dev, ks, kw, dist.rank, wl)
            bms = statistics.mean(bw["step_ms"]) / 1e3
            bk = statistics.mean(bw["kern_ms"]) / 1e3
            extra["backward_" + wl] = {
                "tflops": bw["flops"] / bms / 1e12, "ms_per_step": bms * 1e3,
                "routed_frac": bw["routed_frac"], "useful_tflop": bw["flops"] / 1e12,
                "roofline": {"bound": "tensor", "achieved": bw["flops"] / bk / 1e12,
                             "peak": peak, "unit": "TFLOP/s",
                             "frac": bw["flops"] / bk / 1e12 / peak,
                             "traffic": measured_traffic("backward") if wl == "dual_8k" else None,
                             "kernel": "dkdv_kernel + dq_kernel"},
                "workload": desc}
        rb = route_backward_section(swa, timer, dev, ks, kw, dist.rank)
        rbs = statistics.mean(rb["step_ms"]) / 1e3
        rbk = statistics.mean(rb["kern_ms"]) / 1e3
        extra["route_backward"] = {
            "gbs": rb["bytes"] / rbs / 1e9, "ms_per_step": rbs * 1e3,
            "roofline": {"bound": "hbm", "achieved": rb["bytes"] / rbk / 1e9, "peak": hbm,
                         "unit": "GB/s", "frac": rb["bytes"] / rbk / 1e9 / hbm,
                         "traffic": measured_traffic("route_backward"),
                         "kernel": "route_bwd_logit_kernel + route_bwd_dh_kernel + "
                                   "route_bwd_reduce_kernel"},
            "workload": "router backward bf16: 16384 tokens, 2048 outputs per token, d_model 2048"}
        extra["decode"] = decode_entry

    cpu = None
    if dist.rank == 0 and dist.world == 1 and not args.no_cpu_baseline:
        r = oracle_sample(main["d"], budget_s=args.cpu_budget)
        cpu = {"value": r["flops_per_s"] / 1e12, "unit": "TFLOP/s", "cores": r["cores"],
               "kind": "oracle",
               "sample": f"{r['rows']} random (row, head) outputs of the N=32768 workload, "
                         f"{r['seconds']:.1f} s of fp64 oracle work on {r['cores']} threads"}
        r1 = oracle_single_core_4k()
        cpu["single_core_prefill_4k"] = {
            "value": r1["flops_per_s"] / 1e12, "unit": "TFLOP/s", "cores": r1["cores"],
            "sample": f"{r1['rows']} random (row, head) outputs of the single-layer N=4096 "
                      f"workload, {r1['seconds']:.1f} s on one core"}

    if dist.rank == 0:
        d = main["d"]
        line = {
            "metric": METRIC, "value": value / 1e12, "unit": "TFLOP/s", "n_gpus": dist.world,
            "steps": args.steps, "warmup": args.warmup,
            "ms_per_step": 1e3 * slowest / args.steps, "higher_is_better": True,
            "scaling": "weak", "vs_baseline": None, "dtype": "bf16", "data": "synthetic",
            "config": {"workload": f"long-context routed prefill bf16: B=1 H=16 d=128 N={d['N']} "
                                   "W=1024, gates in runs (mean routed run 64) at routed "
                                   "fraction 0.13",
                       "B": d["B"], "N": d["N"], "H": d["Hq"], "d": d["d"], "W": d["W"],
                       "realised_routed_fraction": main["realised_frac"],
                       "useful_tflop_per_step": main["flops"] / 1e12,
                       "l2": "flushed before every timed step (256 MiB written, then read back)",
                       "parallelism": f"replicas x{dist.world}, one sequence per GPU"},
            "roofline": {"bound": "tensor", "achieved": achieved, "peak": peak,
                         "unit": "TFLOP/s", "frac": achieved / peak,
                         "traffic": traffic, "kernel": "prefill_kernel",
                         "peak_source": f"{peaks_src} bf16 dense (burst)"},
            "cpu_baseline": cpu,
            "e2e": e2e,
            "gpu_launches": 2 * args.steps,   # plan_kernel + prefill_kernel per step
            "clocks": clk,
            "wall_s_headline": wall,
        }
        line.update(extra)
        print(json.dumps(line), flush=True)


def run_backward_only(args):
    """One backward workload alone (a profiling aid, not the bench line)."""
    dev = torch.device("cuda", 0)
    torch.cuda.set_device(dev)
    import sliding_window_attention_router_gb300 as swa
    swa._load()
    bw = backward_section(swa, Timer(dev), dev, args.steps, args.warmup, 0, args.only_backward)
    bms = statistics.mean(bw["step_ms"]) / 1e3
    bk = statistics.mean(bw["kern_ms"]) / 1e3
    print(json.dumps({"workload": args.only_backward, "tflops": bw["flops"] / bms / 1e12,
                      "kernel_tflops": bw["flops"] / bk / 1e12, "ms_per_step": bms * 1e3,
                      "useful_tflop": bw["flops"] / 1e12}), flush=True)


def run_section_only(args):
    """The decode (16 x 32K), dual-branch (8K), router or router-backward
    section alone (a profiling aid, not the bench line)."""
    dev = torch.device("cuda", 0)
    torch.cuda.set_device(dev)
    import sliding_window_attention_router_gb300 as swa
    swa._load()
    timer = Timer(dev)
    if args.only == "decode":
        r = decode_section(swa, timer, dev, args.steps, args.warmup, 0)
        k = statistics.mean(r["kern_ms"]) / 1e3
        print(json.dumps({"section": "decode", "kernel_gbs": r["bytes"] / k / 1e9,
                          "bytes_per_step": r["bytes"], "n_routed": r["n_routed"]}), flush=True)
    elif args.only in ("route", "route_backward"):
        fn = route_section if args.only == "route" else route_backward_section
        r = fn(swa, timer, dev, args.steps, args.warmup, 0)
        k = statistics.mean(r["kern_ms"]) / 1e3
        print(json.dumps({"section": args.only, "kernel_gbs": r["bytes"] / k / 1e9,
                          "bytes_per_step": r["bytes"]}), flush=True)
    else:
        r = dual_section(swa, timer, dev, args.steps, args.warmup, 0)
        k = statistics.mean(r["kern_ms"]) / 1e3
        print(json.dumps({"section": "dual", "kernel_tflops": r["flops"] / k / 1e12}), flush=True)


def main():
    ap = argparse.ArgumentParser()
    ap.add_argument("--gpus", type=int, default=1)
    ap.add_argument("--steps", type=int, default=20)
    ap.add_argument("--warmup", type=int, default=3)
    ap.add_argument("--impl", choices=["ours", "reference"], default="ours")
    ap.add_argument("--headline-only", action="store_true")
    ap.add_argument("--no-cpu-baseline", action="store_true")
    ap.add_argument("--cpu-budget", type=float, default=15.0)
    ap.add_argument("--n", type=int, default=32768,
                    help="sequence length of the headline workload (profiling runs only)")
    ap.add_argument("--no-e2e", action="store_true")
    ap.add_argument("--ref-step-budget", type=float, default=3.0,
                    help="seconds of oracle work per step of the reference arm")
    ap.add_argument("--only-backward", choices=["dual_8k", "prefill_32k"], default=None,
                    help="profiling runs only: time just the training backward on one workload")
    ap.add_argument("--only", choices=["decode", "dual", "route", "route_backward"], default=None,
                    help="profiling runs only: time just one section (decode, dual branch, "
                         "router, router backward)")
    args = ap.parse_args()
    if args.warmup < 3:
        args.warmup = 3
    dist = Dist()
    try:
        if args.impl == "reference":
            run_reference(args, dist)
        elif args.only_backward:
            run_backward_only(args)
        elif args.only:
            run_section_only(args)
        else:
            run_ours(args, dist)
    finally:
        dist.close()


if __name__ == "__main__":
    main()
