"""Benchmark of the MXFP8 x MXFP4 top-16 MoE decode layer on GB300.

    python bench.py [--gpus N] [--steps K] [--warmup W] [--impl ours|reference]
                    [--config tp8_b1] [--no-extra]

A step is one moe_run call over one batch. A call of one or two tokens is
one launch of the small-batch experts kernel (MXFP8 quantize, grouping, FC1,
FC2, BF16 rows); any other call is the prep grid (quantize + grouping) and
the persistent grid experts kernel. Metric: microseconds per call and
touched-weight HBM GB/s. The main workload is the TP8 shard at B = 1
(E = 384, H = 3584, I = 384, uniform distinct top-16 ids); the TP16 B = 8,
TP8 B = 64 (Zipf 1.1) and TP8 B = 256 (Zipf 1.1, 1% x50 rows) workloads are
reported under "configs". Inputs are synthetic and seeded (workload/).

L2: every call reads a different replica of the weights (R replicas, each a
separate moe_prepare of the same weights) with (R - 1) x touched bytes >= 3 x
L2, so no call finds its weights in the 126 MiB L2. The K timed calls are
replayed from one CUDA graph (K <= 256; beyond, graphs of whole rounds over
the replicas), queued behind a spin kernel so that the host's launch of the
graph stays out of the timed region, bracketed by a barrier and a device
synchronize, and timed with CUDA events.

Roofline: the experts kernel's own time per call (kernel_us). When a call is
one launch, consecutive launches overlap (programmatic dependent launch), so
its time per call is the timed per-call time; its launch-clock span (first
CTA start to last CTA end, moe_debug_kernel_span) includes waiting for the
previous launch and is kept as kernel_span_us. Otherwise kernel_us is that
span for the experts kernel inside the step. kernel_us_isolated: CUDA events
around moe_experts alone (the grid kernel, after separate moe_quantize and
moe_group launches).

Parity: the CPU-baseline leg runs the float64 oracle on the main workload;
the same run compares one GPU call against it (activation plan and unit
table bit for bit, output relative L2 and worst |err| / rms(row), hidden
requant code and scale flips) and reports the result under "parity".

e2e: moe_run_host with pinned host buffers per step. On a GPU with native
atomics on host memory (Grace's coherent link) the kernels read x and ids from
those buffers and write out into them in place (each call one launch of a
graph the handle captured on its first such call, made before timing);
elsewhere the call copies them. Either way the input and output bytes cross
between host and device inside the timed region, and a synchronize ends
every step.

--impl reference times the float64 CPU oracle (oracle/) on the host cores on
the same workload: each step is one whole call.
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
import threading
import time

import numpy as np

ROOT = os.path.dirname(os.path.abspath(__file__))
sys.path.insert(0, ROOT)

import workload  # noqa: E402

MAIN_CONFIG = "tp8_b1"
EXTRA_CONFIGS = ["tp16_b8", "tp8_b64", "tp8_b256"]
L2_FALLBACK_BYTES = 126 * 2 ** 20
PROFILE_SUMMARY = os.path.join(ROOT, "profiles", "small_kernel_tp8_b1.md")
KERNEL_SOURCES = ["experts.cu", "small.cu", "pipeline.cuh", "ptx.cuh", "common.cuh", "kernels.h"]


def parse():
    p = argparse.ArgumentParser()
    p.add_argument("--gpus", type=int, default=1)
    p.add_argument("--steps", type=int, default=2000)
    p.add_argument("--warmup", type=int, default=20)
    p.add_argument("--impl", choices=["ours", "reference"], default="ours")
    p.add_argument("--config", default=MAIN_CONFIG)
    p.add_argument("--no-extra", action="store_true", help="skip the other workloads")
    p.add_argument("--profile-case", action="store_true",
                   help="no timing: prepare one layer and run --steps calls of --config "
                        "(a small case for ncu captures)")
    return p.parse_args()


def dist_env():
    rank = int(os.environ.get("RANK", "0"))
    world = int(os.environ.get("WORLD_SIZE", "1"))
    local = int(os.environ.get("LOCAL_RANK", "0"))
    return rank, world, local


def max_over_ranks(value, world, device):
    """The largest of one float per rank (every rank gets it); with one rank,
    the value itself. Each rank times its own replica, so the job's time per
    call is the slowest rank's."""
    if world <= 1:
        return value
    import torch

    t = torch.tensor([value], device=device, dtype=torch.float64)
    torch.distributed.all_reduce(t, op=torch.distributed.ReduceOp.MAX)
    return float(t.item())


def describe(cfg):
    return (f"{cfg.name}: E={cfg.experts} H={cfg.hidden} I={cfg.inter} B={cfg.batch} top-16 "
            f"{cfg.ids} ids" + (f", {cfg.outlier_fraction:.0%} rows x50" if cfg.outlier_fraction else ""))


def measured_peaks():
    path = os.path.join(ROOT, "MEASURED_PEAKS.json")
    try:
        with open(path) as f:
            peaks = json.load(f)
        return float(peaks["hbm_gbs"]), "measured"
    except (OSError, KeyError, ValueError):
        return 6800.0, "fallback"


def code_only(text):
    """C++ source without its comments and with whitespace runs collapsed, so
    that editing a comment does not count as changing the kernel."""
    text = re.sub(r"/\*.*?\*/", " ", text, flags=re.S)
    text = re.sub(r"//[^\n]*", " ", text)
    return " ".join(text.split())


def kernel_hash(read=None):
    """sha256[:16] of the experts kernel's code (comments and whitespace
    ignored), as recorded in the ncu summaries."""
    h = hashlib.sha256()
    for name in KERNEL_SOURCES:
        if read is None:
            with open(os.path.join(ROOT, "mxfp4_weight_mxfp8_gb300", "csrc", name), encoding="utf-8") as f:
                text = f.read()
        else:
            text = read(name)
        h.update(code_only(text).encode())
    return h.hexdigest()[:16]


def profiled_traffic():
    """DRAM bytes per experts-kernel launch from the committed ncu summary,
    if it was taken on the current kernel source."""
    try:
        text = open(PROFILE_SUMMARY).read()
    except OSError:
        return None
    fields = dict(line.split(": ", 1) for line in text.splitlines() if line.startswith("- ") and ": " in line)
    fields = {k[2:].strip(): v.strip() for k, v in fields.items()}
    if fields.get("kernel source sha256[:16]") != kernel_hash():
        return None
    try:
        return float(fields["dram bytes per launch"].split()[0])
    except (KeyError, ValueError):
        return None


class ClockSampler:
    """nvidia-smi clocks and throttle reasons, every 50 ms, in a background process."""

    QUERY = ("index,clocks.sm,clocks.max.sm,power.draw,clocks_event_reasons.active,"
             "clocks_event_reasons.hw_slowdown,clocks_event_reasons.hw_thermal_slowdown,"
             "clocks_event_reasons.sw_thermal_slowdown,clocks_event_reasons.sw_power_cap")

    def __init__(self, index):
        self.index = index
        self.lines = []
        self.proc = None
        self.thread = None

    def start(self):
        try:
            self.proc = subprocess.Popen(
                ["nvidia-smi", f"--id={self.index}", f"--query-gpu={self.QUERY}",
                 "--format=csv,noheader,nounits", "-lms", "50"],
                stdout=subprocess.PIPE, stderr=subprocess.DEVNULL, text=True)
        except OSError:
            self.proc = None
            return
        self.thread = threading.Thread(target=self._read, daemon=True)
        self.thread.start()

    def _read(self):
        for line in self.proc.stdout:
            self.lines.append((time.monotonic(), line.strip()))

    def mark(self):
        return time.monotonic()

    def stop(self):
        if self.proc is not None:
            self.proc.terminate()
            try:
                self.proc.wait(timeout=5)
            except subprocess.TimeoutExpired:
                self.proc.kill()
        if self.thread is not None:
            self.thread.join(timeout=5)

    def summary(self, t0, t1):
        rows = [l for t, l in self.lines if t0 <= t <= t1] or [l for t, l in self.lines]
        mhz, max_mhz, reasons = [], None, set()
        names = ["hw_slowdown", "hw_thermal_slowdown", "sw_thermal_slowdown", "sw_power_cap"]
        for line in rows:
            parts = [x.strip() for x in line.split(",")]
            if len(parts) < 9:
                continue
            try:
                mhz.append(float(parts[1]))
                max_mhz = float(parts[2])
            except ValueError:
                continue
            for name, flag in zip(names, parts[5:9]):
                if flag.lower() == "active":
                    reasons.add(name)
        return {"sm_mhz": statistics.median(mhz) if mhz else None, "sm_max_mhz": max_mhz,
                "reasons": sorted(reasons), "samples": len(mhz)}


def replicas_for(touched_bytes, l2_bytes, per_replica_bytes, free_bytes):
    want = max(2, math.ceil(3 * l2_bytes / max(touched_bytes, 1)) + 1)
    fit = max(2, int(0.5 * free_bytes // max(per_replica_bytes, 1)))
    return min(want, fit)


def oracle_call_seconds(weights, x, ids, repeats):
    import oracle

    times = []
    for _ in range(repeats):
        t = time.perf_counter()
        xq, xs = oracle.quantize_x(x)
        oracle.pairs_forward(weights, xq, xs, ids)
        times.append(time.perf_counter() - t)
    return times


def cpu_baseline(cfg, weights, x, ids, budget_s=12.0):
    """The oracle timed on the host cores, and its result of the same call:
    (baseline dict, dict(xq, xs, units, pairs result with hidden codes))."""
    import oracle

    first = oracle_call_seconds(weights, x, ids, 1)[0]
    threads = oracle.default_threads()
    repeats = max(1, min(50, int(budget_s / max(first * threads, 1e-3))))
    times = oracle_call_seconds(weights, x, ids, repeats)
    per_call = statistics.median(times)
    xq, xs = oracle.quantize_x(x)
    ref = {"xq": xq, "xs": xs, "units": oracle.group(ids, cfg.experts),
           "pairs": oracle.pairs_forward(weights, xq, xs, ids, want_hidden=True)}
    return ({"value": per_call * 1e6, "unit": "us/call", "cores": threads, "kind": "oracle",
             "sample": f"{repeats} whole {cfg.name} calls (all {ids.size} pairs), median; "
                       f"float64 C oracle, OpenMP over pairs"}, ref)


def parity_report(arm, ref):
    """One GPU call of the arm's workload against the oracle's result."""
    moe, torch, cfg = arm.moe, arm.torch, arm.cfg
    B, H, I = cfg.batch, cfg.hidden, cfg.inter
    layer = arm.layers[0]
    out = torch.empty((B, 16, H), dtype=torch.bfloat16, device=arm.device)
    moe.moe_run(layer.handle, arm.x, arm.ids, out, B)
    status = moe.moe_sync_status(layer.handle)
    codes = np.zeros((B, H), np.uint8)
    scales = np.zeros((B, H // 32), np.uint8)
    moe.moe_copy_plan(layer.handle, codes, scales, B)
    cap = B * 16 + 2 * B
    count = np.zeros(1, np.int32)
    ue = np.zeros(cap, np.int32)
    ur = np.zeros(cap * 8, np.int16)
    moe.moe_copy_units(layer.handle, count, ue, ur, cap)
    n = int(count[0])
    hq = np.zeros((n, 8, I), np.uint8)
    hs = np.zeros((n, 8, I // 32), np.uint8)
    moe.moe_copy_hidden(layer.handle, hq, hs, n)
    bits = out.view(torch.int16).cpu().numpy().view(np.uint16).reshape(B * 16, H)
    f = lambda b: (b.astype(np.uint32) << 16).view(np.float32).astype(np.float64)
    got, want = f(bits), f(ref["pairs"]["out"])
    rel = float(np.linalg.norm(got - want) / max(np.linalg.norm(want), 1e-300))
    rms = np.sqrt(np.mean(want ** 2, axis=1, keepdims=True))
    worst = float(np.max(np.abs(got - want) / np.maximum(rms, 1e-300)))
    ref_ue, ref_ur = ref["units"]
    units_exact = n == len(ref_ue) and np.array_equal(ue[:n], ref_ue) and np.array_equal(
        ur[: n * 8].reshape(n, 8), ref_ur)
    code_flips = scale_flips = 0
    rows = ur[: n * 8].reshape(n, 8)
    for u in range(n):
        for r in range(8):
            p = int(rows[u, r])
            if p < 0:
                continue
            code_flips += int(np.count_nonzero(hq[u, r] != ref["pairs"]["hq"][p]))
            scale_flips += int(np.count_nonzero(hs[u, r] != ref["pairs"]["hs"][p]))
    return {
        "workload": describe(cfg), "status": int(status),
        "plan_bit_exact": bool(np.array_equal(codes, ref["xq"]) and np.array_equal(scales, ref["xs"])),
        "units_bit_exact": bool(units_exact),
        "rel_l2": rel, "worst_err_over_rms_row": worst,
        "hidden_code_flips": code_flips, "hidden_scale_flips": scale_flips,
        "hidden_codes": int(B * 16 * I),
        "bars": "plan and units bit-exact; rel_l2 <= 1e-2; |err| <= 3e-2 rms(row); flips reported",
        "pass": bool(status == 0 and rel <= 1e-2 and worst <= 3e-2 and units_exact),
    }


class OurArm:
    def __init__(self, cfg, device):
        import torch

        import mxfp4_weight_mxfp8_gb300 as moe

        self.moe, self.torch, self.cfg, self.device = moe, torch, cfg, device
        self.weights_np, self.x_np, self.ids_np = None, None, None

    def setup(self, weights_np, x_np, ids_np, l2_bytes):
        torch, moe, cfg = self.torch, self.moe, self.cfg
        self.weights_np, self.x_np, self.ids_np = weights_np, x_np, ids_np
        dev_w = tuple(torch.from_numpy(w).to(self.device) for w in weights_np)
        touched = len(workload.touched_experts(ids_np)) * workload.expert_bytes(cfg.hidden, cfg.inter)
        self.touched = touched
        per_replica = sum(w.numel() for w in dev_w) * 17408 // 16384 + 64 * 2 ** 20
        free, _ = torch.cuda.mem_get_info(self.device)
        self.R = replicas_for(touched, l2_bytes, per_replica, free)
        self.layers = [moe.MoeLayer(dev_w) for _ in range(self.R)]
        del dev_w
        B = cfg.batch
        self.x = torch.from_numpy(x_np.view(np.int16)).to(self.device).view(torch.bfloat16)
        self.ids = torch.from_numpy(ids_np).to(self.device)
        self.out = torch.empty((B, 16, cfg.hidden), dtype=torch.bfloat16, device=self.device)
        self.io_bytes = {"x": B * cfg.hidden * 2, "ids": B * 16 * 4, "out": B * 16 * cfg.hidden * 2}
        # Routing weights for the combined call: positive, summing to one per token.
        rw = np.random.default_rng(5).random((B, 16)).astype(np.float32) + 0.1
        self.rw = torch.from_numpy(rw / rw.sum(axis=1, keepdims=True)).to(self.device)
        self.out_combined = torch.empty((B, cfg.hidden), dtype=torch.bfloat16, device=self.device)
        self.combined = False

    def call(self, i):
        layer = self.layers[i % self.R]
        if self.combined:
            self.moe.moe_run_combined(layer.handle, self.x, self.ids, self.rw, self.out_combined,
                                      self.cfg.batch)
        else:
            self.moe.moe_run(layer.handle, self.x, self.ids, self.out, self.cfg.batch)

    def check_status(self):
        for layer in self.layers:
            status = self.moe.moe_sync_status(layer.handle)
            if status != self.moe.MOE_OK:
                raise RuntimeError(f"device status {status}: {self.moe.moe_error_string(status)}")

    def kernel_span_us(self, replays, calls_per_graph):
        """In-step span of the experts kernel (us, mean over samples) and the
        per-call time (ms) of `replays` replays of a graph of
        `calls_per_graph` back-to-back calls captured with the launch clock on.
        After each replay every handle holds the span of its last launch in
        it; the launch that opens a replay (after the host's synchronize) is
        left out."""
        moe, torch = self.moe, self.torch
        for layer in self.layers:
            moe.moe_debug_kernel_span(layer.handle, 1)
        g = self.graph(calls_per_graph)
        g.replay()
        torch.cuda.synchronize()
        for layer in self.layers:
            moe.moe_read_kernel_span(layer.handle)
        spans, total_ms = [], 0.0
        for _ in range(replays):
            total_ms += self.time_graphs([(g, 1)], calls_per_graph) * calls_per_graph
            for i, layer in enumerate(self.layers):
                if i == 0 and calls_per_graph == self.R:
                    moe.moe_read_kernel_span(layer.handle)  # the replay's first launch
                    continue
                spans.append(moe.moe_read_kernel_span(layer.handle) / 1e3)
        for layer in self.layers:
            moe.moe_debug_kernel_span(layer.handle, 0)
        return statistics.mean(spans), total_ms / (replays * calls_per_graph), len(spans)

    def graph(self, calls):
        torch = self.torch
        g = torch.cuda.CUDAGraph()
        stream = torch.cuda.Stream(device=self.device)
        stream.wait_stream(torch.cuda.current_stream())
        with torch.cuda.stream(stream):
            self.call(0)  # the capture stream's first use outside capture
        torch.cuda.current_stream().wait_stream(stream)
        torch.cuda.synchronize()
        with torch.cuda.graph(g, stream=stream):
            for i in range(calls):
                self.call(i)
        torch.cuda.synchronize()
        return g

    def time_graphs(self, plan, calls):
        """Replay [(graph, times), ...] between two CUDA events; ms per call.
        A 100 us spin kernel goes first, so the start event and the graph
        launches are queued on a busy GPU: the timed region holds the calls'
        device work, not the host's launch of the first graph."""
        torch = self.torch
        start, end = torch.cuda.Event(enable_timing=True), torch.cuda.Event(enable_timing=True)
        torch.cuda.synchronize()
        torch.cuda._sleep(200_000)
        start.record()
        for g, times in plan:
            for _ in range(times):
                g.replay()
        end.record()
        torch.cuda.synchronize()
        return start.elapsed_time(end) / calls

    def launches_per_call(self):
        """Kernels one moe_run of this workload launches: the small-batch
        kernel alone, or the prep grid and an experts kernel."""
        path = self.moe.moe_kernel_path(self.layers[0].handle, self.cfg.batch)
        return 1 if path == self.moe.PATH_SMALL else 2

    def kernel_label(self):
        handle, B = self.layers[0].handle, self.cfg.batch
        path = self.moe.moe_kernel_path(handle, B)
        if path == self.moe.PATH_SMALL:
            return ("small_kernel (the whole call in one launch, two CTAs per SM, one of each of "
                    "two consecutive calls; one or two tokens: packed x and hidden images and a "
                    "3-slot weight ring: MXFP8 quantize and unit table in the kernel; FC1 segments "
                    "claimed from a counter, their sums gathered by every FC2 CTA; tcgen05 "
                    "block-scaled MMA)")
        if path == self.moe.PATH_CLUSTER:
            C = self.moe.moe_cluster_size(handle, B)
            return (f"cluster_kernel (experts kernel on thread-block clusters of {C} CTAs, "
                    "one per unit; tcgen05 block-scaled MMA)")
        rows = 16 if B > 8 else 8
        return (f"experts_kernel<{rows}> (persistent, {rows}-row units, tcgen05 block-scaled MMA "
                f"N = {rows}, two scale-copy warps)")

    def experts_kernel_ms(self, calls):
        """Mean device time of the experts kernel alone: moe_quantize and
        moe_group run first; CUDA events bracket only moe_experts. Every call is
        queued behind a spin kernel so the host enqueue never starves the GPU."""
        torch, moe, B = self.torch, self.moe, self.cfg.batch
        pairs = [(torch.cuda.Event(enable_timing=True), torch.cuda.Event(enable_timing=True))
                 for _ in range(calls)]
        torch.cuda.synchronize()
        torch.cuda._sleep(int(2e9 * max(0.02, calls * 40e-6)))
        for i in range(calls):
            layer = self.layers[i % self.R]
            moe.moe_quantize(layer.handle, self.x, B)
            moe.moe_group(layer.handle, self.ids, B)
            pairs[i][0].record()
            moe.moe_experts(layer.handle, self.out, B)
            pairs[i][1].record()
        torch.cuda.synchronize()
        return statistics.mean(a.elapsed_time(b) for a, b in pairs)

    def e2e_us(self, steps):
        torch, moe, B, H = self.torch, self.moe, self.cfg.batch, self.cfg.hidden
        xh = torch.from_numpy(self.x_np.view(np.int16)).pin_memory()
        idsh = torch.from_numpy(self.ids_np).pin_memory()
        outh = torch.empty((B, 16, H), dtype=torch.int16).pin_memory()
        # One untimed call per layer first: each handle captures its replay
        # graph on its first in-place call.
        for i in range(max(3, self.R)):
            moe.moe_run_host(self.layers[i % self.R].handle, xh, idsh, outh, B)
        torch.cuda.synchronize()
        t = time.perf_counter()
        for i in range(steps):
            rc = moe.moe_run_host(self.layers[i % self.R].handle, xh, idsh, outh, B)
        elapsed = time.perf_counter() - t
        return elapsed / steps * 1e6

    def close(self):
        for layer in self.layers:
            layer.close()
        self.layers = []


def run_ours(args, rank, world, local):
    import torch

    device = torch.device("cuda", local)
    torch.cuda.set_device(device)
    if world > 1:
        import torch.distributed as dist

        dist.init_process_group("nccl", device_id=device)
    props = torch.cuda.get_device_properties(device)
    l2_bytes = getattr(props, "L2_cache_size", L2_FALLBACK_BYTES) or L2_FALLBACK_BYTES
    peak, peak_kind = measured_peaks()

    cfg = workload.CONFIGS[args.config]
    weight_cache = {}

    def inputs(c):
        shape = (c.experts, c.hidden, c.inter)
        if shape not in weight_cache:
            weight_cache[shape] = workload.make_weights(*shape)
        x = workload.make_x(c.batch, c.hidden, outlier_fraction=c.outlier_fraction)
        ids = workload.make_ids(c.batch, c.experts, dist=c.ids, s=c.zipf_s)
        return weight_cache[shape], x, ids

    weights, x, ids = inputs(cfg)
    arm = OurArm(cfg, device)
    arm.setup(weights, x, ids, l2_bytes)
    for i in range(max(3, args.warmup)):
        arm.call(i)
    arm.check_status()

    # Exactly K timed calls. Up to 256: one graph of the K calls (rotating
    # over the R replicas), replayed once. Beyond: a graph of c calls (a
    # multiple of R) replayed K // c times, then a graph of the K % c rest.
    steps = max(1, args.steps)
    if steps <= 256:
        calls_per_graph = steps
    else:
        calls_per_graph = max(arm.R, 256 // arm.R * arm.R)
    replays = steps // calls_per_graph
    g = arm.graph(calls_per_graph)
    tail = arm.graph(steps - replays * calls_per_graph) if steps % calls_per_graph else None
    sampler = ClockSampler(local)
    sampler.start()
    t_warm = sampler.mark()
    warm_end = time.monotonic() + 0.5
    while time.monotonic() < warm_end:  # steady clocks before the timed region
        g.replay()
    torch.cuda.synchronize()
    if world > 1:
        torch.distributed.barrier()
    torch.cuda.synchronize()
    t0 = sampler.mark()
    ms_per_call = arm.time_graphs([(g, replays)] + ([(tail, 1)] if tail else []), steps)
    t1 = sampler.mark()
    if world > 1:
        torch.distributed.barrier()
    sampler.stop()
    arm.check_status()
    clocks = sampler.summary(t_warm, t1)
    ms_per_call = max_over_ranks(ms_per_call, world, device)

    # The launch clock pass: a graph of whole rounds over the R replicas.
    span_calls = max(arm.R, min(steps, 256) // arm.R * arm.R)
    span_us, span_pass_ms, span_samples = arm.kernel_span_us(max(4, min(40, replays * 4)),
                                                              span_calls)
    arm.check_status()
    kernel_ms = arm.experts_kernel_ms(min(200, max(20, args.steps // 10)))
    arm.check_status()
    e2e_us = arm.e2e_us(max(200, min(1000, args.steps)))
    arm.check_status()

    us_per_call = ms_per_call * 1e3
    # Replicas on every rank: the job completes `world` calls per slowest
    # rank's call time, so the job's time per call is that over `world`.
    aggregate_us = us_per_call / world
    gbs = arm.touched / (us_per_call * 1e-6) / 1e9
    single_launch = arm.launches_per_call() == 1
    # A call that is one kernel launch: consecutive launches overlap
    # (programmatic dependent launch), so a launch's span from its first CTA
    # to its last includes waiting for the previous launch; the kernel's own
    # time per call is then the call time itself.
    kernel_us = us_per_call if single_launch else span_us
    kernel_gbs = arm.touched / (kernel_us * 1e-6) / 1e9
    traffic = profiled_traffic()
    result = {
        "metric": "us/call (touched-weight HBM GB/s, % of peak) of one top-16 MoE decode layer call",
        "value": round(aggregate_us, 3),
        "unit": "us/call" if world == 1 else "us/call (job: calls of all replicas)",
        "per_replica_us_per_call": round(us_per_call, 3),
        "calls_per_s": round(world / (us_per_call * 1e-6), 1),
        "n_gpus": world,
        "steps": steps,
        "warmup": args.warmup,
        "ms_per_step": round(ms_per_call, 6),
        "higher_is_better": False,
        "scaling": "weak",
        "vs_baseline": None,
        "dtype": "e2m1 x e4m3 -> f32",
        "data": "synthetic (seeded: BF16 N(0,0.02) weights -> MXFP4, x ~ N(0,1))",
        "config": {
            "workload": describe(cfg),
            "touched_weight_bytes": arm.touched,
            "touched_gbs": round(gbs, 1),
            "touched_frac_of_peak": round(gbs / peak, 4),
            "l2": f"inputs larger than L2: {arm.R} weight replicas rotated "
                  f"({arm.R - 1} x {arm.touched / 1e6:.1f} MB >= 3 x {l2_bytes / 2**20:.0f} MiB L2)",
            "timing": f"CUDA graph of {calls_per_graph} back-to-back moe_run calls x {replays} "
                      f"replays, CUDA events",
            "parallelism": "replicas only" if world > 1 else "single GPU",
        },
        "roofline": {
            "bound": "hbm",
            "achieved": round(kernel_gbs, 1),
            "peak": peak,
            "unit": "GB/s",
            "frac": round(kernel_gbs / peak, 4),
            "traffic": traffic,
            "kernel": arm.kernel_label(),
            "kernel_us": round(kernel_us, 3),
            "kernel_us_how": (
                "the call is this one kernel launch, and back-to-back launches overlap, so the "
                "kernel's time per call is the timed per-call time; "
                if single_launch else "") +
                "in-step span of the experts kernel (first CTA start to last CTA end, device "
                f"clock): mean {span_us:.3f} us over {span_samples} launches inside replays of a "
                f"graph of {span_calls} back-to-back calls with the launch clock on "
                f"({span_pass_ms * 1e3:.3f} us/call in those replays)",
            "kernel_span_us": round(span_us, 3),
            "kernel_us_isolated": round(kernel_ms * 1e3, 3),
            "algorithmic_bytes": arm.touched,
            "peak_kind": f"{peak_kind} (copy bandwidth)",
        },
        "e2e": {
            "value": round(e2e_us, 3),
            "unit": "us/call",
            "h2d_bytes_per_step": arm.io_bytes["x"] + arm.io_bytes["ids"],
            "d2h_bytes_per_step": arm.io_bytes["out"],
        },
        "gpu_launches": arm.launches_per_call() * steps,
        "clocks": clocks,
    }

    if rank == 0:
        result["cpu_baseline"], oracle_ref = cpu_baseline(cfg, weights, x, ids)
        result["parity"] = parity_report(arm, oracle_ref)
    arm.close()
    if not args.no_extra:
        def graph_us(a, combined):
            """us per call of a graph of back-to-back calls (moe_run or moe_run_combined)."""
            a.combined = combined
            for i in range(max(3, args.warmup)):
                a.call(i)
            a.check_status()
            calls = max(a.R, min(64, args.steps))
            calls -= calls % a.R
            gg = a.graph(calls)
            gg.replay()
            reps = max(1, math.ceil(200 / calls))
            ms = a.time_graphs([(gg, reps)], reps * calls)
            a.check_status()
            a.combined = False
            return ms * 1e3

        extra = {}
        for name in [args.config] + EXTRA_CONFIGS:
            c = workload.CONFIGS[name]
            w, xx, ii = inputs(c)
            a = OurArm(c, device)
            a.setup(w, xx, ii, l2_bytes)
            combined_us = graph_us(a, True)
            if name == args.config:
                extra[name + " combined"] = {
                    "workload": describe(c) + ", routing-weighted combine to [B, H]",
                    "us_per_call": round(combined_us, 3)}
                a.close()
                continue
            ms = graph_us(a, False) * 1e-3
            kms = a.experts_kernel_ms(30)
            a.check_status()
            extra[name] = {
                "workload": describe(c), "us_per_call": round(ms * 1e3, 3),
                "combined_us_per_call": round(combined_us, 3),
                "touched_weight_bytes": a.touched,
                "touched_gbs": round(a.touched / (ms * 1e-3) / 1e9, 1),
                "touched_frac_of_peak": round(a.touched / (ms * 1e-3) / 1e9 / peak, 4),
                "experts_kernel_us": round(kms * 1e3, 3),
                "experts_kernel_frac_of_peak": round(a.touched / (kms * 1e-3) / 1e9 / peak, 4),
                "replicas": a.R,
            }
            a.close()
        result["configs"] = extra
    if world > 1:
        torch.distributed.destroy_process_group()
    if rank == 0:
        print(json.dumps(result), flush=True)


def run_reference(args, rank, world):
    if rank != 0:
        return
    import oracle

    cfg = workload.CONFIGS[args.config]
    weights, x, ids = workload.make_inputs(cfg)
    oracle_call_seconds(weights, x, ids, max(0, min(args.warmup, 3)))
    steps = max(1, min(args.steps, 20))
    times = oracle_call_seconds(weights, x, ids, steps)
    total = sum(times)
    us = total / steps * 1e6
    threads = oracle.default_threads()
    result = {
        "metric": "us/call (touched-weight HBM GB/s, % of peak) of one top-16 MoE decode layer call",
        "value": round(us, 1), "unit": "us/call", "n_gpus": world, "steps": steps,
        "warmup": args.warmup, "ms_per_step": round(us / 1e3, 3), "higher_is_better": False,
        "scaling": "weak", "vs_baseline": None, "dtype": "f64",
        "data": "synthetic (seeded: BF16 N(0,0.02) weights -> MXFP4, x ~ N(0,1))",
        "config": {"workload": describe(cfg), "parallelism": "host cores"},
        "impl": "reference",
        "cpu_baseline": {"value": round(us, 1), "unit": "us/call", "cores": threads,
                         "kind": "oracle",
                         "sample": f"{steps} whole {cfg.name} calls (all {ids.size} pairs); "
                                   f"--steps capped at 20 to bound the run"},
        "e2e": {"value": round(us, 1), "unit": "us/call", "h2d_bytes_per_step": 0,
                "d2h_bytes_per_step": 0},
    }
    print(json.dumps(result), flush=True)


def profile_case(args):
    """Run --steps calls of one workload on one prepared layer, nothing else."""
    import torch

    import mxfp4_weight_mxfp8_gb300 as moe

    cfg = workload.CONFIGS[args.config]
    weights, x, ids = workload.make_inputs(cfg)
    device = torch.device("cuda", 0)
    layer = moe.MoeLayer(tuple(torch.from_numpy(w).to(device) for w in weights))
    xd = torch.from_numpy(x.view(np.int16)).to(device).view(torch.bfloat16)
    idsd = torch.from_numpy(ids).to(device)
    for _ in range(max(1, args.steps)):
        layer(xd, idsd)
    status = moe.moe_sync_status(layer.handle)
    print(json.dumps({"profile_case": describe(cfg), "calls": args.steps, "status": status}))
    layer.close()
    if status != moe.MOE_OK:
        sys.exit(1)


def main():
    args = parse()
    rank, world, local = dist_env()
    if args.profile_case:
        profile_case(args)
        return
    if args.impl == "reference":
        run_reference(args, rank, world)
    else:
        run_ours(args, rank, world, local)


if __name__ == "__main__":
    main()
