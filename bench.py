#!/usr/bin/env python
"""Benchmark of the decode-attention hot path (append + split-KV decode with its merge).

Workload: the MHA decode sweep — B=1, 16 query heads on 16 KV heads, head_dim
128, fp16, kv_len in {1024, 4096, 8192} with capacity = kv_len. One step is
one decode token through every layer of a model whose layers each own a
static cache: for each kv_len, `layers` caches (enough that the caches of one
kv_len total at least 3x the L2 size, so every layer reads cold HBM), and for
every layer an in-place append at kv_len - 1 followed by attention over the
kv_len rows. The step's public API calls are captured once in a CUDA graph
and replayed (one graph per kv_len more for the per-kv_len rows); timing
uses CUDA events on the launching stream. The headline uses the library's default ordering; the same sweep
captured under its ordering promise (da_set_prefix_ready, which holds here
because consecutive calls use different layer caches) is reported beside it
as `other_ordering` (`--ordering ready` swaps the two).

Printed: one JSON line with the whole-job achieved HBM GB/s over algorithmic
bytes (K/V prefix read once + q read + out write + the appended rows), the
us per layer-step for each kv_len, the decode kernel's roofline (its own
launches timed with CUDA events placed around it), the end-to-end number
with per-step host<->device copies, the fp64 CPU oracle timed on the host's
cores, and the SM clocks seen during the run.

--impl reference times the CPU oracle alone on a bounded sample of the same
workload (the slow baseline arm).
"""
from __future__ import annotations

import argparse
import json
import math
import os
import pathlib
import statistics
import subprocess
import sys
import threading
import time

ROOT = pathlib.Path(__file__).resolve().parent
if str(ROOT) not in sys.path:
    sys.path.insert(0, str(ROOT))

METRIC = "decode-attn achieved HBM GB/s (% of GB300 peak); µs per layer-step vs kv_len"
UNIT = "GB/s"
SWEEP = (1024, 4096, 8192)
B, N_HEAD, N_KV_HEAD, HEAD_DIM = 1, 16, 16, 128
ELEM = 2  # fp16
WORKLOAD = ("MHA decode sweep: B=1, 16 query / 16 KV heads, head_dim 128, fp16, kv_len in {1024, 4096, 8192}, "
            "capacity = kv_len, append at kv_len-1 then attend")
FALLBACK_HBM_GBS = 6800.0
NOMINAL_HBM_GBS = 7900.0


# ---------------------------------------------------------------------------
# Byte model (algorithmic bytes: what the method must move at minimum).

def attend_bytes(batch: int, n_head: int, n_kv_head: int, head_dim: int, kv_lens, elem: int = ELEM) -> int:
    """K and V prefix rows read once, q read, out written."""
    return 2 * elem * n_kv_head * head_dim * int(sum(kv_lens)) + 2 * elem * batch * n_head * head_dim


def append_bytes(batch: int, n_kv_head: int, head_dim: int, elem: int = ELEM) -> int:
    """k_new and v_new read, one K row and one V row written per (b, kv head)."""
    return 4 * elem * batch * n_kv_head * head_dim


def expanded_full_capacity_bytes(n_head: int, capacity: int, head_dim: int, elem: int) -> int:
    """Logical K+V bytes of one layer when the KV heads are expanded to all
    query heads and the whole capacity is consumed (the cost the active-prefix
    slice removes)."""
    return 2 * n_head * capacity * head_dim * elem


def layers_for(kv_len: int, l2_bytes: int) -> int:
    """Layer caches per kv_len so that their K+V total at least 3x L2."""
    per_layer = 2 * N_KV_HEAD * kv_len * HEAD_DIM * ELEM
    return max(2, math.ceil(3 * l2_bytes / per_layer))


def measured_peaks() -> dict:
    p = ROOT / "MEASURED_PEAKS.json"
    if p.exists():
        try:
            return json.loads(p.read_text())
        except (OSError, ValueError):
            pass
    return {}


# ---------------------------------------------------------------------------
# Clock sampling with nvidia-smi during the run.

CLOCK_QUERY = ("index,clocks.sm,clocks.max.sm,power.draw,clocks_event_reasons.active,"
               "clocks_event_reasons.hw_slowdown,clocks_event_reasons.hw_thermal_slowdown,"
               "clocks_event_reasons.sw_thermal_slowdown,clocks_event_reasons.sw_power_cap")


class ClockSampler:
    def __init__(self, gpu_id: str | None, period_ms: int = 100):
        self.samples: list[list[str]] = []
        self.proc = None
        cmd = ["nvidia-smi", f"--query-gpu={CLOCK_QUERY}", "--format=csv,noheader,nounits", f"-lms={period_ms}"]
        if gpu_id:
            cmd.insert(1, f"--id={gpu_id}")
        try:
            self.proc = subprocess.Popen(cmd, stdout=subprocess.PIPE, stderr=subprocess.DEVNULL, text=True)
        except OSError:
            self.proc = None
            return
        self.thread = threading.Thread(target=self._read, daemon=True)
        self.thread.start()

    def _read(self):
        for line in self.proc.stdout:
            parts = [x.strip() for x in line.split(",")]
            if len(parts) >= 9:
                self.samples.append(parts)

    def stop(self) -> dict:
        if self.proc is None:
            return {"sm_mhz": None, "sm_max_mhz": None, "reasons": ["nvidia-smi unavailable"], "samples": 0}
        self.proc.terminate()
        try:
            self.proc.wait(timeout=5)
        except subprocess.TimeoutExpired:
            self.proc.kill()
        self.thread.join(timeout=5)
        sm, smax, reasons = [], [], set()
        names = ["hw_slowdown", "hw_thermal_slowdown", "sw_thermal_slowdown", "sw_power_cap"]
        for s in self.samples:
            try:
                sm.append(float(s[1]))
                smax.append(float(s[2]))
            except ValueError:
                continue
            for name, val in zip(names, s[5:9]):
                if val.lower().startswith("active"):
                    reasons.add(name)
        return {"sm_mhz": statistics.median(sm) if sm else None, "sm_max_mhz": max(smax) if smax else None,
                "reasons": sorted(reasons), "samples": len(sm)}


# ---------------------------------------------------------------------------
# The GPU arm.

class SweepStep:
    """Device state of one benchmark step and its CUDA-graph capture."""

    def __init__(self, torch, da, device, seed: int, fused: bool, kv_lens=SWEEP, ready: bool = False):
        self.torch, self.da, self.device, self.fused = torch, da, device, fused
        # ordering promise (da_set_prefix_ready): every call attends over its
        # own layer cache, written by no kernel still running when it starts
        self.ready = ready and fused
        props = torch.cuda.get_device_properties(device)
        self.l2_bytes = int(props.L2_cache_size)
        dt = torch.float16
        self.groups = []
        calls = []
        for kv in kv_lens:
            n_layers = layers_for(kv, self.l2_bytes)
            gen = torch.Generator(device=device)
            gen.manual_seed(seed * 1000003 + kv)
            shape = (n_layers, B, N_KV_HEAD, kv, HEAD_DIM)
            k = torch.empty(shape, dtype=dt, device=device)
            v = torch.empty(shape, dtype=dt, device=device)
            for t in (k, v):
                for layer in range(n_layers):  # layer by layer keeps the fp32 temporary small
                    t[layer].copy_(torch.randn(shape[1:], generator=gen, device=device, dtype=torch.float32))
            self.groups.append({"kv_len": kv, "layers": n_layers, "k": k, "v": v})
            calls += [(len(self.groups) - 1, layer) for layer in range(n_layers)]
        self.calls = calls
        n = len(calls)
        # Per-step inputs packed in one buffer: [call, (q, k_new, v_new), B, heads, D] plus positions.
        # One device buffer holds everything a step reads from the host side, so
        # that the end-to-end leg moves it with one copy: [inputs | positions |
        # kv_lens] (the inputs' size is a multiple of 16 bytes).
        in_bytes = n * 3 * B * N_HEAD * HEAD_DIM * ELEM
        self.packed = torch.empty(in_bytes + 2 * n * 4, dtype=torch.uint8, device=device)
        self.inputs = self.packed[:in_bytes].view(dt).view(n, 3, B, N_HEAD, HEAD_DIM)
        self.positions = self.packed[in_bytes:in_bytes + n * 4].view(torch.int32).view(n, 1)
        self.kv_lens = self.packed[in_bytes + n * 4:].view(torch.int32).view(n, 1)
        # bytes of the packed buffer the step's calls read (kv_lens only in the two-call path)
        self.h2d_bytes = in_bytes + n * 4 * (1 if fused else 2)
        gen = torch.Generator(device=device)
        gen.manual_seed(seed * 7 + 1)
        self.inputs.copy_(torch.randn(self.inputs.shape, generator=gen, device=device, dtype=torch.float32))
        self.positions.copy_(torch.tensor([[self.groups[g]["kv_len"] - 1] for g, _ in calls], dtype=torch.int32))
        self.kv_lens.copy_(self.positions + 1)
        self.out = torch.empty((n, B, N_HEAD, HEAD_DIM), dtype=dt, device=device)
        self.err = torch.zeros(1, dtype=torch.int32, device=device)
        ws = max(da.decode_attn_workspace_size(B, N_HEAD, N_KV_HEAD, HEAD_DIM, kv) for kv in kv_lens)
        self.workspace = torch.zeros(max(ws, 16), dtype=torch.uint8, device=device)  # counters start at zero
        # (splits, cluster size) of each kv_len's calls
        self.splits = {kv: da.splits_for(B, N_HEAD, N_KV_HEAD, HEAD_DIM, kv, kv, dt) for kv in kv_lens}

    # bytes -------------------------------------------------------------
    def call_attend_bytes(self, i: int) -> int:
        return attend_bytes(B, N_HEAD, N_KV_HEAD, HEAD_DIM, [self.groups[self.calls[i][0]]["kv_len"]])

    def step_bytes(self) -> int:
        return sum(self.call_attend_bytes(i) + append_bytes(B, N_KV_HEAD, HEAD_DIM) for i in range(len(self.calls)))

    def launches_per_step(self) -> int:
        # one decode launch per layer (the split merge runs inside it), plus
        # the append launch unless the step is fused
        return len(self.calls) * (1 if self.fused else 2)

    # issue -------------------------------------------------------------
    def issue(self, timing_events=None, group=None):
        da = self.da
        for i, (g, layer) in enumerate(self.calls):
            if group is not None and g != group:
                continue
            grp = self.groups[g]
            q, kn, vn = self.inputs[i, 0], self.inputs[i, 1], self.inputs[i, 2]
            kc, vc = grp["k"][layer], grp["v"][layer]
            if timing_events is not None:
                da.set_timing_events(*timing_events[i])
            if self.fused:
                da.decode_step_fwd(q, kc, vc, kn, vn, self.positions[i], out=self.out[i], workspace=self.workspace,
                                   max_kv_len_hint=grp["kv_len"], err_flag=self.err)
            else:
                da.kvcache_append(kc, vc, kn, vn, self.positions[i], err_flag=self.err)
                da.decode_attn_fwd(q, kc, vc, self.kv_lens[i], out=self.out[i], workspace=self.workspace,
                                   max_kv_len_hint=grp["kv_len"], err_flag=self.err)
        if timing_events is not None:
            da.set_timing_events(None, None)

    def capture(self, timing_events=None, group=None, ready=None):
        torch = self.torch
        ready = self.ready if ready is None else ready
        s = torch.cuda.Stream(self.device)
        s.wait_stream(torch.cuda.current_stream(self.device))
        with torch.cuda.stream(s):
            self.issue(group=group)  # eager warm-up: kernel attributes set before capture
        torch.cuda.current_stream(self.device).wait_stream(s)
        torch.cuda.synchronize(self.device)
        g = torch.cuda.CUDAGraph()
        self.da.set_prefix_ready(ready)
        try:
            with torch.cuda.graph(g):
                self.issue(timing_events, group)
        finally:
            self.da.set_prefix_ready(False)
        torch.cuda.synchronize(self.device)
        return g

    def group_calls(self, gi: int) -> list[int]:
        return [i for i, (g, _) in enumerate(self.calls) if g == gi]


def e2e_calls(torch, da, step, h_in, d_in, h_out, args, world, device, stream, mode: str) -> dict:
    """The end-to-end step without a CUDA graph: per step one pinned H2D copy
    of the inputs, every layer's public call issued from the host, one D2H
    copy of the outputs. mode "c_abi" calls the C entry point through ctypes
    with its arguments marshalled once (the host cost is the library's own:
    validation, split plan, launch); "binding" calls the Python binding (which
    also checks every tensor). Returns the time per step (ms) and the host
    time per call (µs)."""
    import ctypes

    lib = da.load_library()
    fused = step.fused
    calls = []
    sptr = ctypes.c_void_p(stream.cuda_stream)
    vp = lambda t: ctypes.c_void_p(t.data_ptr())  # noqa: E731
    ws_bytes = step.workspace.numel()
    for i, (g, layer) in enumerate(step.calls):
        grp = step.groups[g]
        q, kn, vn = step.inputs[i, 0], step.inputs[i, 1], step.inputs[i, 2]
        kc, vc = grp["k"][layer], grp["v"][layer]
        kv = grp["kv_len"]
        if mode == "c_abi":
            if fused:
                calls.append((lib.decode_step_fwd, (vp(q), vp(kc), vp(vc), vp(kn), vp(vn), vp(step.positions[i]), B,
                                                     N_HEAD, N_KV_HEAD, HEAD_DIM, kv, HEAD_DIM ** -0.5,
                                                     vp(step.out[i]), vp(step.workspace), ws_bytes, kv, 0,
                                                     vp(step.err), sptr)))
            else:
                calls.append((lib.kvcache_append, (vp(kc), vp(vc), vp(kn), vp(vn), vp(step.positions[i]), B,
                                                    N_KV_HEAD, HEAD_DIM, kv, 0, vp(step.err), sptr)))
                calls.append((lib.decode_attn_fwd, (vp(q), vp(kc), vp(vc), vp(step.kv_lens[i]), B, N_HEAD, N_KV_HEAD,
                                                     HEAD_DIM, kv, HEAD_DIM ** -0.5, vp(step.out[i]),
                                                     vp(step.workspace), ws_bytes, kv, 0, vp(step.err), sptr)))
        else:
            calls.append((i, q, kc, vc, kn, vn, kv))

    def issue():
        if mode == "c_abi":
            for fn, a in calls:
                if fn(*a) != 0:
                    raise RuntimeError("decode call failed")
        else:
            for i, q, kc, vc, kn, vn, kv in calls:
                if fused:
                    da.decode_step_fwd(q, kc, vc, kn, vn, step.positions[i], out=step.out[i],
                                       workspace=step.workspace, max_kv_len_hint=kv, err_flag=step.err)
                else:
                    da.kvcache_append(kc, vc, kn, vn, step.positions[i], err_flag=step.err)
                    da.decode_attn_fwd(q, kc, vc, step.kv_lens[i], out=step.out[i], workspace=step.workspace,
                                       max_kv_len_hint=kv, err_flag=step.err)

    with torch.cuda.stream(stream):
        for _ in range(max(3, args.warmup // 4)):
            d_in.copy_(h_in, non_blocking=True)
            issue()
            h_out.copy_(step.out, non_blocking=True)
        barrier(world, device)
        torch.cuda.synchronize(device)
        e0, e1 = torch.cuda.Event(enable_timing=True), torch.cuda.Event(enable_timing=True)
        host_s = 0.0
        wall0 = time.perf_counter()
        e0.record(stream)
        for _ in range(args.steps):
            d_in.copy_(h_in, non_blocking=True)
            t = time.perf_counter()
            issue()
            host_s += time.perf_counter() - t
            h_out.copy_(step.out, non_blocking=True)
        e1.record(stream)
        torch.cuda.synchronize(device)
        wall_ms = (time.perf_counter() - wall0) * 1e3
    ms = max(e0.elapsed_time(e1), wall_ms)
    ms_max = max_over_ranks(ms, world, device)
    n_calls = len(calls) * (2 if (mode == "binding" and not fused) else 1)
    return {"ms": ms_max, "host_us_per_call": round(host_s / (args.steps * n_calls) * 1e6, 2)}


def dist_env():
    world = int(os.environ.get("WORLD_SIZE", "1"))
    rank = int(os.environ.get("RANK", "0"))
    local = int(os.environ.get("LOCAL_RANK", "0"))
    return rank, world, local


def max_over_ranks(value: float, world: int, device=None) -> float:
    if world <= 1:
        return value
    import torch
    import torch.distributed as dist

    t = torch.tensor([value], dtype=torch.float64, device=device)
    dist.all_reduce(t, op=dist.ReduceOp.MAX)
    return float(t.item())


def barrier(world: int, device=None):
    if world > 1:
        import torch.distributed as dist

        if device is not None and str(device).startswith("cuda"):
            dist.barrier(device_ids=[device.index if hasattr(device, "index") else 0])
        else:
            dist.barrier()


def aggregate_value(bytes_per_rank_step: int, steps: int, world: int, max_ms: float) -> float:
    """Whole-job GB/s: the bytes all ranks processed over the slowest rank's time."""
    return world * bytes_per_rank_step * steps / (max_ms * 1e-3) / 1e9


def traffic_from_profiles(source_hash: str) -> dict | None:
    """ncu DRAM traffic per decode-kernel launch recorded under profiles/, if
    it was taken on the current kernel sources."""
    p = ROOT / "profiles" / "decode_split_kernel_mha_sweep.md"
    if not p.exists():
        return None
    rec = {}
    for line in p.read_text().splitlines():
        if line.startswith("- ") and ":" in line:
            k, _, v = line[2:].partition(":")
            rec[k.strip()] = v.strip().strip("`")
    if rec.get("kernel_source_sha256") != source_hash:
        return None
    try:
        return {kv: float(rec[f"traffic_bytes_kv{kv}"]) for kv in SWEEP}
    except (KeyError, ValueError):
        return None


def strip_comments(src: str) -> str:
    """C/C++ source without its comments and blank lines (string literals in
    these sources hold no comment markers)."""
    import re

    src = re.sub(r"/\*.*?\*/", "", src, flags=re.S)
    src = re.sub(r"//[^\n]*", "", src)
    return "\n".join(line.rstrip() for line in src.splitlines() if line.strip())


def kernel_source_hash() -> str:
    """Hash of the CUDA sources' code (comments excluded), which ties the ncu
    figures under profiles/ to the code they were taken on."""
    import hashlib

    h = hashlib.sha256()
    for f in sorted((ROOT / "decode_attention_static_gb300" / "csrc").glob("*")):
        h.update(f.name.encode())
        h.update(strip_comments(f.read_text()).encode())
    return h.hexdigest()[:16]


def run_ours(args) -> dict | None:
    import torch

    import decode_attention_static_gb300 as da

    rank, world, local = dist_env()
    if not torch.cuda.is_available():
        raise RuntimeError("bench.py needs a CUDA device for the GPU arm")
    device = torch.device("cuda", local)
    torch.cuda.set_device(device)
    if world > 1:
        import torch.distributed as dist

        dist.init_process_group("nccl", device_id=device)
    da.build_library()
    da.load_library()

    kv_lens = tuple(int(x) for x in args.kv_lens.split(","))
    step = SweepStep(torch, da, device, seed=args.seed + rank, fused=args.path == "fused", kv_lens=kv_lens,
                     ready=args.ordering == "ready")
    # one graph for the whole step (every layer of every kv_len, in order), and
    # one per kv_len for the per-kv_len timings
    step_graph = step.capture()
    graphs = [step.capture(group=gi) for gi in range(len(step.groups))]

    def replay_step():
        step_graph.replay()

    uuid = None
    try:
        uuid = "GPU-" + str(torch.cuda.get_device_properties(device).uuid)
    except Exception:  # noqa: BLE001 - older torch: sample every GPU
        uuid = None
    # sampled from the warm-up to the end of the last end-to-end leg (the
    # timed region alone can be shorter than one sampling period)
    clocks = ClockSampler(uuid)

    for _ in range(args.warmup):
        replay_step()
    torch.cuda.synchronize(device)
    if int(step.err.item()) != 0:
        raise RuntimeError(f"device error flag {int(step.err.item())}")

    # ---- timed region: exactly K steps ----
    stream = torch.cuda.current_stream(device)
    t0, t1 = torch.cuda.Event(enable_timing=True), torch.cuda.Event(enable_timing=True)
    barrier(world, device)
    torch.cuda.synchronize(device)
    t0.record(stream)
    for _ in range(args.steps):
        replay_step()
    t1.record(stream)
    torch.cuda.synchronize(device)
    barrier(world, device)
    ms = t0.elapsed_time(t1)
    ms_max = max_over_ranks(ms, world, device)

    # ---- us per layer-step for each kv_len: each group's graph timed alone ----
    group_ms = []
    for gi, g in enumerate(graphs):
        g.replay()
        a, b = torch.cuda.Event(enable_timing=True), torch.cuda.Event(enable_timing=True)
        torch.cuda.synchronize(device)
        a.record(stream)
        for _ in range(args.steps):
            g.replay()
        b.record(stream)
        torch.cuda.synchronize(device)
        group_ms.append(a.elapsed_time(b) / args.steps)

    # ---- the same sweep under the other ordering, beside it ----
    other = None
    if step.fused:
        def graph_ms(g) -> float:
            for _ in range(3):
                g.replay()
            a, b = torch.cuda.Event(enable_timing=True), torch.cuda.Event(enable_timing=True)
            torch.cuda.synchronize(device)
            a.record(stream)
            for _ in range(args.steps):
                g.replay()
            b.record(stream)
            torch.cuda.synchronize(device)
            return a.elapsed_time(b) / args.steps

        g = step.capture(ready=not step.ready)
        other = {"step_ms": graph_ms(g), "group_ms": []}
        del g
        for gi in range(len(step.groups)):
            g = step.capture(group=gi, ready=not step.ready)
            other["group_ms"].append(graph_ms(g))
            del g

    # ---- decode-kernel launch duration ----
    n = len(step.calls)
    if step.fused:
        # every launch of the timed region is a decode kernel: the average
        # launch duration is the timed region / its launches (the per-kv_len
        # rows below take each kv_len's graph timed alone)
        per_call = [group_ms[g] / step.groups[g]["layers"] for g, _ in step.calls]
        kernel_timing = "timed region / decode launches (the fused step launches only the decode kernel)"
    else:
        # events the library records right before and after each decode launch
        # (graph event nodes: includes the launch latency the nodes expose)
        evs = [(torch.cuda.Event(enable_timing=True), torch.cuda.Event(enable_timing=True)) for _ in range(n)]
        for a, b in evs:  # torch creates the CUDA event on its first record
            a.record(stream)
            b.record(stream)
        torch.cuda.synchronize(device)
        kgraph = step.capture(timing_events=evs)
        per_call = [0.0] * n
        reps = max(3, min(20, args.steps // 10))
        for _ in range(reps):
            kgraph.replay()
            torch.cuda.synchronize(device)
            for i, (a, b) in enumerate(evs):
                per_call[i] += a.elapsed_time(b)
        per_call = [x / reps for x in per_call]
        kernel_timing = "events recorded by the library around each decode launch (upper bound)"

    # ---- end to end: per-step H2D of the inputs and D2H of the outputs ----
    h_in = torch.empty(step.h2d_bytes, dtype=torch.uint8, pin_memory=True)
    h_in.copy_(step.packed[:step.h2d_bytes])
    d_in = step.packed[:step.h2d_bytes]
    h_out = torch.empty(step.out.shape, dtype=step.out.dtype, pin_memory=True)
    e0, e1 = torch.cuda.Event(enable_timing=True), torch.cuda.Event(enable_timing=True)
    for _ in range(max(1, args.warmup // 4)):
        d_in.copy_(h_in, non_blocking=True)
        replay_step()
        h_out.copy_(step.out, non_blocking=True)
    barrier(world, device)
    torch.cuda.synchronize(device)
    wall0 = time.perf_counter()
    e0.record(stream)
    for _ in range(args.steps):
        d_in.copy_(h_in, non_blocking=True)
        replay_step()
        h_out.copy_(step.out, non_blocking=True)
    e1.record(stream)
    torch.cuda.synchronize(device)
    wall_ms = (time.perf_counter() - wall0) * 1e3
    e2e_ms = max(e0.elapsed_time(e1), wall_ms)
    e2e_ms_max = max_over_ranks(e2e_ms, world, device)

    # ---- end to end without a graph: every layer's call made each step ----
    direct = e2e_calls(torch, da, step, h_in, d_in, h_out, args, world, device, stream, mode="c_abi")
    binding = e2e_calls(torch, da, step, h_in, d_in, h_out, args, world, device, stream, mode="binding")
    if int(step.err.item()) != 0:
        raise RuntimeError(f"device error flag {int(step.err.item())}")

    if world > 1:
        import torch.distributed as dist

        dist.destroy_process_group()
    if rank != 0:
        clocks.stop()
        return None

    bytes_step = step.step_bytes()
    value = aggregate_value(bytes_step, args.steps, world, ms_max)
    peaks = measured_peaks()
    peak = float(peaks.get("hbm_gbs") or FALLBACK_HBM_GBS)
    peak_src = "measured" if peaks.get("hbm_gbs") else "fallback"

    sweep = []
    for gi, grp in enumerate(step.groups):
        idx = step.group_calls(gi)
        kms = sum(per_call[i] for i in idx)
        kb = sum(step.call_attend_bytes(i) for i in idx)
        step_b = sum(step.call_attend_bytes(i) + append_bytes(B, N_KV_HEAD, HEAD_DIM) for i in idx)
        splits, cluster = step.splits[grp["kv_len"]]
        sweep.append({"kv_len": grp["kv_len"], "layers": grp["layers"], "splits": splits, "cluster": cluster,
                      "us_per_layer_step": round(group_ms[gi] / len(idx) * 1e3, 3),
                      "gbs": round(step_b / (group_ms[gi] * 1e-3) / 1e9, 1),
                      "decode_kernel_us": round(kms / len(idx) * 1e3, 3),
                      "decode_kernel_gbs": round(kb / (kms * 1e-3) / 1e9, 1)})

    k_bytes = sum(step.call_attend_bytes(i) for i in range(n))
    k_ms = ms_max / args.steps if step.fused else sum(per_call)
    achieved = k_bytes / (k_ms * 1e-3) / 1e9
    traffic = traffic_from_profiles(kernel_source_hash())
    traffic_per_launch = None
    if traffic:
        traffic_per_launch = sum(traffic[step.groups[g]["kv_len"]] for g, _ in step.calls) / n

    out = {
        "metric": METRIC, "value": round(value, 1), "unit": UNIT, "n_gpus": world, "steps": args.steps,
        "warmup": args.warmup, "ms_per_step": round(ms_max / args.steps, 5), "higher_is_better": True,
        "scaling": "weak", "vs_baseline": None, "dtype": "f16", "data": "synthetic",
        "config": {"workload": WORKLOAD if kv_lens == SWEEP else f"{WORKLOAD} (subset kv_len {list(kv_lens)})",
                   "path": "fused append+attend" if step.fused else "append, then attend",
                   "layers_per_kv_len": {str(g["kv_len"]): g["layers"] for g in step.groups},
                   "l2": f"inputs larger than L2: each kv_len's layer caches total >= 3x L2 ({step.l2_bytes} B)",
                   "timing": "CUDA-graph replay of the public calls (one graph per step; one per kv_len for "
                             "the per-kv_len rows), CUDA events on the launching stream",
                   "ordering": ("prefix ready: da_set_prefix_ready(1) for the captured calls (each layer's cache "
                                "is written by no kernel still running when its call starts), so short chunks are "
                                "copied before the grid wait" if step.ready else
                                "strict: every decode kernel waits for the previous kernel before reading"),
                   "parallelism": f"replicas x{world}" if world > 1 else "single GPU",
                   "bytes_per_step": bytes_step},
        "pct_of_peak_hbm": round(100 * value / peak, 1),
        "pct_of_nominal_hbm": round(100 * value / NOMINAL_HBM_GBS, 1),
        "sweep": sweep,
        "roofline": {"kernel": "decode_split_kernel", "bound": "hbm", "achieved": round(achieved, 1),
                     "peak": peak, "peak_source": peak_src, "unit": "GB/s", "frac": round(achieved / peak, 4),
                     "traffic": None if traffic_per_launch is None else round(traffic_per_launch),
                     "algorithmic_bytes_per_launch": round(k_bytes / n),
                     "avg_launch_us": round(k_ms / n * 1e3, 3), "timing": kernel_timing},
        "e2e": {"value": round(aggregate_value(bytes_step, args.steps, world, e2e_ms_max), 1), "unit": UNIT,
                "h2d_bytes_per_step": step.h2d_bytes,
                "d2h_bytes_per_step": step.out.numel() * ELEM,
                "mode": "one pinned H2D copy of every layer's q/k_new/v_new and positions, graph replay, one D2H "
                        "copy of the outputs"},
        "e2e_direct": {"value": round(aggregate_value(bytes_step, args.steps, world, direct["ms"]), 1), "unit": UNIT,
                       "h2d_bytes_per_step": step.h2d_bytes, "d2h_bytes_per_step": step.out.numel() * ELEM,
                       "host_us_per_call": direct["host_us_per_call"],
                       "mode": "no graph: one pinned H2D copy of the step's inputs, then every layer's call made "
                               "through the C ABI (ctypes, arguments marshalled once), then one D2H copy of the "
                               "outputs; wall clock and CUDA events, the larger"},
        "e2e_binding": {"value": round(aggregate_value(bytes_step, args.steps, world, binding["ms"]), 1), "unit": UNIT,
                        "host_us_per_call": binding["host_us_per_call"],
                        "mode": "as e2e_direct, every call through the Python binding (tensor checks per call)"},
        "gpu_launches": step.launches_per_step() * args.steps,
    }
    if other is not None:
        idx = [step.group_calls(gi) for gi in range(len(step.groups))]
        out["other_ordering"] = {
            "ordering": "strict" if step.ready else "prefix ready",
            "value": round(bytes_step / (other["step_ms"] * 1e-3) / 1e9, 1), "unit": UNIT,
            "ms_per_step": round(other["step_ms"], 5),
            "us_per_layer_step": {str(grp["kv_len"]): round(other["group_ms"][gi] / len(idx[gi]) * 1e3, 3)
                                  for gi, grp in enumerate(step.groups)},
            "timing": "the step's graph and each kv_len's graph captured under the other ordering, timed like the "
                      "headline"}
    if not args.no_extras and rank == 0:
        out["attend_only"] = attend_only(torch, da, device, step.l2_bytes)
        out["sweep_layers_call"] = sweep_layers_call(torch, da, step, device, args.steps)
        out["kv_curve"] = kv_curve(torch, da, device, step.l2_bytes)
        out["configs"] = other_configs(torch, da, device, step.l2_bytes)
    # clocks seen from the warm-up to the end of the last GPU leg
    out["clocks"] = clocks.stop()
    if not args.no_cpu_baseline:
        out["cpu_baseline"] = cpu_baseline(args.cpu_seconds)
    return out


# ---------------------------------------------------------------------------
# Other configurations, reported beside the headline sweep (not part of
# `value`): the µs-vs-kv_len curve at the long-context shape and the other
# workloads of the method, each timed as a CUDA graph of public calls.

CURVE_KV = (256, 512, 1024, 2048, 4096, 8192, 16384, 32768)


def graph_us_per_call(torch, device, issue, calls: int, reps: int, flush=None) -> float:
    """µs per public call: `issue()` makes `calls` calls; it is captured once
    in a CUDA graph and replayed `reps` times between CUDA events. With
    `flush`, L2 is flushed before every replay, outside the timed events."""
    issue()
    torch.cuda.synchronize(device)
    g = torch.cuda.CUDAGraph()
    with torch.cuda.graph(g):
        issue()
    for _ in range(3):
        g.replay()
    torch.cuda.synchronize(device)
    if flush is None:
        a, b = torch.cuda.Event(enable_timing=True), torch.cuda.Event(enable_timing=True)
        a.record()
        for _ in range(reps):
            g.replay()
        b.record()
        torch.cuda.synchronize(device)
        return a.elapsed_time(b) * 1e3 / (reps * calls)
    total = 0.0
    for _ in range(reps):
        flush()
        a, b = torch.cuda.Event(enable_timing=True), torch.cuda.Event(enable_timing=True)
        a.record()
        g.replay()
        b.record()
        torch.cuda.synchronize(device)
        total += a.elapsed_time(b)
    return total * 1e3 / (reps * calls)


def kv_curve(torch, da, device, l2_bytes: int) -> list:
    """Long-context shape (B=1, 32 query / 8 KV heads, head_dim 128, bf16),
    fused append + attend per call, over rotating layer caches totalling at
    least 3x L2, for each kv_len of CURVE_KV."""
    H, Hkv, D, dt = 32, 8, 128, torch.bfloat16
    gen = torch.Generator(device="cpu").manual_seed(11)
    res = []
    for kv in CURVE_KV:
        per_layer = 2 * Hkv * kv * D * 2
        layers = max(2, math.ceil(3 * l2_bytes / per_layer))
        k = torch.empty(layers, 1, Hkv, kv, D, dtype=dt, device=device).normal_()
        v = torch.empty_like(k).normal_()
        q = torch.randn(layers, 1, H, D, generator=gen).to(dt).to(device)
        kn = torch.randn(layers, 1, Hkv, D, generator=gen).to(dt).to(device)
        vn = torch.randn(layers, 1, Hkv, D, generator=gen).to(dt).to(device)
        out = torch.empty_like(q)
        pos = torch.full((1,), kv - 1, dtype=torch.int32, device=device)
        ws = da.alloc_workspace(1, H, Hkv, D, kv)

        def issue():
            for l in range(layers):
                da.decode_step_fwd(q[l], k[l], v[l], kn[l], vn[l], pos, out=out[l], workspace=ws,
                                   max_kv_len_hint=kv)

        us = graph_us_per_call(torch, device, issue, layers, reps=max(3, 2000 // layers))
        b = attend_bytes(1, H, Hkv, D, [kv], 2) + append_bytes(1, Hkv, D, 2)
        s, cs = da.splits_for(1, H, Hkv, D, kv, kv, dt)
        res.append({"kv_len": kv, "layers": layers, "splits": s, "cluster": cs,
                    "kernel": da.kernel_for(1, H, Hkv, D, kv, kv, dt), "us_per_layer_step": round(us, 3),
                    "gbs": round(b / (us * 1e-6) / 1e9, 1)})
        del k, v
    return res


def sweep_layers_call(torch, da, step, device, steps: int) -> dict:
    """The headline step with every kv_len's layers in ONE decode_step_layers_fwd
    launch (3 launches per step instead of 69): what the library gives a caller
    that holds every layer's inputs at once. Not the headline, which times one
    dependent call per layer."""
    ws = {}
    for gi, grp in enumerate(step.groups):
        n = grp["layers"]
        ws[gi] = da.alloc_workspace(n * B, N_HEAD, N_KV_HEAD, HEAD_DIM, grp["kv_len"], device)
    idx = [step.group_calls(gi) for gi in range(len(step.groups))]

    def issue():
        for gi, grp in enumerate(step.groups):
            i0, i1 = idx[gi][0], idx[gi][-1] + 1   # this group's calls are consecutive
            q = step.inputs[i0:i1, 0]
            kn, vn = step.inputs[i0:i1, 1], step.inputs[i0:i1, 2]
            # each layer's positions are the same: one [B] vector
            da.decode_step_layers_fwd(q.contiguous(), grp["k"], grp["v"], kn.contiguous(), vn.contiguous(),
                                      step.positions[i0], out=step.out[i0:i1], workspace=ws[gi],
                                      max_kv_len_hint=grp["kv_len"], err_flag=step.err)

    ms = graph_us_per_call(torch, device, issue, 1, max(3, steps)) / 1e3
    b = step.step_bytes()
    return {"ms_per_step": round(ms, 5), "value": round(b / (ms * 1e-3) / 1e9, 1), "unit": UNIT,
            "launches_per_step": len(step.groups),
            "timing": "one CUDA graph of 3 decode_step_layers_fwd calls (one per kv_len) replayed; the q, k_new and "
                      "v_new of a group are copied into contiguous stacks inside the graph"}


def attend_only(torch, da, device, l2_bytes: int) -> list:
    """The sweep's shape (B=1, 16/16 heads, head_dim 128, fp16) with attention
    alone (decode_attn_fwd on a prefix already in the cache, no append), over
    rotating layer caches totalling at least 3x L2: the step without its
    append."""
    res = []
    for kv in SWEEP:
        layers = layers_for(kv, l2_bytes)
        k = torch.empty(layers, B, N_KV_HEAD, kv, HEAD_DIM, dtype=torch.float16, device=device).normal_()
        v = torch.empty_like(k).normal_()
        q = torch.empty(layers, B, N_HEAD, HEAD_DIM, dtype=torch.float16, device=device).normal_()
        out = torch.empty_like(q)
        lens = torch.full((B,), kv, dtype=torch.int32, device=device)
        ws = da.alloc_workspace(B, N_HEAD, N_KV_HEAD, HEAD_DIM, kv)

        def issue():
            for l in range(layers):
                da.decode_attn_fwd(q[l], k[l], v[l], lens, out=out[l], workspace=ws, max_kv_len_hint=kv)

        us = graph_us_per_call(torch, device, issue, layers, reps=max(3, 2000 // layers))
        b = attend_bytes(B, N_HEAD, N_KV_HEAD, HEAD_DIM, [kv])
        res.append({"kv_len": kv, "us_per_call": round(us, 3), "gbs": round(b / (us * 1e-6) / 1e9, 1)})
        del k, v
    return res


def other_configs(torch, da, device, l2_bytes: int) -> dict:
    """The tiny GQA step, the batched streaming step and S2-Pro-shaped
    generation layer-steps (36 layers of 32 / 8 heads, bf16, capacity 32768)."""
    import workloads as W

    res = {}
    flush_buf = torch.empty(3 * l2_bytes // 4 + 1, dtype=torch.int32, device=device)

    def flush():
        flush_buf.fill_(1)

    # tiny GQA: one fused step, launch-bound
    t = W.tiny_gqa(seed=0)
    t_hint = int(t.position_ids.max()) + 1
    t = t.to(device)
    ws = da.alloc_workspace(t.B, t.n_head, t.n_kv_head, t.head_dim, t.capacity)

    def issue_tiny():
        for _ in range(64):
            da.decode_step_fwd(t.q, t.k_cache, t.v_cache, t.k_new, t.v_new, t.position_ids, workspace=ws,
                               max_kv_len_hint=t_hint)

    res["tiny_gqa"] = {"us_per_layer_step": round(graph_us_per_call(torch, device, issue_tiny, 64, 50), 3),
                       "kernel": da.kernel_for(t.B, t.n_head, t.n_kv_head, t.head_dim, t.capacity, t_hint,
                                               t.q.dtype)}

    # batched streaming: B=8, 16 / 8 heads, capacity 8192, ragged lengths; three
    # copies of the caches rotate so that consecutive calls read cold HBM
    s0 = W.batched_streaming(seed=4)
    hint = int(s0.position_ids.max()) + 1
    kvs = (s0.position_ids + 1).tolist()
    s0 = s0.to(device)
    kc = [s0.k_cache] + [s0.k_cache.clone() for _ in range(2)]
    vc = [s0.v_cache] + [s0.v_cache.clone() for _ in range(2)]
    ws = da.alloc_workspace(s0.B, s0.n_head, s0.n_kv_head, s0.head_dim, s0.capacity)

    def issue_batch():
        for i in range(6):
            da.decode_step_fwd(s0.q, kc[i % 3], vc[i % 3], s0.k_new, s0.v_new, s0.position_ids, workspace=ws,
                               max_kv_len_hint=hint)

    us = graph_us_per_call(torch, device, issue_batch, 6, 30)
    b = attend_bytes(s0.B, s0.n_head, s0.n_kv_head, s0.head_dim, kvs, 2) + append_bytes(s0.B, s0.n_kv_head,
                                                                                        s0.head_dim, 2)
    res["batched_streaming"] = {"us_per_layer_step": round(us, 3), "gbs": round(b / (us * 1e-6) / 1e9, 1),
                                "sum_kv_len": int(sum(kvs)),
                                "kernel": da.kernel_for(s0.B, s0.n_head, s0.n_kv_head, s0.head_dim, s0.capacity,
                                                        hint, s0.q.dtype)}
    del kc, vc, s0

    # S2-Pro-shaped generation: every layer's step at three positions of the
    # 400-step run (kv_len 235, 435, 634), as run (prefix warm in L2, as right
    # after the previous step) and with L2 flushed before each 36-layer step
    layers, H, Hkv, D, cap, dt = 36, 32, 8, 128, 32768, torch.bfloat16
    k = torch.empty(layers, 1, Hkv, cap, D, dtype=dt, device=device).normal_()
    v = torch.empty_like(k).normal_()
    gen = torch.Generator(device="cpu").manual_seed(12)
    q = torch.randn(layers, 1, H, D, generator=gen).to(dt).to(device)
    kn = torch.randn(layers, 1, Hkv, D, generator=gen).to(dt).to(device)
    vn = torch.randn(layers, 1, Hkv, D, generator=gen).to(dt).to(device)
    out = torch.empty_like(q)
    ws = da.alloc_workspace(1, H, Hkv, D, cap)
    ws_layers = da.alloc_workspace(layers, H, Hkv, D, cap)
    gen_res = []
    for kv in (235, 435, 634):
        pos = torch.full((1,), kv - 1, dtype=torch.int32, device=device)

        def issue_s2():
            for l in range(layers):
                da.decode_step_fwd(q[l], k[l], v[l], kn[l], vn[l], pos, out=out[l], workspace=ws,
                                   max_kv_len_hint=kv)

        def issue_layers():
            da.decode_step_layers_fwd(q, k, v, kn, vn, pos, out=out, workspace=ws_layers, max_kv_len_hint=kv)

        warm = graph_us_per_call(torch, device, issue_s2, layers, 50)
        cold = graph_us_per_call(torch, device, issue_s2, layers, 20, flush=flush)
        # every layer of the step in one launch (decode_step_layers_fwd), per layer-step
        lw = graph_us_per_call(torch, device, issue_layers, 1, 200) / layers
        lc = graph_us_per_call(torch, device, issue_layers, 1, 20, flush=flush) / layers
        b = attend_bytes(1, H, Hkv, D, [kv], 2) + append_bytes(1, Hkv, D, 2)
        gen_res.append({"kv_len": kv, "kernel": da.kernel_for(1, H, Hkv, D, cap, kv, dt),
                        "layers_call_kernel": da.kernel_for(layers, H, Hkv, D, cap, kv, dt),
                        "us_per_layer_step_as_run": round(warm, 3),
                        "us_per_layer_step_l2_flushed": round(cold, 3),
                        "gbs_l2_flushed": round(b / (cold * 1e-6) / 1e9, 1),
                        "layers_call_us_per_layer_step_as_run": round(lw, 3),
                        "layers_call_us_per_layer_step_l2_flushed": round(lc, 3),
                        "layers_call_gbs_l2_flushed": round(b / (lc * 1e-6) / 1e9, 1)})
    res["s2pro_generation"] = gen_res
    del k, v, flush_buf
    return res


# ---------------------------------------------------------------------------
# The CPU oracle (the baseline arm and the cpu_baseline leg).

def cpu_sample(n_heads: int = N_HEAD, seed: int = 0):
    """One layer-step per kv_len of the sweep on the host (first n_heads heads)."""
    import workloads as W

    items = []
    for kv in SWEEP:
        s = W.mha_sweep(kv, seed=seed)
        items.append({
            "kv_len": kv,
            "q": W.raw_bits(s.q[:, :n_heads]).copy(),
            "k": W.raw_bits(s.k_cache[:, :n_heads]).copy(),
            "v": W.raw_bits(s.v_cache[:, :n_heads]).copy(),
            "k_new": W.raw_bits(s.k_new[:, :n_heads]).copy(),
            "v_new": W.raw_bits(s.v_new[:, :n_heads]).copy(),
            "pos": s.position_ids.numpy().copy(),
        })
    bytes_ = sum(attend_bytes(B, n_heads, n_heads, HEAD_DIM, [it["kv_len"]]) + append_bytes(B, n_heads, HEAD_DIM)
                 for it in items)
    return items, bytes_


def oracle_pass(ora, items, n_heads: int, threads: int):
    for it in items:
        ora.kvcache_append(it["k"], it["v"], it["k_new"], it["v_new"], it["pos"])
        ora.decode_attn(it["q"], it["k"], it["v"], it["pos"] + 1, n_heads, n_heads, "f16", threads=threads)


def cpu_baseline(budget_s: float) -> dict:
    import oracle

    ora = oracle.default()
    threads = min(os.cpu_count() or 1, N_HEAD)
    items, bytes_ = cpu_sample()
    oracle_pass(ora, items, N_HEAD, threads)  # warm
    passes, t0 = 0, time.perf_counter()
    while True:
        oracle_pass(ora, items, N_HEAD, threads)
        passes += 1
        el = time.perf_counter() - t0
        if el >= budget_s:
            break
    value = bytes_ * passes / el / 1e9
    passes1, t1 = 0, time.perf_counter()
    while True:
        oracle_pass(ora, items, N_HEAD, 1)
        passes1 += 1
        el1 = time.perf_counter() - t1
        if el1 >= budget_s / 2:
            break
    return {"value": round(value, 4), "unit": UNIT, "cores": threads, "kind": "oracle",
            "value_1_thread": round(bytes_ * passes1 / el1 / 1e9, 4), "cpu_model": cpu_model(),
            "sample": f"{passes} pass(es) of one layer-step per kv_len in {{1024, 4096, 8192}} (16 heads, append "
                      f"+ attend) in {el:.1f} s, fp64 C oracle, OpenMP over query heads; then {passes1} pass(es) "
                      f"on one thread in {el1:.1f} s"}


def cpu_model() -> str:
    """The host CPU's model string (or architecture when none is published)."""
    try:
        out = subprocess.run(["lscpu"], capture_output=True, text=True, timeout=10).stdout
        for line in out.splitlines():
            if line.lower().startswith("model name:"):
                name = line.split(":", 1)[1].strip()
                if name and name != "-":
                    return name
    except (OSError, subprocess.SubprocessError):
        pass
    try:
        for line in pathlib.Path("/proc/cpuinfo").read_text().splitlines():
            key = line.split(":")[0].strip().lower()
            if key in ("model name", "cpu model", "hardware"):
                return line.split(":", 1)[1].strip()
    except OSError:
        pass
    import platform

    return platform.machine() or "unknown"


def run_reference(args) -> dict | None:
    rank, world, _ = dist_env()
    if rank != 0:
        return None
    import oracle

    ora = oracle.default()
    threads = min(os.cpu_count() or 1, N_HEAD)
    # size the sample so that warmup + steps fit in about two minutes
    items, bytes_ = cpu_sample()
    t = time.perf_counter()
    oracle_pass(ora, items, N_HEAD, threads)
    full = time.perf_counter() - t
    per_step_budget = 120.0 / max(1, args.steps + args.warmup)
    n_heads = max(1, min(N_HEAD, int(N_HEAD * per_step_budget / max(full, 1e-9))))
    items, bytes_ = cpu_sample(n_heads)
    threads = min(threads, n_heads)
    for _ in range(args.warmup):
        oracle_pass(ora, items, n_heads, threads)
    t0 = time.perf_counter()
    for _ in range(args.steps):
        oracle_pass(ora, items, n_heads, threads)
    el = time.perf_counter() - t0
    value = bytes_ * args.steps / el / 1e9
    sample = (f"each step: one layer-step per kv_len in {{1024, 4096, 8192}} on {n_heads} of the 16 heads "
              f"(append + attend), fp64 C oracle, {threads} OpenMP thread(s)")
    return {
        "impl": "reference", "metric": METRIC, "value": round(value, 4), "unit": UNIT, "n_gpus": world,
        "steps": args.steps, "warmup": args.warmup, "ms_per_step": round(el / args.steps * 1e3, 3),
        "higher_is_better": True, "scaling": "weak", "vs_baseline": None, "dtype": "f64", "data": "synthetic",
        "config": {"workload": WORKLOAD, "sample_heads": n_heads},
        "cpu_baseline": {"value": round(value, 4), "unit": UNIT, "cores": threads, "kind": "oracle",
                         "sample": sample},
        "e2e": {"value": round(value, 4), "unit": UNIT, "h2d_bytes_per_step": 0, "d2h_bytes_per_step": 0},
    }


def run_case(args) -> dict:
    """One named workload alone (for profiling one kernel instance): its CUDA
    graph of public calls over rotating layer caches (>= 3x L2) replayed
    `--warmup` then `--steps` times. Cases: long_context:<kv> (B=1, 32 / 8
    heads, bf16, fused step), rope:<kv> (the same with rotary embedding),
    mha:<kv> (B=1, 16 / 16 heads, fp16, fused step), batched (B=8, 16 / 8
    heads, bf16, capacity 8192, ragged positions), s2pro_layers:<kv> (36
    layers of 32 / 8 heads, bf16, capacity 32768, one decode_step_layers_fwd
    launch per step)."""
    import torch

    import decode_attention_static_gb300 as da
    import workloads as W

    device = torch.device("cuda", 0)
    torch.cuda.set_device(device)
    da.build_library()
    da.load_library()
    l2 = int(torch.cuda.get_device_properties(device).L2_cache_size)
    name, _, arg = args.case.partition(":")
    kv = int(arg) if arg else 8192
    gen = torch.Generator(device="cpu").manual_seed(13)
    if name in ("long_context", "rope", "mha"):
        H, Hkv, dt = (16, 16, torch.float16) if name == "mha" else (32, 8, torch.bfloat16)
        D = 128
        layers = max(2, math.ceil(3 * l2 / (2 * Hkv * kv * D * 2)))
        k = torch.empty(layers, 1, Hkv, kv, D, dtype=dt, device=device).normal_()
        v = torch.empty_like(k).normal_()
        q = torch.randn(layers, 1, H, D, generator=gen).to(dt).to(device)
        kn = torch.randn(layers, 1, Hkv, D, generator=gen).to(dt).to(device)
        vn = torch.randn(layers, 1, Hkv, D, generator=gen).to(dt).to(device)
        out = torch.empty_like(q)
        pos = torch.full((1,), kv - 1, dtype=torch.int32, device=device)
        ws = da.alloc_workspace(1, H, Hkv, D, kv)
        cos, sin = W.rope_tables(kv, D)
        cos, sin = cos.to(device), sin.to(device)
        calls = layers

        def issue():
            for l in range(layers):
                if name == "rope":
                    da.decode_step_rope_fwd(q[l], k[l], v[l], kn[l], vn[l], cos, sin, pos, out=out[l], workspace=ws,
                                            max_kv_len_hint=kv)
                else:
                    da.decode_step_fwd(q[l], k[l], v[l], kn[l], vn[l], pos, out=out[l], workspace=ws,
                                       max_kv_len_hint=kv)
        nbytes = layers * (attend_bytes(1, H, Hkv, D, [kv], 2) + append_bytes(1, Hkv, D, 2))
    elif name == "batched":
        s0 = W.batched_streaming(seed=4)
        hint = int(s0.position_ids.max()) + 1
        kvs = (s0.position_ids + 1).tolist()
        s0 = s0.to(device)
        kc = [s0.k_cache] + [s0.k_cache.clone() for _ in range(2)]
        vc = [s0.v_cache] + [s0.v_cache.clone() for _ in range(2)]
        ws = da.alloc_workspace(s0.B, s0.n_head, s0.n_kv_head, s0.head_dim, s0.capacity)
        calls = 6

        def issue():
            for i in range(calls):
                da.decode_step_fwd(s0.q, kc[i % 3], vc[i % 3], s0.k_new, s0.v_new, s0.position_ids, workspace=ws,
                                   max_kv_len_hint=hint)
        nbytes = calls * (attend_bytes(s0.B, s0.n_head, s0.n_kv_head, s0.head_dim, kvs, 2)
                          + append_bytes(s0.B, s0.n_kv_head, s0.head_dim, 2))
    elif name == "s2pro_layers":
        layers, H, Hkv, D, cap, dt = 36, 32, 8, 128, 32768, torch.bfloat16
        k = torch.empty(layers, 1, Hkv, cap, D, dtype=dt, device=device).normal_()
        v = torch.empty_like(k).normal_()
        q = torch.randn(layers, 1, H, D, generator=gen).to(dt).to(device)
        kn = torch.randn(layers, 1, Hkv, D, generator=gen).to(dt).to(device)
        vn = torch.randn(layers, 1, Hkv, D, generator=gen).to(dt).to(device)
        out = torch.empty_like(q)
        pos = torch.full((1,), kv - 1, dtype=torch.int32, device=device)
        ws = da.alloc_workspace(layers, H, Hkv, D, cap)
        calls = 1

        def issue():
            da.decode_step_layers_fwd(q, k, v, kn, vn, pos, out=out, workspace=ws, max_kv_len_hint=kv)
        nbytes = layers * (attend_bytes(1, H, Hkv, D, [kv], 2) + append_bytes(1, Hkv, D, 2))
    else:
        raise SystemExit(f"unknown case {args.case!r}")
    issue()
    torch.cuda.synchronize(device)
    g = torch.cuda.CUDAGraph()
    with torch.cuda.graph(g):
        issue()
    for _ in range(args.warmup):
        g.replay()
    torch.cuda.synchronize(device)
    a, b = torch.cuda.Event(enable_timing=True), torch.cuda.Event(enable_timing=True)
    a.record()
    for _ in range(args.steps):
        g.replay()
    b.record()
    torch.cuda.synchronize(device)
    ms = a.elapsed_time(b) / args.steps
    return {"case": args.case, "calls_per_replay": calls, "us_per_call": round(ms * 1e3 / calls, 3),
            "gbs": round(nbytes / (ms * 1e-3) / 1e9, 1), "steps": args.steps, "warmup": args.warmup}


def main(argv=None):
    ap = argparse.ArgumentParser(description=__doc__.splitlines()[0])
    ap.add_argument("--gpus", type=int, default=1)
    ap.add_argument("--steps", type=int, default=2000)
    ap.add_argument("--warmup", type=int, default=50)
    ap.add_argument("--impl", choices=["ours", "reference"], default="ours")
    ap.add_argument("--path", choices=["two_call", "fused"], default="fused",
                    help="fused: one decode_step_fwd per layer; two_call: kvcache_append then decode_attn_fwd")
    ap.add_argument("--ordering", choices=["strict", "ready"], default="strict",
                    help="strict: the library's default ordering; ready: capture the fused calls under "
                         "da_set_prefix_ready (each layer's cache is written by no kernel still running when its "
                         "call starts). The other one is reported beside the headline.")
    ap.add_argument("--seed", type=int, default=0)
    ap.add_argument("--kv-lens", default=",".join(map(str, SWEEP)),
                    help="kv_len values of the sweep to run (a subset gives a smaller case, e.g. for profiling)")
    ap.add_argument("--cpu-seconds", type=float, default=10.0)
    ap.add_argument("--no-cpu-baseline", action="store_true")
    ap.add_argument("--no-extras", action="store_true",
                    help="skip the kv_len curve and the other configurations (reported beside the sweep)")
    ap.add_argument("--case", default=None,
                    help="run one named workload alone and print its timing (for profiling one kernel instance): "
                         "long_context:<kv>, rope:<kv>, mha:<kv>, batched, s2pro_layers:<kv>")
    args = ap.parse_args(argv)
    if args.warmup < 3:
        ap.error("--warmup must be at least 3")
    if args.case:
        print(json.dumps(run_case(args)), flush=True)
        return
    res = run_reference(args) if args.impl == "reference" else run_ours(args)
    if res is not None:
        print(json.dumps(res), flush=True)


if __name__ == "__main__":
    main()
