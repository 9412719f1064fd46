#!/usr/bin/env python
"""Benchmark of the FP8 live-quant MoE expert projection on GB300.

One step = one full MoE layer forward for M tokens through the C ABI
(moeq_moe_layer: route, fused quant + gate_up + SwiGLU, fused quant + down,
combine) on a layer of hidden 6144, 256 routed experts (gate_up 6144->4096,
down 2048->6144) plus one shared expert, FP8 E4M3 weights with 128x128 fp32
block scales, top-8 routing.  Steps rotate over a stack of 8 independently
seeded layers (about 77.6 GB of FP8 weights resident in HBM) and a pool of
seeded token batches, so every step reads its ~340 MB (M = 1) cold from HBM
(inputs larger than L2; no flush needed).

Headline metric: effective weight bandwidth = unique weight + scale bytes
the step touches / step time, in GB/s, at M = 1; the sweep key adds
M = 1, 2, 4, 8, 16.  `roofline` reports the one kernel of the step (the fused
layer kernel) against the measured HBM copy bandwidth; `e2e` is the same metric
with the per-step host->device copy of x and logits and the device->host
copy of the output inside the timed region (the copies run on their own
streams, double-buffered, overlapping the neighbouring steps' compute; 16
steps at a time replayed from one CUDA graph); `cpu_baseline` is the oracle
(test infrastructure, single-threaded C) on one M = 1 layer.

--impl reference runs the oracle as the reference arm on the host cores
(rank 0 only), on a shape-reduced sample of the same layer sized to finish
within a few minutes.
"""
from __future__ import annotations

import argparse
import json
import os
import statistics
import subprocess
import sys
import threading
import time

ROOT = os.path.dirname(os.path.abspath(__file__))
sys.path.insert(0, ROOT)

import numpy as np  # noqa: E402
import torch  # noqa: E402

import synth  # noqa: E402

METRIC = "FP8 quant+MoE expert GEMM: weight GB/s and % of HBM peak at M=1/4/16"
CFG = synth.MOE_LAYER
H, I, E, TOPK = CFG["H"], CFG["I"], CFG["E"], CFG["top_k"]
GU_BYTES = 2 * I * H + (2 * I // 128) * (H // 128) * 4      # 25,171,968 per expert
DN_BYTES = H * I + (H // 128) * (I // 128) * 4              # 12,585,984 per expert
EXPERT_BYTES = GU_BYTES + DN_BYTES                          # 37,757,952


# ------------------------------------------------------------------ helpers
def dist_setup():
    ws = int(os.environ.get("WORLD_SIZE", "1"))
    rank = int(os.environ.get("RANK", "0"))
    local = int(os.environ.get("LOCAL_RANK", "0"))
    if ws > 1:
        import torch.distributed as dist
        backend = "nccl" if torch.cuda.is_available() else "gloo"
        if backend == "nccl":
            torch.cuda.set_device(local)
        dist.init_process_group(backend)
    elif torch.cuda.is_available():
        torch.cuda.set_device(local)
    return ws, rank, local


def barrier(ws):
    if ws > 1:
        import torch.distributed as dist
        dist.barrier()


def max_over_ranks(v: float, ws: int) -> float:
    """Max of a float over ranks (the job's time is its slowest rank's)."""
    if ws == 1:
        return v
    import torch.distributed as dist
    dev = "cuda" if dist.get_backend() == "nccl" else "cpu"
    t = torch.tensor([v], dtype=torch.float64, device=dev)
    dist.all_reduce(t, op=dist.ReduceOp.MAX)
    return float(t.item())


def sum_over_ranks(v: float, ws: int) -> float:
    if ws == 1:
        return v
    import torch.distributed as dist
    dev = "cuda" if dist.get_backend() == "nccl" else "cpu"
    t = torch.tensor([v], dtype=torch.float64, device=dev)
    dist.all_reduce(t, op=dist.ReduceOp.SUM)
    return float(t.item())


def load_peaks():
    p = os.path.join(ROOT, "MEASURED_PEAKS.json")
    try:
        with open(p) as f:
            d = json.load(f)
        return float(d["hbm_gbs"]), "measured"
    except Exception:
        return 6800.0, "fallback"


class ClockSampler:
    """nvidia-smi clocks / throttle reasons sampled every 50 ms."""
    FIELDS = ("index,clocks.sm,clocks.max.sm,power.draw,clocks_event_reasons.active,"
              "clocks_event_reasons.hw_slowdown,clocks_event_reasons.hw_thermal_slowdown,"
              "clocks_event_reasons.sw_thermal_slowdown,clocks_event_reasons.sw_power_cap")

    def __init__(self, gpu: int):
        self.gpu, self.rows, self.proc = gpu, [], None

    def start(self):
        try:
            self.proc = subprocess.Popen(
                ["nvidia-smi", "-i", str(self.gpu), f"--query-gpu={self.FIELDS}", "--format=csv,noheader,nounits",
                 "-lms", "50"], stdout=subprocess.PIPE, stderr=subprocess.DEVNULL, text=True)
            self.th = threading.Thread(target=self._read, daemon=True)
            self.th.start()
        except Exception:
            self.proc = None

    def _read(self):
        for line in self.proc.stdout:
            self.rows.append((time.time(), [c.strip() for c in line.split(",")]))

    def stop(self):
        if self.proc:
            self.proc.terminate()
            try:
                self.proc.wait(timeout=5)
            except Exception:
                self.proc.kill()

    def summary(self, t0: float, t1: float):
        rows = [r for t, r in self.rows if t0 <= t <= t1] or \
               [r for t, r in self.rows if t0 - 0.5 <= t <= t1 + 0.5]
        if not rows:
            return {"sm_mhz": None, "sm_max_mhz": None, "reasons": ["no samples"]}
        sm = [float(r[1]) for r in rows if r[1].replace(".", "").isdigit()]
        mx = [float(r[2]) for r in rows if r[2].replace(".", "").isdigit()]
        reasons = set()
        names = ["hw_slowdown", "hw_thermal_slowdown", "sw_thermal_slowdown", "sw_power_cap"]
        for r in rows:
            for n, v in zip(names, r[5:9]):
                if v.strip().lower() == "active":
                    reasons.add(n)
        return {"sm_mhz": statistics.median(sm) if sm else None, "sm_max_mhz": max(mx) if mx else None,
                "reasons": sorted(reasons), "samples": len(rows)}


# The sources each layer kernel is built from (a traffic record names its set).
KERNEL_SOURCES = {
    "token": ("moeq_token.cu", "moeq_device.cuh", "moeq_route.cuh", "moeq_internal.h"),
    "mtok": ("moeq_mtok.cu", "moeq_device.cuh", "moeq_route.cuh", "moeq_internal.h"),
    "stream": ("moeq_stream.cuh", "moeq_stream.cu", "moeq_stream_mma.cu", "moeq_device.cuh", "moeq_route.cuh",
               "moeq_internal.h"),
}


def code_hash(texts):
    """Hash of C/CUDA sources with comments and whitespace removed: the
    traffic record follows changes of the code, not of its comments."""
    import hashlib
    import re
    h = hashlib.sha256()
    for src in texts:
        src = re.sub(r"/\*.*?\*/", "", src, flags=re.S)
        src = re.sub(r"//[^\n]*", "", src)
        h.update("".join(src.split()).encode())
    return h.hexdigest()[:16]


def kernel_source_hash(which: str):
    texts = []
    for f in KERNEL_SOURCES[which]:
        with open(os.path.join(ROOT, "bandwidth_bound_fp8_gb300", "csrc", f), encoding="utf-8") as fh:
            texts.append(fh.read())
    return code_hash(texts)


def ncu_traffic(kernel: str, M: int, launch_bytes: float | None = None):
    """DRAM bytes per launch from the committed ncu summary, if it was taken
    on the current kernel source; else None.  A record taken on a smaller
    case (its algorithmic bytes below the launch's) is scaled to the launch
    by the algorithmic bytes: the traffic follows the unique experts
    streamed."""
    p = os.path.join(ROOT, "profiles", "traffic.json")
    try:
        with open(p) as f:
            d = json.load(f)
        e = d[f"{kernel}_m{M}"]
        if e["source_hash"] != kernel_source_hash(e["sources"]):
            return None
        t = float(e["dram_bytes_per_launch"])
        if launch_bytes and e.get("algorithmic_bytes") and abs(launch_bytes - e["algorithmic_bytes"]) > 1:
            t *= launch_bytes / float(e["algorithmic_bytes"])
        return t
    except Exception:
        return None


# ------------------------------------------------------------------ the stack
class Stack:
    """L independently seeded MoE layers resident in HBM."""

    def __init__(self, L: int, seed: int):
        from bandwidth_bound_fp8_gb300 import moeq
        self.L = L
        self.gu_q = torch.empty((L, E + 1, 2 * I, H), dtype=torch.uint8, device="cuda")
        self.gu_s = torch.empty((L, E + 1, 2 * I // 128, H // 128), dtype=torch.float32, device="cuda")
        self.dn_q = torch.empty((L, E + 1, H, I), dtype=torch.uint8, device="cuda")
        self.dn_s = torch.empty((L, E + 1, H // 128, I // 128), dtype=torch.float32, device="cuda")
        buf_gu = torch.empty((2 * I, H), dtype=torch.float32, device="cuda")
        buf_dn = torch.empty((H, I), dtype=torch.float32, device="cuda")
        self.seed = seed
        for l in range(L):
            for e in range(E + 1):
                synth.weight_f32(2 * I, H, synth.expert_seed(seed, l, e, 0), device="cuda", out=buf_gu)
                moeq.moeq_quant_weight(buf_gu[None], self.gu_q[l, e:e + 1], self.gu_s[l, e:e + 1])
                synth.weight_f32(H, I, synth.expert_seed(seed, l, e, 1), device="cuda", out=buf_dn)
                moeq.moeq_quant_weight(buf_dn[None], self.dn_q[l, e:e + 1], self.dn_s[l, e:e + 1])
        torch.cuda.synchronize()

    def f32(self, l, e, which):
        if which == 0:
            return synth.weight_f32(2 * I, H, synth.expert_seed(self.seed, l, e, 0), device="cuda").cpu().numpy()
        return synth.weight_f32(H, I, synth.expert_seed(self.seed, l, e, 1), device="cuda").cpu().numpy()


def make_inputs(n: int, M: int, seed: int):
    xs = torch.empty((n, M, H), dtype=torch.bfloat16, device="cuda")
    lg = torch.empty((n, M, E), dtype=torch.float32, device="cuda")
    for i in range(n):
        xs[i] = synth.activations_bf16(M, H, seed + 2 * i, CFG["n_outlier"], CFG["outlier_scale"], device="cuda")
        lg[i] = synth.logits_f32(M, E, seed + 2 * i + 1, device="cuda")
    return xs, lg


def unique_counts(lg: torch.Tensor, M: int):
    """U (unique experts incl. the shared one) of each input set, read back from
    the library's own route plan."""
    from bandwidth_bound_fp8_gb300 import moeq
    plan = moeq.RoutePlan(M, E, TOPK)
    out = []
    for i in range(lg.shape[0]):
        moeq.moeq_route(lg[i], plan, TOPK)
        out.append(plan.n_uniq.clone())
    torch.cuda.synchronize()
    return [int(t.item()) for t in out]


def make_events(steps, events_every):
    """Per-stage timing events for every events_every-th step, created (by one
    record each) before the timed region so that creating them costs nothing there."""
    recs = []
    if events_every:
        for _ in range(0, steps, events_every):
            ev = [torch.cuda.Event(enable_timing=True) for _ in range(2)]
            for e in ev:
                e.record()
            recs.append(ev)
    torch.cuda.synchronize()
    return recs


def run_steps(stack, xs, lg, M, ws, outs, steps, start, events_every=0, recs=()):
    """Launch `steps` layer forwards, passing recs[i // events_every] to every
    events_every-th step for per-launch timing (events_every = 0: none, so
    consecutive launches stay back to back)."""
    from bandwidth_bound_fp8_gb300 import moeq
    n = xs.shape[0]
    for i in range(steps):
        j = start + i
        l, s = j % stack.L, j % n
        ev = recs[i // events_every] if (events_every and i % events_every == 0) else None
        moeq.moeq_moe_layer(xs[s], lg[s], H, I, E, TOPK, stack.gu_q[l], stack.gu_s[l], stack.dn_q[l],
                            stack.dn_s[l], outs[j % 2], ws, events=ev)


def bench_M(stack, M, steps, warmup, ws_world, seed, isolated=64):
    """Timed region: `steps` layer calls back to back on one stream, events
    only at its two ends.  A step is exactly one launch of the layer kernel,
    so the kernel's average launch duration is the region's time / steps
    (consecutive launches overlap by programmatic dependent launch: the next
    layer streams its shared expert while this one finishes).  After the
    region, `isolated` more launches are timed one by one with events on
    their own stream, which breaks that overlap: the single-launch figure."""
    from bandwidth_bound_fp8_gb300 import moeq
    pool = max(16, min(256, steps + warmup))
    xs, lg = make_inputs(pool, M, seed)
    U = unique_counts(lg, M)
    ws = moeq.Workspace(moeq.moeq_workspace_size(M, H, I, E + 1, TOPK))
    outs = [torch.empty((M, H), dtype=torch.bfloat16, device="cuda") for _ in range(2)]
    run_steps(stack, xs, lg, M, ws, outs, warmup, 0)
    torch.cuda.synchronize()
    barrier(ws_world)
    torch.cuda.synchronize()
    t0e, t1e = torch.cuda.Event(enable_timing=True), torch.cuda.Event(enable_timing=True)
    wall0 = time.time()
    t0e.record()
    run_steps(stack, xs, lg, M, ws, outs, steps, warmup)
    t1e.record()
    torch.cuda.synchronize()
    wall1 = time.time()
    barrier(ws_world)
    ms = t0e.elapsed_time(t1e)
    if moeq.moeq_read_device_status(ws.t, ws.nbytes) != 0:
        raise RuntimeError("device status word set during the bench")
    byts = sum(U[(warmup + i) % pool] * EXPERT_BYTES for i in range(steps))
    recs = make_events(isolated, 1)
    run_steps(stack, xs, lg, M, ws, outs, isolated, warmup + steps, 1, recs)
    torch.cuda.synchronize()
    iso = [ev[0].elapsed_time(ev[1]) for ev in recs]
    iso_bytes = [U[(warmup + steps + k) % pool] * EXPERT_BYTES for k in range(isolated)]
    return dict(ms=ms, bytes=byts, steps=steps, U_mean=float(np.mean([U[(warmup + i) % pool] for i in range(steps)])),
                kernel_ms=ms / steps, kernel_bytes=byts / steps,
                isolated_ms=float(np.median(iso)) if iso else None,
                isolated_bytes=float(np.mean(iso_bytes)) if iso else None, wall=(wall0, wall1),
                xs=xs, lg=lg, U=U, ws=ws)


def bench_stack(stack, M, calls, seed, peak):
    """The L-layer stack through moeq_moe_stack: one call = one decode step
    through every layer (one CUDA graph launch; the first call captures it).
    Layer l routes its own seeded logits; x is the previous layer's output.
    Timed: `calls` calls back to back, events at the region's two ends.
    Every call reads each layer's experts cold (the stack's weights are far
    larger than L2)."""
    from bandwidth_bound_fp8_gb300 import moeq
    L = stack.L
    x = synth.activations_bf16(M, H, seed, CFG["n_outlier"], CFG["outlier_scale"], device="cuda")
    logits = torch.stack([synth.logits_f32(M, E, seed + 1 + l, device="cuda") for l in range(L)])
    out = torch.empty((L, M, H), dtype=torch.bfloat16, device="cuda")
    ws = moeq.Workspace(moeq.moeq_stack_workspace_size(L, M, H, I, E + 1, TOPK))
    w = ([stack.gu_q[l] for l in range(L)], [stack.gu_s[l] for l in range(L)],
         [stack.dn_q[l] for l in range(L)], [stack.dn_s[l] for l in range(L)])
    for _ in range(3):
        moeq.moeq_moe_stack(x, logits, H, I, E, TOPK, *w, out, ws)
    torch.cuda.synchronize()
    U = [int(moeq.moeq_stack_plan(ws, L, M, H, I, E, TOPK, l).n_uniq.item()) for l in range(L)]
    a, e = torch.cuda.Event(enable_timing=True), torch.cuda.Event(enable_timing=True)
    a.record()
    for _ in range(calls):
        moeq.moeq_moe_stack(x, logits, H, I, E, TOPK, *w, out, ws)
    e.record()
    torch.cuda.synchronize()
    if moeq.moeq_read_device_status(ws.t, ws.nbytes) != 0:
        raise RuntimeError("device status word set during the stack bench")
    ms = a.elapsed_time(e)
    byts = calls * sum(U) * EXPERT_BYTES
    gbs = byts / (ms * 1e-3) / 1e9
    return {"layers": L, "calls": calls, "us_per_layer": round(ms * 1e3 / (calls * L), 2),
            "us_per_step": round(ms * 1e3 / calls, 1), "weight_GBps": round(gbs, 1),
            "frac_of_measured_hbm": round(gbs / peak, 4), "frac_of_8TBps": round(gbs / 8000, 4),
            "U_per_layer": U}


def bench_e2e(stack, M, steps, seed):
    """Same metric through the public call, with host<->device copies per step:
    each step copies its x and logits from pinned host memory and reads its
    output back.  The copies run on their own streams, double-buffered, so that
    step j+1's inputs and step j-1's output move while step j computes; the
    timed region holds every step's copies.  Sixteen steps (one per input set,
    two rounds of the 8 layers) are captured once in a CUDA graph and replayed,
    so the host's per-step stream, event and copy calls leave the timed
    region; if capture fails the same steps run eagerly and `mode` says so."""
    from bandwidth_bound_fp8_gb300 import moeq
    pool = 16
    xs, lg = make_inputs(pool, M, seed)
    U = unique_counts(lg, M)
    hx = xs.cpu().pin_memory()
    hl = lg.cpu().pin_memory()
    hout = torch.empty((2, M, H), dtype=torch.bfloat16).pin_memory()
    dx = [torch.empty((M, H), dtype=torch.bfloat16, device="cuda") for _ in range(2)]
    dl = [torch.empty((M, E), dtype=torch.float32, device="cuda") for _ in range(2)]
    dout = [torch.empty((M, H), dtype=torch.bfloat16, device="cuda") for _ in range(2)]
    ws = moeq.Workspace(moeq.moeq_workspace_size(M, H, I, E + 1, TOPK))
    up, down = torch.cuda.Stream(), torch.cuda.Stream()
    ev_in = [torch.cuda.Event() for _ in range(2)]     # inputs of slot b landed
    ev_done = [torch.cuda.Event() for _ in range(2)]   # the layer that used slot b finished
    ev_out = [torch.cuda.Event() for _ in range(2)]    # slot b's output read back

    def sequence(comp):
        """Steps 0 .. pool-1 on stream comp; the copy streams fork from and
        join back into comp, so the sequence is one unit of stream order."""
        up.wait_stream(comp)
        down.wait_stream(comp)
        for j in range(pool):
            b, l = j % 2, j % stack.L
            with torch.cuda.stream(up):
                if j >= 2:
                    up.wait_event(ev_done[b])          # slot b's previous inputs are consumed
                dx[b].copy_(hx[j], non_blocking=True)
                dl[b].copy_(hl[j], non_blocking=True)
                ev_in[b].record(up)
            comp.wait_event(ev_in[b])
            if j >= 2:
                comp.wait_event(ev_out[b])             # slot b's previous output is read back
            moeq.moeq_moe_layer(dx[b], dl[b], H, I, E, TOPK, stack.gu_q[l], stack.gu_s[l], stack.dn_q[l],
                                stack.dn_s[l], dout[b], ws, stream=comp)
            ev_done[b].record(comp)
            with torch.cuda.stream(down):
                down.wait_event(ev_done[b])
                hout[b].copy_(dout[b], non_blocking=True)
                ev_out[b].record(down)
        comp.wait_stream(up)
        comp.wait_stream(down)                         # the last output is on the host

    # the first calls on the capture's stream happen outside the capture
    side = torch.cuda.Stream()
    side.wait_stream(torch.cuda.current_stream())
    with torch.cuda.stream(side):
        sequence(side)
    torch.cuda.current_stream().wait_stream(side)
    torch.cuda.synchronize()
    graph, mode = None, "cuda_graph"
    try:
        g = torch.cuda.CUDAGraph()
        with torch.cuda.graph(g):
            sequence(torch.cuda.current_stream())
        torch.cuda.synchronize()
        graph = g
    except Exception as ex:   # noqa: BLE001 -- reported, the eager steps are timed instead
        torch.cuda.synchronize()
        mode = f"eager (graph capture failed: {type(ex).__name__})"
    comp = torch.cuda.current_stream()

    def run_once():
        if graph is not None:
            graph.replay()
        else:
            sequence(comp)

    for _ in range(3):
        run_once()
    torch.cuda.synchronize()
    reps = max(1, steps // pool)
    a, e = torch.cuda.Event(enable_timing=True), torch.cuda.Event(enable_timing=True)
    a.record(comp)
    for _ in range(reps):
        run_once()
    e.record(comp)
    torch.cuda.synchronize()
    ms = a.elapsed_time(e)
    n = reps * pool
    byts = reps * sum(U[j] * EXPERT_BYTES for j in range(pool))
    h2d = M * H * 2 + M * E * 4
    d2h = M * H * 2
    return dict(value=byts / (ms * 1e-3) / 1e9, h2d=h2d, d2h=d2h, ms_per_step=ms / n, mode=mode)


def bench_e2e_batch(stack, M, steps, seed):
    """The e2e metric with the copies batched per 16 steps: one host->device
    copy of the 16 steps' inputs (each step's x and logits packed one after
    another in one pinned buffer), the 16 layer calls, one device->host copy
    of their 16 outputs, captured in one CUDA graph and replayed.  Every
    step's inputs and output still cross the host link inside the timed
    region.  With per-step copies (bench_e2e) every layer kernel gains graph
    edges to copy nodes, and consecutive layers no longer overlap by
    programmatic dependent launch; here the 16 launches follow one another
    directly."""
    from bandwidth_bound_fp8_gb300 import moeq
    pool = 16
    xs, lg = make_inputs(pool, M, seed)
    U = unique_counts(lg, M)
    xb, lb = M * H * 2, M * E * 4
    sb = xb + lb                                   # a step's input bytes (16-byte multiple)
    hpack = torch.empty((pool * sb,), dtype=torch.uint8)
    for j in range(pool):
        hpack[j * sb: j * sb + xb] = xs[j].cpu().view(torch.uint8).reshape(-1)
        hpack[j * sb + xb: (j + 1) * sb] = lg[j].cpu().view(torch.uint8).reshape(-1)
    hpack = hpack.pin_memory()
    dpack = torch.empty((pool * sb,), dtype=torch.uint8, device="cuda")
    px = [dpack[j * sb: j * sb + xb].view(torch.bfloat16).view(M, H) for j in range(pool)]
    pl = [dpack[j * sb + xb: (j + 1) * sb].view(torch.float32).view(M, E) for j in range(pool)]
    dout = torch.empty((pool, M, H), dtype=torch.bfloat16, device="cuda")
    hout = torch.empty((pool, M, H), dtype=torch.bfloat16).pin_memory()
    ws = moeq.Workspace(moeq.moeq_workspace_size(M, H, I, E + 1, TOPK))

    def sequence(comp):
        dpack.copy_(hpack, non_blocking=True)
        for j in range(pool):
            l = j % stack.L
            moeq.moeq_moe_layer(px[j], pl[j], H, I, E, TOPK, stack.gu_q[l], stack.gu_s[l], stack.dn_q[l],
                                stack.dn_s[l], dout[j], ws, stream=comp)
        hout.copy_(dout, non_blocking=True)

    side = torch.cuda.Stream()
    side.wait_stream(torch.cuda.current_stream())
    with torch.cuda.stream(side):
        sequence(side)
    torch.cuda.current_stream().wait_stream(side)
    torch.cuda.synchronize()
    graph, mode = None, "cuda_graph: one copy of 16 steps' inputs, 16 layer calls, one copy of 16 outputs"
    try:
        g = torch.cuda.CUDAGraph()
        with torch.cuda.graph(g):
            sequence(torch.cuda.current_stream())
        torch.cuda.synchronize()
        graph = g
    except Exception as ex:   # noqa: BLE001 -- reported, the eager steps are timed instead
        torch.cuda.synchronize()
        mode = f"eager (graph capture failed: {type(ex).__name__})"
    comp = torch.cuda.current_stream()
    run_once = graph.replay if graph is not None else (lambda: sequence(comp))
    for _ in range(3):
        run_once()
    torch.cuda.synchronize()
    reps = max(1, steps // pool)
    a, e = torch.cuda.Event(enable_timing=True), torch.cuda.Event(enable_timing=True)
    a.record(comp)
    for _ in range(reps):
        run_once()
    e.record(comp)
    torch.cuda.synchronize()
    ms = a.elapsed_time(e)
    n = reps * pool
    byts = reps * sum(U[j] * EXPERT_BYTES for j in range(pool))
    return dict(value=byts / (ms * 1e-3) / 1e9, h2d=sb, d2h=M * H * 2, ms_per_step=ms / n, mode=mode)


def cpu_baseline(stack, M, seed, budget_s=10.0):
    """The oracle (single-threaded C) on full M = 1 layers of layer 0 of the
    stack, repeated until about budget_s seconds of CPU work."""
    import concurrent.futures as cf

    import oracle
    xs, lg = make_inputs(1, M, seed)
    x_bits = xs[0].view(torch.uint16).cpu().numpy()
    logits = lg[0].cpu().numpy()
    r = oracle.route(logits, TOPK)
    f32 = {int(e): (stack.f32(0, int(e), 0), stack.f32(0, int(e), 1)) for e in r.uniq}
    with cf.ThreadPoolExecutor(max_workers=min(16, os.cpu_count() or 1)) as ex:
        fut = {e: (ex.submit(oracle.quant_weight, a), ex.submit(oracle.quant_weight, b)) for e, (a, b) in f32.items()}
        experts = {e: (*fa.result(), *fb.result()) for e, (fa, fb) in fut.items()}
    n, t_total = 0, 0.0
    while t_total < budget_s or n < 1:
        t = time.perf_counter()
        oracle.moe_layer(x_bits, logits, TOPK, experts, H, I)
        t_total += time.perf_counter() - t
        n += 1
    byts = len(r.uniq) * EXPERT_BYTES
    return {"value": round(byts * n / t_total / 1e9, 4), "unit": "GB/s", "cores": 1, "kind": "oracle",
            "sample": f"{n} full M={M} layer forwards (route, quant, {len(r.uniq)} experts' gate_up+SwiGLU+down, "
                      f"combine) in the single-threaded C oracle, fp64 accumulation; host has {os.cpu_count()} cores",
            "seconds": round(t_total, 2)}


# ------------------------------------------------------------------ dense configs and the gate_up ladder
L2_BYTES = 129 * 1024 * 1024


def time_scrubbed(fn, reps: int, warmup: int):
    """Median / p10 / p90 ms of fn() over `reps` CUDA-event timings, each
    after a write of more than twice L2 (outside the timed region), so the
    weights come from HBM every time."""
    scrub = torch.empty(2 * L2_BYTES // 4 + 1024, dtype=torch.float32, device="cuda")
    for _ in range(warmup):
        fn()
    ts = []
    for _ in range(reps):
        scrub.zero_()
        e0, e1 = torch.cuda.Event(enable_timing=True), torch.cuda.Event(enable_timing=True)
        e0.record()
        fn()
        e1.record()
        torch.cuda.synchronize()
        ts.append(e0.elapsed_time(e1))
    ts.sort()
    return ts[len(ts) // 2], ts[len(ts) // 10], ts[(len(ts) * 9) // 10]


def _line(name, byts, t, peak, oracle_s=None):
    med, p10, p90 = t
    d = {"workload": name, "us": round(med * 1e3, 2), "us_p10": round(p10 * 1e3, 2), "us_p90": round(p90 * 1e3, 2),
         "weight_bytes": byts, "weight_GBps": round(byts / (med * 1e-3) / 1e9, 1),
         "frac_of_measured_hbm": round(byts / (med * 1e-3) / 1e9 / peak, 4),
         "frac_of_8TBps": round(byts / (med * 1e-3) / 1e9 / 8000, 4), "l2": "scrubbed (> 2x L2 written) before each rep"}
    if oracle_s is not None:
        d["oracle_ms_1core"] = round(oracle_s * 1e3, 2)
    return d


def bench_dense(peak, reps=50, with_oracle=True):
    """The two dense configurations at M = 1, each call timed alone:
    C0 the projection K 2048 -> N 4096 (one moeq_expert_gemm_down call, x bf16
    in, y fp32 out); C1 the FFN hidden 6144 / intermediate 12288 through
    moeq_dense_ffn (one kernel), and through the three separate calls (gate_up
    + SwiGLU, down, the bf16 cast through moeq_combine).  Beside each, the
    oracle (one core) on the same inputs."""
    from bandwidth_bound_fp8_gb300 import moeq
    out = {}
    # C0
    c = synth.DENSE_PROJ
    K, N = c["K"], c["N"]
    wq = torch.empty((1, N, K), dtype=torch.uint8, device="cuda")
    ws_ = torch.empty((1, N // 128, K // 128), dtype=torch.float32, device="cuda")
    w32 = synth.weight_f32(N, K, synth.expert_seed(c["seed"], 0, 0, 1), device="cuda")
    moeq.moeq_quant_weight(w32[None], wq, ws_)
    x = synth.activations_bf16(1, K, c["seed"], c["n_outlier"], c["outlier_scale"], device="cuda")
    one = lambda v: torch.tensor(v, dtype=torch.int32, device="cuda")
    uq, of, nu = one([0]), one([0, 1]), one([1])
    y = torch.empty((1, N), dtype=torch.float32, device="cuda")
    wsp = moeq.Workspace(moeq.moeq_gemm_workspace_size(N, K, 1, 1, 0))
    torch.cuda.synchronize()
    t = time_scrubbed(lambda: moeq.moeq_expert_gemm_down(x, K, N, wq, ws_, 1, uq, of, nu, 1, 1, y, wsp), reps, 5)
    osec = None
    if with_oracle:
        import oracle
        qw, sw = oracle.quant_weight(w32.cpu().numpy())
        xb = x.view(torch.uint16).cpu().numpy()
        t0 = time.perf_counter()
        qa, sa = oracle.quant_act(xb)
        oracle.gemm(qa, sa, qw, sw)
        osec = time.perf_counter() - t0
    out["C0"] = _line(c["name"], N * K + (N // 128) * (K // 128) * 4, t, peak, osec)
    del wq, ws_, w32
    # C1
    c = synth.DENSE_FFN
    Hh, Ii = c["H"], c["I"]
    gq = torch.empty((1, 2 * Ii, Hh), dtype=torch.uint8, device="cuda")
    gs = torch.empty((1, 2 * Ii // 128, Hh // 128), dtype=torch.float32, device="cuda")
    dq = torch.empty((1, Hh, Ii), dtype=torch.uint8, device="cuda")
    dsc = torch.empty((1, Hh // 128, Ii // 128), dtype=torch.float32, device="cuda")
    g32 = synth.weight_f32(2 * Ii, Hh, synth.expert_seed(c["seed"], 0, 0, 0), device="cuda")
    moeq.moeq_quant_weight(g32[None], gq, gs)
    d32 = synth.weight_f32(Hh, Ii, synth.expert_seed(c["seed"], 0, 0, 1), device="cuda")
    moeq.moeq_quant_weight(d32[None], dq, dsc)
    x = synth.activations_bf16(1, Hh, c["seed"], c["n_outlier"], c["outlier_scale"], device="cuda")
    pt = one([0])
    h = torch.empty((1, Ii), dtype=torch.float32, device="cuda")
    y = torch.empty((1, Hh), dtype=torch.float32, device="cuda")
    o16 = torch.empty((1, Hh), dtype=torch.bfloat16, device="cuda")
    wgu = moeq.Workspace(moeq.moeq_gemm_workspace_size(2 * Ii, Hh, 1, 1, 1))
    wdn = moeq.Workspace(moeq.moeq_gemm_workspace_size(Hh, Ii, 1, 1, 0))
    plan = moeq.RoutePlan(1, 1, 1)
    plan.pair_of.view(-1)[0] = 0
    torch.cuda.synchronize()

    def ffn():
        moeq.moeq_expert_gemm_gateup_swiglu(x, Hh, Ii, gq, gs, 1, uq, of, pt, nu, 1, 1, h, wgu)
        moeq.moeq_expert_gemm_down(h, Ii, Hh, dq, dsc, 1, uq, of, nu, 1, 1, y, wdn)
        moeq.moeq_combine(y, Hh, plan, 1, 0, o16)

    t_calls = time_scrubbed(ffn, reps, 5)
    wff = moeq.Workspace(moeq.moeq_dense_ffn_workspace_size(1, Hh, Ii))
    torch.cuda.synchronize()
    t = time_scrubbed(lambda: moeq.moeq_dense_ffn(x, Hh, Ii, gq, gs, dq, dsc, o16, wff), reps, 5)
    osec = None
    if with_oracle:
        import oracle
        qg, sg = oracle.quant_weight(g32.cpu().numpy())
        qd, sd = oracle.quant_weight(d32.cpu().numpy())
        xb = x.view(torch.uint16).cpu().numpy()
        t0 = time.perf_counter()
        qa, sa = oracle.quant_act(xb)
        gy = oracle.gemm(qa, sa, qg, sg, with_T=False)
        hh = oracle.swiglu_vec(gy[:, :Ii], gy[:, Ii:])
        qh, sh = oracle.quant_act(hh)
        yy = oracle.gemm(qh, sh, qd, sd, with_T=False)
        [oracle.f64_to_bf16_bits(v) for v in yy[0]]
        osec = time.perf_counter() - t0
    byts = 2 * Ii * Hh + (2 * Ii // 128) * (Hh // 128) * 4 + Hh * Ii + (Hh // 128) * (Ii // 128) * 4
    out["C1"] = _line(c["name"], byts, t, peak, osec)
    out["C1"]["call"] = "moeq_dense_ffn (one kernel)"
    out["C1_gemm_calls"] = _line(c["name"], byts, t_calls, peak)
    out["C1_gemm_calls"]["call"] = "moeq_expert_gemm_gateup_swiglu + moeq_expert_gemm_down + moeq_combine"
    out["C0"]["call"] = "moeq_expert_gemm_down"
    return out


LM_HEAD_K, LM_HEAD_N = 6144, 151552


def lm_head_calls():
    """The LM head's seeded FP8 weight (N x K, quantised from fp32 draws in
    slabs of 4096 rows) and, for M = 1 and 4, a closure making one
    moeq_expert_gemm_down call over it: yields (M, call, workspace)."""
    from bandwidth_bound_fp8_gb300 import moeq
    K, N = LM_HEAD_K, LM_HEAD_N
    wq = torch.empty((1, N, K), dtype=torch.uint8, device="cuda")
    ws_ = torch.empty((1, N // 128, K // 128), dtype=torch.float32, device="cuda")
    rows = 4096   # whole 128-row blocks per slab; bounds the fp32 draw
    for r0 in range(0, N, rows):
        r1 = min(N, r0 + rows)
        w32 = synth.weight_f32(r1 - r0, K, synth.expert_seed(3100, 0, r0 // rows, 1), device="cuda")
        moeq.moeq_quant_weight(w32[None], wq[:, r0:r1], ws_[:, r0 // 128:r1 // 128])
        del w32
    one = lambda v: torch.tensor(v, dtype=torch.int32, device="cuda")
    for M in (1, 4):
        x = synth.activations_bf16(M, K, 3101 + M, 61, 30.0, device="cuda")
        uq, of, nu = one([0]), one([0, M]), one([1])
        y = torch.empty((M, N), dtype=torch.float32, device="cuda")
        wsp = moeq.Workspace(moeq.moeq_gemm_workspace_size(N, K, M, 1, 0))
        yield M, (lambda x=x, uq=uq, of=of, nu=nu, M=M, y=y, wsp=wsp:
                  moeq.moeq_expert_gemm_down(x, K, N, wq, ws_, 1, uq, of, nu, 1, M, y, wsp)), wsp


def bench_lm_head(peak, reps=30):
    """An FP8 LM head (GLM-5.2 x10 §8b), the vocabulary projection
    N = 151,552 x K = 6144 (931 MB of E4M3 codes), through the down GEMM call
    with one expert and the trivial plan, at 1 and 4 tokens; each call timed
    alone (the weight is larger than L2 and L2 is scrubbed between calls).
    N is above the multi-token kernel's 6144, so the persistent engine serves
    it, on tcgen05 at both row counts."""
    from bandwidth_bound_fp8_gb300 import moeq
    K, N = LM_HEAD_K, LM_HEAD_N
    out = {}
    for M, call, wsp in lm_head_calls():
        torch.cuda.synchronize()
        t = time_scrubbed(call, reps, 5)
        if moeq.moeq_read_device_status(wsp.t, wsp.nbytes) != 0:
            raise RuntimeError(f"lm_head M={M}: device status word set")
        out[f"M{M}"] = _line(f"lm_head_m{M}_k{K}_n{N}", N * K + (N // 128) * (K // 128) * 4, t, peak)
        out[f"M{M}"]["call"] = "moeq_expert_gemm_down (one expert; the persistent engine, tcgen05)"
    return out


def gate_up_ladder(peak, variants=("split_all_sms", "quant_launch_first"), reps=30):
    """The one-token gate_up of a layer (the shared expert and 8 routed
    experts: 226.5 MB) in the variants the GLM-5.2 x10 page measured (§1):
    split over every SM (this library's call); the activations' quantisation
    as a launch of its own ahead of the GEMM (which still quantises its input
    itself); and, in a child process with MOEQ_GRID_LIMIT=4, four CTAs."""
    from bandwidth_bound_fp8_gb300 import moeq
    n_exp = 9
    gq = torch.empty((n_exp, 2 * I, H), dtype=torch.uint8, device="cuda")
    gs = torch.empty((n_exp, 2 * I // 128, H // 128), dtype=torch.float32, device="cuda")
    for e in range(n_exp):
        w = synth.weight_f32(2 * I, H, synth.expert_seed(CFG["seed"], 9, e, 0), device="cuda")
        moeq.moeq_quant_weight(w[None], gq[e:e + 1], gs[e:e + 1])
    del w
    x = synth.activations_bf16(1, H, 3, CFG["n_outlier"], CFG["outlier_scale"], device="cuda")
    t = lambda v: torch.tensor(v, dtype=torch.int32, device="cuda")
    uq, of, pt, nu = t(list(range(n_exp))), t(list(range(n_exp + 1))), t([0] * n_exp), t([n_exp])
    h = torch.empty((n_exp, I), dtype=torch.float32, device="cuda")
    qx = torch.empty((1, H), dtype=torch.uint8, device="cuda")
    sx = torch.empty((1, H // 128), dtype=torch.float32, device="cuda")
    ws = moeq.Workspace(moeq.moeq_gemm_workspace_size(2 * I, H, 1, n_exp, 1))
    torch.cuda.synchronize()
    gemm = lambda: moeq.moeq_expert_gemm_gateup_swiglu(x, H, I, gq, gs, n_exp, uq, of, pt, nu, n_exp, n_exp, h, ws)
    byts = n_exp * GU_BYTES
    out = {}
    for v in variants:
        if v == "quant_launch_first":
            fn = lambda: (moeq.moeq_quant_act(x, qx, sx), gemm())
        else:
            fn = gemm
        out[v] = _line(f"gate_up_m1_9experts_h{H}_i{I} ({v})", byts, time_scrubbed(fn, reps, 3), peak)
    return out


def gate_up_ladder_child(peak):
    """The ladder's four-CTA leg, in a child process (the grid limit is read
    once per process)."""
    env = dict(os.environ, MOEQ_GRID_LIMIT="4")
    r = subprocess.run([sys.executable, os.path.abspath(__file__), "--ladder-child"], env=env,
                       capture_output=True, text=True, timeout=600)
    if r.returncode != 0:
        return {"error": (r.stderr or r.stdout)[-300:]}
    return json.loads(r.stdout.strip().splitlines()[-1])


# ------------------------------------------------------------------ reference arm
def reference_arm(args, ws, rank):
    """The oracle as the reference arm, on a shape-reduced sample of the layer:
    same routing (256 experts, top-8 + shared, M tokens) and block structure,
    hidden Hs and intermediate Is cut to fit (steps + warmup) in ~150 s."""
    import oracle
    if rank != 0:
        return
    M = args.M
    budget = 150.0
    total = args.steps + args.warmup
    ladder = [(6144, 2048), (6144, 512), (3072, 256), (2048, 128), (1024, 128), (512, 128), (256, 128), (128, 128)]
    # rough oracle cost: ~1.3 ns per weight byte per pair + fixed overhead
    pairs = M * TOPK + M
    for Hs, Is in ladder:
        per = pairs * 3 * Hs * Is * 1.5e-9 + 2e-4
        if per * total <= budget:
            break
    g = torch.Generator().manual_seed(4242)
    experts = {}
    xs = [synth.activations_bf16(M, Hs, 900 + i, max(1, round(0.01 * Hs)), 30.0) for i in range(4)]
    lgs = [synth.logits_f32(M, E, 950 + i) for i in range(4)]
    need = set()
    for lg in lgs:
        need |= set(int(e) for e in oracle.route(lg.numpy(), TOPK).uniq)
    for e in need:
        a = synth.weight_f32(2 * Is, Hs, synth.expert_seed(77, 0, e, 0))
        b = synth.weight_f32(Hs, Is, synth.expert_seed(77, 0, e, 1))
        experts[e] = (*oracle.quant_weight(a.numpy()), *oracle.quant_weight(b.numpy()))
    del g
    ebytes = 3 * Hs * Is + (2 * Is // 128) * (Hs // 128) * 4 + (Hs // 128) * (Is // 128) * 4
    for i in range(args.warmup):
        oracle.moe_layer(xs[i % 4].view(torch.uint16).numpy(), lgs[i % 4].numpy(), TOPK, experts, Hs, Is)
    t0 = time.perf_counter()
    byts = 0
    for i in range(args.steps):
        r = oracle.moe_layer(xs[i % 4].view(torch.uint16).numpy(), lgs[i % 4].numpy(), TOPK, experts, Hs, Is)
        byts += r.route.n_uniq * ebytes
    dt = time.perf_counter() - t0
    v = byts / dt / 1e9
    full = (Hs, Is) == (H, I)
    if full:
        sample = (f"oracle MoE layer at M={M}, 256 experts top-{TOPK} + shared, the full layer shape (hidden {Hs}, "
                  f"intermediate {Is}); {total} steps fit ~{budget:.0f} s")
    else:
        sample = (f"oracle MoE layer at M={M}, 256 experts top-{TOPK} + shared, shape reduced to hidden {Hs}, "
                  f"intermediate {Is} so that {total} steps fit ~{budget:.0f} s")
    workload = f"moe_layer_m{M}_h6144_i2048_e256_top8_shared1" + ("" if full else f" (sample: h{Hs}_i{Is})")
    line = {"impl": "reference", "metric": METRIC, "value": round(v, 6), "unit": "GB/s", "n_gpus": args.gpus,
            "steps": args.steps, "warmup": args.warmup, "ms_per_step": round(dt / args.steps * 1e3, 4),
            "higher_is_better": True, "scaling": "weak", "vs_baseline": None, "dtype": "f64", "data": "synthetic",
            "config": {"workload": workload, "M": M},
            "cpu_baseline": {"value": round(v, 6), "unit": "GB/s", "cores": 1, "kind": "oracle", "sample": sample},
            "e2e": {"value": round(v, 6), "unit": "GB/s", "h2d_bytes_per_step": 0, "d2h_bytes_per_step": 0}}
    print(json.dumps(line), flush=True)


# ------------------------------------------------------------------ profiling case
def profile_case(M: int, reps: int, Er: int = 8):
    """A small launch for ncu captures: the layer kernel with Er routed experts
    and top-8.  Er = 8: a one-token launch does exactly the full layer's work
    (8 routed + the shared expert, ~340 MB) on ~350 MB of weights.  Er = 64
    (2.45 GB of weights): several tokens' picks spread over the experts as in
    the full layer (4 tokens ~27 unique routed experts, 16 tokens ~56), most
    of them serving one or two tokens."""
    from bandwidth_bound_fp8_gb300 import build as b
    b.build()
    from bandwidth_bound_fp8_gb300 import moeq
    gq = torch.empty((Er + 1, 2 * I, H), dtype=torch.uint8, device="cuda")
    gs = torch.empty((Er + 1, 2 * I // 128, H // 128), dtype=torch.float32, device="cuda")
    dq = torch.empty((Er + 1, H, I), dtype=torch.uint8, device="cuda")
    ds = torch.empty((Er + 1, H // 128, I // 128), dtype=torch.float32, device="cuda")
    for e in range(Er + 1):
        w = synth.weight_f32(2 * I, H, synth.expert_seed(CFG["seed"], 0, e, 0), device="cuda")
        moeq.moeq_quant_weight(w[None], gq[e:e + 1], gs[e:e + 1])
        w = synth.weight_f32(H, I, synth.expert_seed(CFG["seed"], 0, e, 1), device="cuda")
        moeq.moeq_quant_weight(w[None], dq[e:e + 1], ds[e:e + 1])
    del w
    x = synth.activations_bf16(M, H, 3, CFG["n_outlier"], CFG["outlier_scale"], device="cuda")
    lg = synth.logits_f32(M, Er, 4, device="cuda")
    out = torch.empty((M, H), dtype=torch.bfloat16, device="cuda")
    ws = moeq.Workspace(moeq.moeq_workspace_size(M, H, I, Er + 1, TOPK))
    plan = moeq.RoutePlan(M, Er, TOPK)
    for _ in range(reps):
        moeq.moeq_moe_layer(x, lg, H, I, Er, TOPK, gq, gs, dq, ds, out, ws, plan=plan)
    torch.cuda.synchronize()
    if moeq.moeq_read_device_status(ws.t, ws.nbytes) != 0:
        raise RuntimeError("device status word set")
    U = int(plan.n_uniq.item())
    print(json.dumps({"profile_case": f"moe_layer_m{M}_h{H}_i{I}_e{Er}_top{TOPK}_shared1", "launches": reps,
                      "unique_experts": U, "algorithmic_bytes": U * EXPERT_BYTES}))


def profile_lm_head(reps: int):
    """Small launch list for ncu captures of the LM head: `reps` calls at
    one token, then `reps` at four (moeq_expert_gemm_down on the persistent
    engine's tcgen05 path, one stream_kernel launch each), each after more
    than L2 has been written, so that the 931 MB weight comes from HBM."""
    from bandwidth_bound_fp8_gb300 import build as b
    b.build()
    from bandwidth_bound_fp8_gb300 import moeq
    scrub = torch.empty(2 * L2_BYTES // 4 + 1024, dtype=torch.float32, device="cuda")
    for M, call, wsp in lm_head_calls():
        for _ in range(reps):
            scrub.zero_()
            call()
        torch.cuda.synchronize()
        if moeq.moeq_read_device_status(wsp.t, wsp.nbytes) != 0:
            raise RuntimeError(f"lm_head M={M}: device status word set")
    print(json.dumps({"profile_lm_head": f"lm_head_k{LM_HEAD_K}_n{LM_HEAD_N}", "M": [1, 4], "launches": reps}))


def profile_dense(reps: int):
    """Small launches for ncu captures of the dense configurations: `reps`
    calls each of the projection K 2048 -> N 4096 (moeq_expert_gemm_down:
    mtok_kernel<2>) and of the FFN hidden 6144 / intermediate 12288
    (moeq_dense_ffn: mtok_kernel<3>), on their seeded weights and inputs,
    with more than L2 written before each call so that the weights come from
    HBM."""
    from bandwidth_bound_fp8_gb300 import build as b
    b.build()
    from bandwidth_bound_fp8_gb300 import moeq
    scrub = torch.empty(2 * L2_BYTES // 4 + 1024, dtype=torch.float32, device="cuda")
    c = synth.DENSE_PROJ
    K, N = c["K"], c["N"]
    wq = torch.empty((1, N, K), dtype=torch.uint8, device="cuda")
    ws_ = torch.empty((1, N // 128, K // 128), dtype=torch.float32, device="cuda")
    moeq.moeq_quant_weight(synth.weight_f32(N, K, synth.expert_seed(c["seed"], 0, 0, 1), device="cuda")[None], wq, ws_)
    x = synth.activations_bf16(1, K, c["seed"], c["n_outlier"], c["outlier_scale"], device="cuda")
    one = lambda v: torch.tensor(v, dtype=torch.int32, device="cuda")
    uq, of, nu = one([0]), one([0, 1]), one([1])
    y = torch.empty((1, N), dtype=torch.float32, device="cuda")
    wsp = moeq.Workspace(moeq.moeq_gemm_workspace_size(N, K, 1, 1, 0))
    for _ in range(reps):
        scrub.zero_()
        moeq.moeq_expert_gemm_down(x, K, N, wq, ws_, 1, uq, of, nu, 1, 1, y, wsp)
    torch.cuda.synchronize()
    if moeq.moeq_read_device_status(wsp.t, wsp.nbytes) != 0:
        raise RuntimeError("device status word set")
    del wq, ws_
    c = synth.DENSE_FFN
    Hh, Ii = c["H"], c["I"]
    gq = torch.empty((1, 2 * Ii, Hh), dtype=torch.uint8, device="cuda")
    gs = torch.empty((1, 2 * Ii // 128, Hh // 128), dtype=torch.float32, device="cuda")
    dq = torch.empty((1, Hh, Ii), dtype=torch.uint8, device="cuda")
    dsc = torch.empty((1, Hh // 128, Ii // 128), dtype=torch.float32, device="cuda")
    moeq.moeq_quant_weight(synth.weight_f32(2 * Ii, Hh, synth.expert_seed(c["seed"], 0, 0, 0), device="cuda")[None],
                           gq, gs)
    moeq.moeq_quant_weight(synth.weight_f32(Hh, Ii, synth.expert_seed(c["seed"], 0, 0, 1), device="cuda")[None],
                           dq, dsc)
    x = synth.activations_bf16(1, Hh, c["seed"], c["n_outlier"], c["outlier_scale"], device="cuda")
    out = torch.empty((1, Hh), dtype=torch.bfloat16, device="cuda")
    wsd = moeq.Workspace(moeq.moeq_dense_ffn_workspace_size(1, Hh, Ii))
    for _ in range(reps):
        scrub.zero_()
        moeq.moeq_dense_ffn(x, Hh, Ii, gq, gs, dq, dsc, out, wsd)
    torch.cuda.synchronize()
    if moeq.moeq_read_device_status(wsd.t, wsd.nbytes) != 0:
        raise RuntimeError("device status word set")
    print(json.dumps({"profile_dense": ["dense_proj_m1_k2048_n4096", "dense_ffn_m1_h6144_i12288"], "launches": reps,
                      "algorithmic_bytes": [N * K + (N // 128) * (K // 128) * 4,
                                            3 * Hh * Ii + 3 * (Hh // 128) * (Ii // 128) * 4]}))


# ------------------------------------------------------------------ main
def main():
    ap = argparse.ArgumentParser()
    ap.add_argument("--gpus", type=int, default=1)
    ap.add_argument("--steps", type=int, default=20000)
    ap.add_argument("--warmup", type=int, default=50)
    ap.add_argument("--impl", default="moeq", choices=["moeq", "reference"])
    ap.add_argument("--M", type=int, default=1)
    ap.add_argument("--layers", type=int, default=8)
    ap.add_argument("--sweep-steps", type=int, default=400)
    ap.add_argument("--no-sweep", action="store_true")
    ap.add_argument("--no-cpu", action="store_true")
    ap.add_argument("--e2e-steps", type=int, default=2000)
    ap.add_argument("--profile-case", action="store_true",
                    help="run a few launches of the small ncu case (8 routed experts, top-8) and exit")
    ap.add_argument("--reps", type=int, default=3)
    ap.add_argument("--profile-experts", type=int, default=8, help="routed experts of the --profile-case layer")
    ap.add_argument("--profile-dense", action="store_true",
                    help="a few launches of the dense configurations (for ncu), no timing")
    ap.add_argument("--profile-lm-head", action="store_true",
                    help="a few launches of the LM head at 1 and 4 tokens (for ncu), no timing")
    ap.add_argument("--no-dense", action="store_true", help="skip the dense configurations and the gate_up ladder")
    ap.add_argument("--no-stack", action="store_true", help="skip the multi-layer stack sweep")
    ap.add_argument("--stack-calls", type=int, default=40)
    ap.add_argument("--ladder-child", action="store_true", help=argparse.SUPPRESS)
    args = ap.parse_args()
    if args.profile_dense:
        profile_dense(args.reps)
        return
    if args.profile_lm_head:
        profile_lm_head(args.reps)
        return
    if args.profile_case:
        profile_case(args.M, args.reps, args.profile_experts)
        return
    if args.ladder_child:
        from bandwidth_bound_fp8_gb300 import build as b
        b.build()
        peak, _ = load_peaks()
        print(json.dumps(gate_up_ladder(peak, variants=("four_ctas",), reps=5)["four_ctas"]))
        return
    if args.warmup < 3:
        raise SystemExit("--warmup must be >= 3")
    world, rank, local = dist_setup()
    if args.impl == "reference":
        reference_arm(args, world, rank)
        return

    from bandwidth_bound_fp8_gb300 import build as b
    b.build()
    from bandwidth_bound_fp8_gb300 import moeq
    moeq.load()
    peak, peak_kind = load_peaks()
    stack = Stack(args.layers, seed=CFG["seed"] + 1000 * rank)

    clk = ClockSampler(local)
    clk.start()
    time.sleep(0.5)
    r = bench_M(stack, args.M, args.steps, args.warmup, world, seed=5000 + rank * 100000)
    clk.stop()
    ms = max_over_ranks(r["ms"], world)
    total_bytes = sum_over_ranks(r["bytes"], world)
    value = total_bytes / (ms * 1e-3) / 1e9
    clocks = clk.summary(*r["wall"])

    k_ms = r["kernel_ms"]
    achieved = r["kernel_bytes"] / (k_ms * 1e-3) / 1e9
    kname = ("mtok_kernel (MoE layer: route, quant x, gate_up+SwiGLU on tcgen05, quant h, down, combine)" if args.M <= 16 else
             "stream_kernel (whole MoE layer: route, gate_up+SwiGLU, down, combine)")
    roof = {"bound": "hbm", "kernel": kname,
            "achieved": round(achieved, 1), "peak": peak, "peak_kind": f"{peak_kind} hbm_gbs (copy), of {peak_kind}",
            "unit": "GB/s", "frac": round(achieved / peak, 4), "traffic": ncu_traffic("layer", args.M, r["kernel_bytes"]),
            "algorithmic_bytes_per_launch": r["kernel_bytes"], "ms_per_launch": round(k_ms, 5),
            "launch_duration": "timed region / launches (one launch per step, launches back to back)",
            "isolated_launch_ms": round(r["isolated_ms"], 5),
            "isolated_frac": round(r["isolated_bytes"] / (r["isolated_ms"] * 1e-3) / 1e9 / peak, 4)}

    sweep = {}
    if not args.no_sweep and rank == 0:
        for M in (1, 2, 4, 8, 16):
            rr = bench_M(stack, M, args.sweep_steps, 10, 1, seed=7000 + M)
            us = rr["ms"] * 1e3 / rr["steps"]
            gbs = rr["bytes"] / (rr["ms"] * 1e-3) / 1e9
            sweep[f"M{M}"] = {"us_per_layer": round(us, 2), "weight_GBps": round(gbs, 1),
                              "frac_of_measured_hbm": round(gbs / peak, 4), "frac_of_8TBps": round(gbs / 8000, 4),
                              "U_mean": rr["U_mean"],
                              "isolated_launch_us": round(rr["isolated_ms"] * 1e3, 2)}
            del rr
    stack_sweep = {}
    if not args.no_stack and rank == 0:
        for M in (1, 2, 4, 8, 16):
            stack_sweep[f"M{M}"] = bench_stack(stack, M, args.stack_calls, seed=8000 + 37 * M, peak=peak)
        stack_sweep["call"] = "moeq_moe_stack (one CUDA graph per step through all layers)"
    dense = None
    if rank == 0 and not args.no_dense:
        dense = bench_dense(peak, with_oracle=not args.no_cpu)
        ladder = gate_up_ladder(peak)
        ladder["four_ctas"] = gate_up_ladder_child(peak)
        dense["gate_up_ladder"] = ladder
        dense["lm_head"] = bench_lm_head(peak)
    e2e = e2e_batch = None
    if rank == 0:
        e = bench_e2e(stack, args.M, min(args.e2e_steps, args.steps), seed=9000)
        e2e = {"value": round(e["value"], 1), "unit": "GB/s", "h2d_bytes_per_step": e["h2d"],
               "d2h_bytes_per_step": e["d2h"], "ms_per_step": round(e["ms_per_step"], 5), "mode": e["mode"]}
        e = bench_e2e_batch(stack, args.M, min(args.e2e_steps, args.steps), seed=9000)
        e2e_batch = {"value": round(e["value"], 1), "unit": "GB/s", "h2d_bytes_per_step": e["h2d"],
                     "d2h_bytes_per_step": e["d2h"], "ms_per_step": round(e["ms_per_step"], 5), "mode": e["mode"]}
    cpu = None
    if rank == 0 and not args.no_cpu:
        cpu = cpu_baseline(stack, 1, seed=9500)

    if rank == 0:
        line = {
            "metric": METRIC, "value": round(value, 1), "unit": "GB/s", "n_gpus": world, "steps": args.steps,
            "warmup": args.warmup, "ms_per_step": round(ms / args.steps, 5), "higher_is_better": True,
            "scaling": "weak", "vs_baseline": None, "dtype": "f32", "data": "synthetic",
            "config": {"workload": f"moe_layer_m{args.M}_h6144_i2048_e256_top8_shared1",
                       "M": args.M, "hidden": H, "intermediate": I, "experts": E, "top_k": TOPK, "shared": 1,
                       "layers_rotated": args.layers, "unique_experts_mean": r["U_mean"],
                       "bytes_per_step_mean": r["bytes"] / r["steps"],
                       "l2": "inputs larger than L2: 8 layers x 9.7 GB rotated, each step reads its experts cold",
                       "parallelism": f"replicas x{world}"},
            "us_per_layer": round(ms * 1e3 / args.steps, 3),
            "frac_of_8TBps": round(value / world / 8000, 4),
            "kernel_us": round(r["kernel_ms"] * 1e3, 3),
            "isolated_launch_us": round(r["isolated_ms"] * 1e3, 3),
            "roofline": roof, "e2e": e2e, "e2e_batch16": e2e_batch, "cpu_baseline": cpu, "clocks": clocks,
            "gpu_launches": args.steps, "sweep": sweep, "stack": stack_sweep, "dense": dense,
        }
        print(json.dumps(line), flush=True)
    if world > 1:
        import torch.distributed as dist
        dist.destroy_process_group()


if __name__ == "__main__":
    main()
