#!/usr/bin/env python
"""Benchmark of the ConvRot W4A8 linear layer on GB300.

One step = one whole layer at the MiniMax-H3 QKV projection shape (M = 19989
tokens, K = 5376, N = 21504, BF16 in / BF16 out): NVFP4 weight preparation
(decode + rotation + S8), activation rotation + S8, and the integer GEMM with
its dequant epilogue -- the three C-ABI calls, weights re-prepared every
call as in the layer's single runtime path.  Inputs are seeded synthetic data
of the workload's shape and distribution, resident in HBM before timing; L2 is
flushed (a write larger than L2) before every timed step.

Prints ONE JSON line.  `value` is effective TOPS = 2 M N K / t.  The layer
runs on one GPU: its GEMM loads operand tiles with cluster-multicast TMA over
tensor maps of this GPU's own memory, so bench.py refuses --gpus > 1 and any
launch with WORLD_SIZE > 1 (the CPU reference arm excepted).

  python bench.py [--steps K] [--warmup W] [--impl ours|reference]
"""
from __future__ import annotations

import argparse
import csv
import dataclasses
import hashlib
import io
import json
import os
import statistics
import subprocess
import sys
import tempfile
import time

ROOT = os.path.dirname(os.path.abspath(__file__))
if ROOT not in sys.path:
    sys.path.insert(0, ROOT)

import numpy as np  # noqa: E402

import synth  # noqa: E402

METRIC = "ms/layer and effective INT8 TOPS at M=19989 (QKV, FFN-down); % of INT8/HBM roofline"
# the pages' QKV layer time on an A40 at M=19989 (context, another machine)
PAGES_QKV_MS = 25.08
FALLBACK_PEAKS = {"hbm_gbs": 6800.0, "bf16_tflops": 1900.0, "bf16_tflops_sustained": 1700.0}
# DRAM traffic (read + write bytes) of one full-size QKV GEMM launch, from an ncu capture of
# this kernel; valid only while code_sha16(gemm.cu) equals this (the hash ignores comments;
# otherwise the bench line reports traffic as null).
GEMM_TRAFFIC = {"sha256_16": "821fc3350e166564", "bytes": 2865981184 + 924844032}


def code_sha16(path: str) -> str:
    """First 16 hex digits of the SHA-256 of a C++ source with its comments and
    blank lines removed: it changes when the code changes, not the comments."""
    import re
    with open(path) as f:
        src = f.read()
    src = re.sub(r"/\*.*?\*/", "", src, flags=re.S)
    src = re.sub(r"//[^\n]*", "", src)
    lines = [ln.rstrip() for ln in src.splitlines() if ln.strip()]
    return hashlib.sha256("\n".join(lines).encode()).hexdigest()[:16]


def load_peaks():
    p = os.path.join(ROOT, "MEASURED_PEAKS.json")
    if os.path.exists(p):
        with open(p) as f:
            d = json.load(f)
        return d, "measured"
    return dict(FALLBACK_PEAKS), "fallback"


# ---------------------------------------------------------------- workload sizes
def norms_pay(Kp: int) -> bool:
    """Whether the layer asks the quantisation kernels for code-norm bounds.
    They cost the kernels a sum of squares (about 10 us each at QKV) and let
    the GEMM run a tile as one FP32 chunk when max bound(A) x max bound(B) <
    2^24, which saves it about as much (the drains of the exact chunks cost
    the QKV GEMM about 1%).
    Rotated rows of ordinary data have codes with an RMS of about 30-36, so a
    bound near 33 sqrt(K_p): the product stays below 2^24 up to K_p of about
    8192-13000 (QKV, K_p = 5376: about 2300 each) and not at K_p = 14336
    (FFN-down: about 4200 each), where the bounds would cost without paying."""
    return Kp <= 8192


def layer_sizes(wl: synth.Workload):
    """Work of one layer.  act_alg / w_alg are the algorithmic bytes of the
    two quantisation kernels with one-byte S8 codes (inputs read once, codes
    and scales written once); act_bytes / w_bytes are the bytes the kernels
    actually move, with the codes held as FP16 (two bytes) for the GEMM."""
    Kp = -(-wl.K // 256) * 256
    Ks = synth.stored_k(wl.K)
    esz = {"bf16": 2, "fp16": 2, "fp32": 4}
    act_in = wl.M * wl.k_in * esz[wl.x_dtype]
    w_in = wl.N * Ks // 2 + wl.N * Ks // 16
    nb = 4 if norms_pay(Kp) else 0          # the norm bounds, when requested
    return dict(Kp=Kp, Ks=Ks, ops=2.0 * wl.M * wl.N * wl.K, gemm_flops=2.0 * wl.M * wl.N * Kp,
                act_alg=act_in + wl.M * Kp + 4 * wl.M, w_alg=w_in + wl.N * Kp + 4 * wl.N,
                act_bytes=act_in + wl.M * Kp * 2 + (4 + nb) * wl.M,
                w_bytes=w_in + 4 + wl.N * Kp * 2 + (4 + nb) * wl.N)


# ---------------------------------------------------------------- clocks
class ClockSampler:
    FIELDS = ("index,pci.bus_id,clocks.sm,clocks.max.sm,power.draw,clocks_event_reasons.active,"
              "clocks_event_reasons.hw_slowdown,clocks_event_reasons.hw_thermal_slowdown,"
              "clocks_event_reasons.sw_thermal_slowdown,clocks_event_reasons.sw_power_cap")

    def __init__(self, bus_id: str | None):
        self.bus_id = bus_id
        self.proc = None
        self.path = None

    def start(self):
        fd, self.path = tempfile.mkstemp(suffix=".csv")
        os.close(fd)
        try:
            self.out = open(self.path, "w")
            self.proc = subprocess.Popen(
                ["nvidia-smi", f"--query-gpu={self.FIELDS}", "--format=csv,noheader,nounits",
                 "-lms", "100"], stdout=self.out, stderr=subprocess.DEVNULL)
        except OSError:
            self.proc = None

    def stop(self):
        if self.proc is None:
            return None
        self.proc.terminate()
        try:
            self.proc.wait(timeout=5)
        except subprocess.TimeoutExpired:
            self.proc.kill()
        self.out.close()
        rows = []
        with open(self.path) as f:
            for r in csv.reader(io.StringIO(f.read())):
                if len(r) < 10:
                    continue
                r = [c.strip() for c in r]
                if self.bus_id and self.bus_id.lower() not in r[1].lower():
                    continue
                rows.append(r)
        os.unlink(self.path)
        if not rows:
            return None
        sm = [float(r[2]) for r in rows if r[2].replace(".", "", 1).isdigit()]
        mx = [float(r[3]) for r in rows if r[3].replace(".", "", 1).isdigit()]
        names = ["hw_slowdown", "hw_thermal_slowdown", "sw_thermal_slowdown", "sw_power_cap"]
        reasons = sorted({n for r in rows for n, v in zip(names, r[6:10]) if v.lower() == "active"})
        return {"sm_mhz": statistics.median(sm) if sm else None,
                "sm_max_mhz": max(mx) if mx else None, "reasons": reasons, "samples": len(rows)}


# ---------------------------------------------------------------- one GPU
SINGLE_GPU_MSG = ("bench.py times the ConvRot layer on one GPU only: its GEMM issues cluster-multicast "
                  "TMA loads over tensor maps of this GPU's own memory, and no run of this code may span "
                  "two or more GPUs.  Token rows shard without any exchange (replicas), but that path is "
                  "not run here.")


def single_gpu_guard(n_gpus: int, world: int) -> None:
    """Refuses a launch on more than one GPU (the product arm)."""
    if n_gpus != 1 or world != 1:
        raise SystemExit(f"refused: --gpus {n_gpus}, WORLD_SIZE {world}. " + SINGLE_GPU_MSG)


# The job-level helpers below are kept general (max over ranks, sum of
# replicas) and are exercised on the CPU by gloo tests; on the single GPU
# that the benchmark runs they reduce to the identity.
def barrier(world):
    if world > 1:
        import torch.distributed as dist
        dist.barrier()


def reduce_max(v: float, world: int) -> float:
    """Maximum of v over the ranks (the slowest rank's time)."""
    if world == 1:
        return v
    import torch
    import torch.distributed as dist
    dev = "cuda" if dist.get_backend() == "nccl" else "cpu"
    t = torch.tensor([v], dtype=torch.float64, device=dev)
    dist.all_reduce(t, op=dist.ReduceOp.MAX)
    return float(t.item())


def aggregate_tops(ops_per_step: float, steps: int, max_ms: float, world: int) -> float:
    """Whole-job throughput: every rank runs its own replica of the step."""
    return world * ops_per_step * steps / (max_ms / 1e3) / 1e12


# ---------------------------------------------------------------- GPU layer
class Layer:
    """Device buffers and the three C-ABI calls of one ConvRot layer."""

    def __init__(self, wl: synth.Workload, dev):
        import torch

        import rotated_w4a8_int8_gb300 as cr
        self.cr = cr
        self.wl = wl
        self.sz = layer_sizes(wl)
        t0 = time.time()
        x = synth.make_activations(wl)
        packed, scales, tscale = synth.make_nvfp4_weight(wl)
        self.gen_s = time.time() - t0
        tdt = {"bf16": torch.bfloat16, "fp16": torch.float16, "fp32": torch.float32}
        if wl.x_dtype == "fp32":
            xh = torch.from_numpy(x)
        else:
            xh = torch.from_numpy(x.view(np.int16)).view(tdt[wl.x_dtype])
        # pinned host copies (the end-to-end leg copies them in every step)
        self.h_x = xh.pin_memory()
        self.h_p = torch.from_numpy(packed).pin_memory()
        self.h_s = torch.from_numpy(scales).pin_memory()
        self.h_t = torch.tensor([float(tscale)], dtype=torch.float32).pin_memory()
        self.x = self.h_x.to(dev)
        self.p = self.h_p.to(dev)
        self.s = self.h_s.to(dev)
        self.t = self.h_t.to(dev)
        Kp = self.sz["Kp"]
        self.aq = torch.empty(wl.M, Kp, dtype=torch.float16, device=dev)
        self.sa = torch.empty(wl.M, dtype=torch.float32, device=dev)
        # code-norm bounds, requested only where they can pay (norms_pay)
        use = norms_pay(Kp)
        self.na = torch.empty(wl.M, dtype=torch.float32, device=dev) if use else None
        self.wq = torch.empty(wl.N, Kp, dtype=torch.float16, device=dev)
        self.sw = torch.empty(wl.N, dtype=torch.float32, device=dev)
        self.nw = torch.empty(wl.N, dtype=torch.float32, device=dev) if use else None
        self.y = torch.empty(wl.M, wl.N, dtype=tdt[wl.out_dtype], device=dev)
        self.h_y = None
        self.in_bytes = sum(t.numel() * t.element_size() for t in (self.h_x, self.h_p, self.h_s, self.h_t))

    def weight(self):
        self.cr.prepare_weight(self.p, self.s, self.t, self.wl.K, self.wq, self.sw, w_norm=self.nw)

    def act(self):
        self.cr.quant_act(self.x, self.wl.K, self.aq, self.sa, swiglu=self.wl.swiglu, a_norm=self.na)

    def gemm(self):
        self.cr.gemm(self.aq, self.sa, self.wq, self.sw, self.y, a_norm=self.na, w_norm=self.nw)

    def step(self):
        self.weight()
        self.act()
        self.gemm()


def time_layer(layer: Layer, steps: int, warmup: int, world: int, flush, sampler=None):
    """K timed steps; per-kernel CUDA events on the launching stream; L2 flushed
    before every step (outside the events)."""
    import torch
    for _ in range(warmup):
        flush()
        layer.step()
    torch.cuda.synchronize()
    ev = [[torch.cuda.Event(enable_timing=True) for _ in range(4)] for _ in range(steps)]
    if sampler:
        sampler.start()
        time.sleep(0.3)
    barrier(world)
    torch.cuda.synchronize()
    for i in range(steps):
        flush()
        ev[i][0].record()
        layer.weight()
        ev[i][1].record()
        layer.act()
        ev[i][2].record()
        layer.gemm()
        ev[i][3].record()
    torch.cuda.synchronize()
    barrier(world)
    clocks = sampler.stop() if sampler else None
    w = [e[0].elapsed_time(e[1]) for e in ev]
    a = [e[1].elapsed_time(e[2]) for e in ev]
    g = [e[2].elapsed_time(e[3]) for e in ev]
    tot = [e[0].elapsed_time(e[3]) for e in ev]
    return dict(total_ms=sum(tot), step_ms=tot, weight_ms=w, act_ms=a, gemm_ms=g, clocks=clocks)


def time_layer_overlapped(layer: Layer, steps: int, warmup: int, world: int, flush, sampler=None):
    """K timed steps of the layer as the pages run it: the weight preparation
    on a second stream beside the activation quantisation (they are
    independent), joined before the GEMM.  One event pair per step on the
    main stream; L2 flushed before every step (outside the events)."""
    import torch
    main = torch.cuda.current_stream()
    side = torch.cuda.Stream(main.device)

    def step():
        side.wait_stream(main)
        with torch.cuda.stream(side):
            layer.weight()
        layer.act()
        main.wait_stream(side)
        layer.gemm()

    for _ in range(warmup):
        flush()
        step()
    torch.cuda.synchronize()
    ev = [[torch.cuda.Event(enable_timing=True) for _ in range(2)] for _ in range(steps)]
    if sampler:
        sampler.start()
        time.sleep(0.3)
    barrier(world)
    torch.cuda.synchronize()
    for i in range(steps):
        flush()
        ev[i][0].record()
        step()
        ev[i][1].record()
    torch.cuda.synchronize()
    barrier(world)
    clocks = sampler.stop() if sampler else None
    tot = [e[0].elapsed_time(e[1]) for e in ev]
    return dict(total_ms=sum(tot), step_ms=tot, clocks=clocks)


class E2EPipeline:
    """The layer through the public API with host buffers, pipelined over steps.

    Every step copies its own inputs (x and the NVFP4 weight) from pinned host
    memory, runs the three calls and copies its whole output back to pinned
    host memory.  Three streams overlap step i+1's input copy and step i-1's
    output copy with step i's kernels; device inputs and outputs are double
    buffered and guarded by events.
    """

    def __init__(self, layer: Layer, copy_streams: int = 2, host_poll: bool = True):
        import torch
        self.L = layer
        # The host polls the pipeline's events instead of sleeping in a blocking
        # wait: on some boxes the device-to-host copies ran at a fraction of the
        # link rate once the host thread went idle.
        self.host_poll = host_poll
        self.torch = torch
        dev = layer.x.device
        self.s_in = torch.cuda.Stream(dev)
        self.s_run = torch.cuda.Stream(dev)
        self.s_out = torch.cuda.Stream(dev)
        # the output copy is split over several streams so that several copy engines work on it
        self.s_out_parts = [torch.cuda.Stream(dev) for _ in range(copy_streams)]
        self.bufs = []
        for _ in range(2):
            self.bufs.append(dict(x=torch.empty_like(layer.x), p=torch.empty_like(layer.p),
                                  s=torch.empty_like(layer.s), t=torch.empty_like(layer.t),
                                  y=torch.empty_like(layer.y),
                                  hy=torch.empty(layer.y.shape, dtype=layer.y.dtype).pin_memory()))
        self.in_bytes = layer.in_bytes
        self.out_bytes = layer.y.numel() * layer.y.element_size()

    def run(self, steps: int) -> float:
        torch, L = self.torch, self.L
        ev = lambda: torch.cuda.Event()
        in_done = [None, None]       # inputs of the buffer landed
        run_done = [None, None]      # kernels of the buffer finished (inputs free)
        out_done = [None, None]      # output of the buffer copied out (y free)
        t0 = torch.cuda.Event(enable_timing=True)
        t1 = torch.cuda.Event(enable_timing=True)
        marks = []                   # each step's output copied out (timing events)
        t0.record(self.s_in)
        for i in range(steps):
            b = self.bufs[i % 2]
            k = i % 2
            if self.host_poll and run_done[k] is not None:
                # the host stays at most two steps ahead, polling (not sleeping)
                while not run_done[k].query():
                    pass
            with torch.cuda.stream(self.s_in):
                if run_done[k] is not None:
                    self.s_in.wait_event(run_done[k])
                b["x"].copy_(L.h_x, non_blocking=True)
                b["p"].copy_(L.h_p, non_blocking=True)
                b["s"].copy_(L.h_s, non_blocking=True)
                b["t"].copy_(L.h_t, non_blocking=True)
                in_done[k] = ev()
                in_done[k].record(self.s_in)
            with torch.cuda.stream(self.s_run):
                self.s_run.wait_event(in_done[k])
                if out_done[k] is not None:
                    self.s_run.wait_event(out_done[k])
                L.cr.prepare_weight(b["p"], b["s"], b["t"], L.wl.K, L.wq, L.sw, w_norm=L.nw)
                L.cr.quant_act(b["x"], L.wl.K, L.aq, L.sa, swiglu=L.wl.swiglu, a_norm=L.na)
                L.cr.gemm(L.aq, L.sa, L.wq, L.sw, b["y"], a_norm=L.na, w_norm=L.nw)
                run_done[k] = ev()
                run_done[k].record(self.s_run)
            parts = self.s_out_parts
            rows = b["y"].shape[0]
            step = -(-rows // len(parts))
            for j, sp in enumerate(parts):
                r0, r1 = j * step, min(rows, (j + 1) * step)
                if r0 >= r1:
                    continue
                with torch.cuda.stream(sp):
                    sp.wait_event(run_done[k])
                    b["hy"][r0:r1].copy_(b["y"][r0:r1], non_blocking=True)
            with torch.cuda.stream(self.s_out):
                for sp in parts:
                    self.s_out.wait_stream(sp)
                out_done[k] = ev()
                out_done[k].record(self.s_out)
                marks.append(torch.cuda.Event(enable_timing=True))
                marks[-1].record(self.s_out)
        self.s_out.wait_stream(self.s_in)
        self.s_out.wait_stream(self.s_run)
        t1.record(self.s_out)
        if self.host_poll:
            while not t1.query():
                pass
        t1.synchronize()
        # intervals between consecutive steps' output completions, and the
        # pipeline's fill: the start to the first step's output
        self.step_ms = [marks[i - 1].elapsed_time(marks[i]) for i in range(1, len(marks))]
        self.first_ms = t0.elapsed_time(marks[0]) if marks else None
        return t0.elapsed_time(t1)


def host_link_gbs(pipe: "E2EPipeline", reps: int = 3):
    """The host link on this machine, right before the timed end-to-end run (best
    of `reps`): the step's output copied to pinned host memory over the
    pipeline's copy streams, alone ("d2h") and while two layers run on the
    pipeline's kernel stream ("d2h_beside_kernels", with the layers' own
    time beside it); the activation input copied in alone ("h2d").  The host
    link is shared with other work on the machine, so the end-to-end figure
    is read against these."""
    import torch
    b = pipe.bufs[0]
    parts = pipe.s_out_parts
    rows = b["y"].shape[0]
    step = -(-rows // len(parts))
    ev = lambda: torch.cuda.Event(enable_timing=True)

    def copy_out():
        t0, t1 = ev(), ev()
        t0.record()
        for j, sp in enumerate(parts):
            sp.wait_stream(torch.cuda.current_stream())
            with torch.cuda.stream(sp):
                b["hy"][j * step:(j + 1) * step].copy_(b["y"][j * step:(j + 1) * step], non_blocking=True)
        for sp in parts:
            torch.cuda.current_stream().wait_stream(sp)
        t1.record()
        return t0, t1

    out = {"d2h": 0.0, "h2d": 0.0, "d2h_beside_kernels": 0.0, "kernels_beside_d2h_ms": None,
           "d2h_beside_h2d": 0.0}
    L = pipe.L
    for _ in range(reps):
        torch.cuda.synchronize()
        t0, t1 = copy_out()
        t1.synchronize()
        out["d2h"] = max(out["d2h"], pipe.out_bytes / (t0.elapsed_time(t1) / 1e3) / 1e9)
        t0, t1 = ev(), ev()
        t0.record()
        b["x"].copy_(L.h_x, non_blocking=True)
        t1.record()
        t1.synchronize()
        out["h2d"] = max(out["h2d"], L.h_x.numel() * L.h_x.element_size() / (t0.elapsed_time(t1) / 1e3) / 1e9)
        # the copy beside two layers on the kernel stream
        torch.cuda.synchronize()
        k0, k1 = ev(), ev()
        pipe.s_run.wait_stream(torch.cuda.current_stream())
        with torch.cuda.stream(pipe.s_run):
            k0.record()
            for _ in range(2):
                L.step()
            k1.record()
        t0, t1 = copy_out()
        torch.cuda.synchronize()
        out["d2h_beside_kernels"] = max(out["d2h_beside_kernels"],
                                        pipe.out_bytes / (t0.elapsed_time(t1) / 1e3) / 1e9)
        out["kernels_beside_d2h_ms"] = k0.elapsed_time(k1) / 2
        # the copy beside the next step's input copy
        pipe.s_in.wait_stream(torch.cuda.current_stream())
        with torch.cuda.stream(pipe.s_in):
            pipe.bufs[1]["x"].copy_(L.h_x, non_blocking=True)
        t0, t1 = copy_out()
        torch.cuda.synchronize()
        out["d2h_beside_h2d"] = max(out["d2h_beside_h2d"], pipe.out_bytes / (t0.elapsed_time(t1) / 1e3) / 1e9)
    return out


E2E_RUNS = 5


def time_e2e(layer: Layer, steps: int, warmup: int, world: int, runs: int = E2E_RUNS):
    """`runs` timed runs of `steps` pipelined steps; returns the median run's
    time and per-step intervals, and every run's ms per step.  On some boxes a
    single step of a run stalled for tens of milliseconds (its neighbours at
    the usual 4.4-4.6 ms), so one run alone can misstate the pipeline."""
    import torch
    pipe = E2EPipeline(layer)
    pipe.run(warmup)
    torch.cuda.synchronize()
    link = host_link_gbs(pipe)
    results = []
    for _ in range(runs):
        barrier(world)
        ms = pipe.run(steps)
        torch.cuda.synchronize()
        barrier(world)
        results.append((ms, list(pipe.step_ms), pipe.first_ms))
    order = sorted(range(runs), key=lambda r: results[r][0])
    ms, step_ms, first_ms = results[order[runs // 2]]
    iv = sorted(step_ms)
    intervals = None
    if iv:
        intervals = {"min": iv[0], "median": iv[len(iv) // 2], "max": iv[-1],
                     "first": step_ms[0], "last": step_ms[-1], "to_first_output": first_ms}
    runs_ms_per_step = [r[0] / steps for r in results]
    return ms, pipe.in_bytes, pipe.out_bytes, link, intervals, runs_ms_per_step


def time_ffn_block(dev, world, flush, warmup, steps=10):
    """The MiniMax-H3 FFN block at M = 19989: fc1 (28672 x 5376) with its NVFP4
    weight prepared, the fused SwiGLU + rotation + S8 of its BF16 output, and
    fc2 (5376 x 14336) with its weight prepared: six kernel launches per step."""
    import torch

    import rotated_w4a8_int8_gb300 as cr
    up = synth.WORKLOADS["ffn_up"]
    up = dataclasses.replace(up, x_dtype="bf16", out_dtype="bf16")
    down = synth.WORKLOADS["ffn_down"]
    M, H, F = up.M, up.K, down.K
    x = synth.make_activations(up)
    p1, s1, t1 = synth.make_nvfp4_weight(up)
    p2, s2, t2 = synth.make_nvfp4_weight(down)
    xd = torch.from_numpy(x.view(np.int16)).to(dev).view(torch.bfloat16)
    P1, S1, T1 = (torch.from_numpy(p1).to(dev), torch.from_numpy(s1).to(dev),
                  torch.tensor([float(t1)], dtype=torch.float32, device=dev))
    P2, S2, T2 = (torch.from_numpy(p2).to(dev), torch.from_numpy(s2).to(dev),
                  torch.tensor([float(t2)], dtype=torch.float32, device=dev))
    Hp, Fp = cr.padded_k(H), cr.padded_k(F)
    w1 = torch.empty(2 * F, Hp, dtype=torch.float16, device=dev)
    sw1 = torch.empty(2 * F, dtype=torch.float32, device=dev)
    nw1 = torch.empty(2 * F, dtype=torch.float32, device=dev) if norms_pay(Hp) else None
    w2 = torch.empty(H, Fp, dtype=torch.float16, device=dev)
    sw2 = torch.empty(H, dtype=torch.float32, device=dev)
    nw2 = torch.empty(H, dtype=torch.float32, device=dev) if norms_pay(Fp) else None
    xq = torch.empty(M, Hp, dtype=torch.float16, device=dev)
    sx = torch.empty(M, dtype=torch.float32, device=dev)
    nx = torch.empty(M, dtype=torch.float32, device=dev) if norms_pay(Hp) else None
    h2 = torch.empty(M, 2 * F, dtype=torch.bfloat16, device=dev)
    hq = torch.empty(M, Fp, dtype=torch.float16, device=dev)
    sh = torch.empty(M, dtype=torch.float32, device=dev)
    nh = torch.empty(M, dtype=torch.float32, device=dev) if norms_pay(Fp) else None
    y = torch.empty(M, H, dtype=torch.bfloat16, device=dev)

    def step():
        cr.prepare_weight(P1, S1, T1, H, w1, sw1, w_norm=nw1)
        cr.quant_act(xd, H, xq, sx, a_norm=nx)
        cr.gemm(xq, sx, w1, sw1, h2, a_norm=nx, w_norm=nw1)
        cr.prepare_weight(P2, S2, T2, F, w2, sw2, w_norm=nw2)
        cr.quant_act(h2, F, hq, sh, swiglu=True, a_norm=nh)
        cr.gemm(hq, sh, w2, sw2, y, a_norm=nh, w_norm=nw2)

    for _ in range(warmup):
        flush()
        step()
    torch.cuda.synchronize()
    barrier(world)
    tot = 0.0
    for _ in range(steps):
        flush()
        a = torch.cuda.Event(enable_timing=True)
        b = torch.cuda.Event(enable_timing=True)
        a.record()
        step()
        b.record()
        b.synchronize()
        tot += a.elapsed_time(b)
    ms = reduce_max(tot, world) / steps
    ops = 2.0 * M * (2 * F) * H + 2.0 * M * H * F
    return {"workload": f"FFN block M={M}: fc1 {2 * F}x{H} -> SwiGLU -> fc2 {H}x{F}, BF16",
            "ms_per_block": ms, "eff_tops": ops / (ms / 1e3) / 1e12, "kernels_per_step": 6}


def time_controls(wl: synth.Workload, dev, world, flush, warmup, steps=20):
    """The pages' comparison points on the main workload, same calls:
    - w8a8_resident_s8: weights prepared once and kept as 1-byte S8 codes,
      widened to the GEMM's FP16 codes every call, + act quant + GEMM;
    - resident_f16_codes: weights prepared once in the GEMM's operand format
      (the 'expanded W8A8' control): act quant + GEMM only;
    - prescale_bias: the full layer with channel pre-scales and a bias."""
    import torch

    import rotated_w4a8_int8_gb300 as cr
    L = Layer(wl, dev)
    Kp = L.sz["Kp"]
    wq8 = torch.empty(wl.N, Kp, dtype=torch.int8, device=dev)
    sw8 = torch.empty(wl.N, dtype=torch.float32, device=dev)
    cr.prepare_weight(L.p, L.s, L.t, wl.K, wq8, sw8)
    L.weight()
    gen = torch.Generator(device="cpu").manual_seed(5)
    pre = torch.exp(torch.rand(wl.K, generator=gen) * 2 - 1).to(dev)
    bias = (torch.randn(wl.N, generator=gen) * 0.1).to(dev)

    def w8a8():
        cr.widen_codes(wq8, L.wq, cols=Kp)
        L.act()
        L.gemm()                    # the weight-norm bounds of L.weight() above still hold

    def resident():
        L.act()
        L.gemm()

    def ps_bias():
        L.weight()
        cr.quant_act(L.x, wl.K, L.aq, L.sa, swiglu=wl.swiglu, pre_scale=pre, a_norm=L.na)
        cr.gemm(L.aq, L.sa, L.wq, L.sw, L.y, bias=bias, a_norm=L.na, w_norm=L.nw)

    out = {}
    for name, fn in (("w8a8_resident_s8", w8a8), ("resident_f16_codes", resident), ("prescale_bias", ps_bias)):
        for _ in range(warmup):
            flush()
            fn()
        torch.cuda.synchronize()
        barrier(world)
        tot = 0.0
        for _ in range(steps):
            flush()
            a = torch.cuda.Event(enable_timing=True)
            b = torch.cuda.Event(enable_timing=True)
            a.record()
            fn()
            b.record()
            b.synchronize()
            tot += a.elapsed_time(b)
        ms = reduce_max(tot, world) / steps
        out[name] = {"ms_per_layer": ms, "eff_tops": L.sz["ops"] / (ms / 1e3) / 1e12}
    out["pages_a40_ms"] = {"w8a8_expanded": 23.40, "convrot_w4a8": 25.08}
    del L
    torch.cuda.empty_cache()
    return out


def time_decode_probe(layer: "Layer", strips: int, g_ms: float, warmup: int, reps: int = 5):
    """The producer of a decode-inside-GEMM measured: convrot_decode_gemm_probe
    runs, one CTA per SM, every work unit of this layer's GEMM (each 256-token
    strip x each 128-row weight half) and builds that unit's FP16 weight codes
    from the NVFP4 bytes into the GEMM's swizzled shared-memory B layout, with
    a consumer that releases each stage at once (an MMA that takes no time).
    A fused GEMM can be no faster than its producer, so `ratio` (the best
    producer time over the layer GEMM's time in this run) bounds what decode
    inside the GEMM would cost; `unit_us` is one SM's time per unit, against
    the GEMM's time per 256 x 256 work item on its CTA pair (tile_mma_us).
    The NVFP4 weight stays in L2 (no flush), which favours the probe.  8 and
    16 producer warps are timed; the best is kept."""
    import torch
    cr = layer.cr
    status = torch.zeros(1, dtype=torch.int32, device=layer.x.device)
    out = {}
    for pw in (8, 16):
        def run():
            cr.decode_gemm_probe(layer.p, layer.s, layer.t, layer.sw, layer.wl.K, strips, pw, status)
        for _ in range(warmup):
            run()
        torch.cuda.synchronize()
        if int(status.item()) != 0:
            raise SystemExit(f"decode-GEMM probe: a wait ran out (code {int(status.item())})")
        ts = []
        for _ in range(reps):
            e0 = torch.cuda.Event(enable_timing=True)
            e1 = torch.cuda.Event(enable_timing=True)
            e0.record()
            run()
            e1.record()
            e1.synchronize()
            ts.append(e0.elapsed_time(e1))
        out[f"pw{pw}_ms"] = statistics.median(ts)
    best = min(out["pw8_ms"], out["pw16_ms"])
    sms = torch.cuda.get_device_properties(layer.x.device).multi_processor_count
    units = strips * -(-layer.wl.N // 128)
    out.update({"ms": best, "units": units, "unit_us": 1e3 * best * min(sms, units) / units,
                "gemm_ms": g_ms, "ratio": best / g_ms,
                "note": "producer of a decode-inside-GEMM alone over this layer's GEMM schedule, "
                        "an instant consumer; a fused GEMM is no faster than this (plus a scales-only pass)"})
    return out


def time_library_controls(layer: "Layer", flush, warmup, steps=20):
    """Library controls on the layer's own operands, timed the way the layer's
    GEMM is (L2 flushed before every call, CUDA events on the launching
    stream), off the product path:
    - cublas_fp16: torch.matmul of the layer's FP16-held activation and weight
      codes, (M x K_p) x (K_p x N): the same tensor-core route, operand width
      and values (the codes' magnitudes set the tensor cores' power draw) as
      the layer's GEMM;
    - int8_mm: torch._int_mm (cuBLASLt S8 x S8 -> int32) on the same codes as
      int8, and on random codes at 8192^3: the rate of the S8 tensor path
      this GPU offers through the library, the denominator of an "INT8
      roofline";
    - int8_mma_sync: this library's register-resident probe of the
      warp-level INT8 tensor instruction (mma.sync m16n8k32 s8) on every SM,
      the hardware side of the same denominator."""
    import torch
    A, B = layer.aq, layer.wq
    M, Kp = A.shape
    N = B.shape[0]
    dev = A.device

    def timed(fn, n):
        for _ in range(warmup):
            flush()
            fn()
        torch.cuda.synchronize()
        tot = 0.0
        for _ in range(n):
            flush()
            a = torch.cuda.Event(enable_timing=True)
            b = torch.cuda.Event(enable_timing=True)
            a.record()
            fn()
            b.record()
            b.synchronize()
            tot += a.elapsed_time(b)
        return tot / n

    out = {}
    ms = timed(lambda: torch.matmul(A, B.t()), steps)
    out["cublas_fp16"] = {"shape": f"{M}x{N}x{Kp}", "operands": "the layer's FP16-held codes", "ms": ms,
                          "tflops": 2.0 * M * N * Kp / (ms / 1e3) / 1e12}
    torch.cuda.empty_cache()
    g = torch.Generator(device=dev).manual_seed(7)
    for name, (m, n, k) in (("int8_mm", (M, N, Kp)), ("int8_mm_8192", (8192, 8192, 8192))):
        try:
            if name == "int8_mm":
                A8, B8 = A.to(torch.int8), B.to(torch.int8)
            else:
                A8 = torch.randint(-127, 128, (m, k), generator=g, device=dev, dtype=torch.int8)
                B8 = torch.randint(-127, 128, (n, k), generator=g, device=dev, dtype=torch.int8)
            ms = timed(lambda: torch._int_mm(A8, B8.t()), 5)
            out[name] = {"shape": f"{m}x{n}x{k}", "ms": ms, "tops": 2.0 * m * n * k / (ms / 1e3) / 1e12}
            del A8, B8
        except RuntimeError as e:            # not offered by this torch build
            out[name] = {"shape": f"{m}x{n}x{k}", "unavailable": str(e).splitlines()[0][:200]}
        torch.cuda.empty_cache()
    # 8 CTAs of 4 warps per SM, 8 independent MMAs per warp and iteration
    sms = torch.cuda.get_device_properties(dev).multi_processor_count
    blocks, iters = 8 * sms, 20000
    res = torch.empty(blocks * 4, dtype=torch.int32, device=dev)
    layer.cr.int8_mma_probe(blocks, 100, res)
    best = None
    for _ in range(5):
        a = torch.cuda.Event(enable_timing=True)
        b = torch.cuda.Event(enable_timing=True)
        a.record()
        layer.cr.int8_mma_probe(blocks, iters, res)
        b.record()
        b.synchronize()
        ms = a.elapsed_time(b)
        best = ms if best is None else min(best, ms)
    if not bool((res == 8 * 32 * iters).all()):
        raise RuntimeError("INT8 MMA probe returned wrong sums")
    ops = blocks * 4 * iters * 8 * (2 * 16 * 8 * 32)
    out["int8_mma_sync"] = {"what": "mma.sync.m16n8k32 s8 x s8 -> s32 from registers, 8 CTAs of 4 warps per SM, "
                                    "best of 5 launches", "ms": best, "tops": ops / (best / 1e3) / 1e12}
    return out


def time_sustained(layer: "Layer", seconds: float, est_ms: float, bus, sm_count: int):
    """Back-to-back layers for about `seconds` s with their own sampled clocks:
    the regime of a long run (many DiT blocks in a row) in which the power cap
    sets the clock.  Operands exceed the L2 (x 215 MB, codes 446 MB at QKV), so
    no flush between layers."""
    n = max(20, int(seconds * 1e3 / max(est_ms, 1e-3)))
    r = time_layer(layer, n, 3, 1, lambda: None, ClockSampler(bus))
    ms = r["total_ms"] / n
    g_ms = statistics.mean(r["gemm_ms"])
    clocks = r["clocks"] or {}
    mhz = clocks.get("sm_mhz")
    out = {"layers": n, "seconds": r["total_ms"] / 1e3, "ms_per_layer": ms,
           "eff_tops": layer.sz["ops"] / (ms / 1e3) / 1e12, "gemm_ms": g_ms,
           "gemm_tflops": layer.sz["gemm_flops"] / (g_ms / 1e3) / 1e12,
           "quant_act_us": 1e3 * statistics.mean(r["act_ms"]),
           "prepare_weight_us": 1e3 * statistics.mean(r["weight_ms"]), "clocks": clocks}
    if mhz:
        out["ms_x_mhz_per_layer"] = ms * mhz
        out["tensor_pipe_peak_at_clock_tflops"] = tensor_pipe_peak(sm_count, mhz)
    return out


def tensor_pipe_peak(sm_count: int, mhz: float) -> float:
    """Dense FP16/BF16 tensor-pipe peak at a given SM clock: 8192 FLOP per
    clock per SM (one 128 x 256 x 16 MMA every 128 clocks)."""
    return 8192.0 * sm_count * mhz * 1e6 / 1e12


# ---------------------------------------------------------------- CPU oracle baseline
class OracleSample:
    """The first m tokens x first n weight rows of a workload, generated once;
    timing covers only the oracle's whole layer on them."""

    def __init__(self, wl: synth.Workload, m_max: int, n_max: int):
        self.wl = wl
        self.m_max, self.n_max = min(wl.M, m_max), min(wl.N, n_max)
        self.x = synth.make_activations(wl, rows=self.m_max)
        self.packed, self.scales, self.t = synth.make_nvfp4_weight(wl, rows=self.n_max)

    def time(self, m: int, n: int) -> float:
        import oracle
        wl = self.wl
        m, n = min(m, self.m_max), min(n, self.n_max)
        t0 = time.perf_counter()
        oracle.convrot_linear(self.x[:m], wl.x_dtype, self.packed[:n], self.scales[:n], self.t,
                              wl.K, wl.out_dtype, wl.swiglu)
        return time.perf_counter() - t0


def calibrate(sample: OracleSample, target_s: float):
    """Grows (m, n) from a small probe until one oracle pass takes about target_s."""
    m, n = 64, 256
    t = sample.time(m, n)
    while t < 0.5 * target_s and (m < sample.m_max or n < sample.n_max):
        f = min(4.0, max(1.25, (target_s / max(t, 1e-3)) ** 0.5))
        m, n = int(min(sample.m_max, m * f)), int(min(sample.n_max, n * f))
        t = sample.time(m, n)
    return m, n, t


def cpu_baseline(wl: synth.Workload, budget_s: float):
    sample = OracleSample(wl, 4096, 16384)
    m, n, t = calibrate(sample, budget_s)
    ops = 2.0 * m * n * wl.K
    cores = len(os.sched_getaffinity(0))
    return {"value": ops / t / 1e12, "unit": "TOPS", "cores": cores, "kind": "oracle",
            "sample": f"{wl.name}: first {m} of {wl.M} tokens x first {n} of {wl.N} weight rows, "
                      f"full K={wl.K}, whole layer (decode, rotation, S8, int GEMM, dequant) in "
                      f"numpy FP64; {t:.2f} s; BLAS threads = cores, elementwise single-threaded",
            "seconds": t}


def reference_arm(args, wl):
    rank = int(os.environ.get("RANK", "0"))
    if rank != 0:
        return
    per_step = min(10.0, max(0.2, 150.0 / max(1, args.steps + args.warmup)))
    sample = OracleSample(wl, 2048, 8192)
    m_s, n_s, _ = calibrate(sample, per_step)
    for _ in range(args.warmup):
        sample.time(m_s, n_s)
    ts = [sample.time(m_s, n_s) for _ in range(args.steps)]
    ops = 2.0 * m_s * n_s * wl.K
    value = ops * len(ts) / sum(ts) / 1e12
    cores = len(os.sched_getaffinity(0))
    sample_txt = (f"{wl.name}: first {m_s} of {wl.M} tokens x first {n_s} of {wl.N} weight rows "
                  f"per step, full K={wl.K}, numpy FP64 oracle, whole layer")
    print(json.dumps({
        "impl": "reference", "metric": METRIC, "value": value, "unit": "TOPS",
        "n_gpus": args.gpus, "steps": args.steps, "warmup": args.warmup,
        "ms_per_step": 1e3 * sum(ts) / len(ts), "higher_is_better": True, "scaling": "weak",
        "vs_baseline": None, "dtype": "f64", "data": "synthetic",
        "config": bench_config(wl, args.overlap),
        "cpu_baseline": {"value": value, "unit": "TOPS", "cores": cores, "kind": "oracle",
                         "sample": sample_txt},
        "e2e": {"value": value, "unit": "TOPS", "h2d_bytes_per_step": 0, "d2h_bytes_per_step": 0},
    }), flush=True)


def bench_config(wl: synth.Workload, overlap: int) -> dict:
    """The workload description shared by both arms of the benchmark."""
    return {"workload": f"{wl.name} M={wl.M} K={wl.K} N={wl.N} {wl.x_dtype}->{wl.out_dtype}",
            "layer": ("NVFP4 weight prep on a second stream beside act rotation/S8, then GEMM, per step"
                      if overlap else "NVFP4 weight prep + act rotation/S8 + GEMM per step"),
            "l2": "flushed before every step (a write of twice the L2 size)",
            "parallelism": "single GPU",
            "arith": "S8 codes held as FP16 on tcgen05 kind::f16, exact int32 (one FP32 chunk per tile where "
                     "the rows' code-norm bounds allow it, else chunks of at most 1024); FP32 rotation"}


# ---------------------------------------------------------------- main
def main():
    ap = argparse.ArgumentParser()
    ap.add_argument("--gpus", type=int, default=1)
    ap.add_argument("--steps", type=int, default=20,
                    help="timed layers (a short run: the unthrottled regime the burst peak is measured in; "
                         "the sustained leg covers the power-capped one)")
    ap.add_argument("--warmup", type=int, default=5)
    ap.add_argument("--impl", choices=["ours", "reference"], default="ours")
    ap.add_argument("--workload", default="qkv", choices=sorted(synth.WORKLOADS))
    # 50 pipelined layers per timed run, as a DiT of 50 blocks runs them back to back; the
    # pipeline's fill (to the first output) is reported beside the per-step intervals
    ap.add_argument("--e2e-steps", type=int, default=50)
    ap.add_argument("--overlap", type=int, default=0,
                    help="1: the headline layer time runs the weight preparation on a second stream beside the "
                         "activation quantisation (per-kernel times come from a serial pass); 0: serial only")
    ap.add_argument("--secondary", default="ffn_down",
                    help="second workload timed in the same run ('' to skip)")
    ap.add_argument("--others", default="ffn_up,ragged,wide_k",
                    help="further workloads timed briefly in the same run ('' to skip)")
    ap.add_argument("--cpu-budget", type=float, default=12.0)
    ap.add_argument("--controls", type=int, default=1,
                    help="also time the W8A8 / resident-weight controls and pre-scale+bias (0 to skip)")
    ap.add_argument("--ffn-block", type=int, default=1,
                    help="also time the FFN block fc1 -> SwiGLU/rotate/S8 -> fc2 (0 to skip)")
    ap.add_argument("--sustained-s", type=float, default=4.0,
                    help="seconds of back-to-back layers for the sustained-clock leg (0 to skip)")
    ap.add_argument("--library", type=int, default=1,
                    help="also time the cuBLAS FP16 and cuBLASLt INT8 controls on the GEMM's shape (0 to skip)")
    ap.add_argument("--decode-probe", type=int, default=1,
                    help="also time the producer of a decode-inside-GEMM over the layer's schedule (0 to skip)")
    ap.add_argument("--rows", type=int, default=0,
                    help="truncate M to this many tokens (small profiling case; not a bench line)")
    args = ap.parse_args()
    if args.warmup < 3:
        raise SystemExit("--warmup must be >= 3")
    wl = synth.WORKLOADS[args.workload]
    if args.rows > 0:
        wl = dataclasses.replace(wl, name=f"{wl.name}_rows{args.rows}", M=min(wl.M, args.rows))
    if args.impl == "reference":
        reference_arm(args, wl)
        return

    world = int(os.environ.get("WORLD_SIZE", "1"))
    single_gpu_guard(args.gpus, world)

    import torch

    import __graft_entry__
    __graft_entry__.build()
    torch.cuda.set_device(0)
    dev = torch.device("cuda", 0)
    props = torch.cuda.get_device_properties(dev)
    sm_count = int(props.multi_processor_count)
    l2 = int(getattr(props, "L2_cache_size", 128 << 20))
    flush_buf = torch.empty(2 * l2 // 4 + 1024, dtype=torch.float32, device=dev)

    def flush():
        flush_buf.fill_(1.0)

    bus = getattr(props, "pci_bus_id", None)
    if isinstance(bus, int):
        bus = None
    peaks, peaks_src = load_peaks()
    hbm = float(peaks.get("hbm_gbs", FALLBACK_PEAKS["hbm_gbs"]))
    peak_burst = float(peaks.get("bf16_tflops", FALLBACK_PEAKS["bf16_tflops"]))
    peak_sust = float(peaks.get("bf16_tflops_sustained", FALLBACK_PEAKS["bf16_tflops_sustained"]))

    layer = Layer(wl, dev)
    sz = layer.sz
    r = time_layer(layer, args.steps, args.warmup, 1, flush, None if args.overlap else ClockSampler(bus))
    serial_ms = r["total_ms"] / args.steps
    if args.overlap:
        ro = time_layer_overlapped(layer, args.steps, args.warmup, 1, flush, ClockSampler(bus))
        t_tot = ro["total_ms"]
        clocks = ro["clocks"]
    else:
        t_tot = r["total_ms"]
        clocks = r["clocks"]
    ms_step = t_tot / args.steps
    value = aggregate_tops(sz["ops"], args.steps, t_tot, 1)
    g_ms = statistics.mean(r["gemm_ms"])
    a_ms = statistics.mean(r["act_ms"])
    w_ms = statistics.mean(r["weight_ms"])
    achieved = sz["gemm_flops"] / (g_ms / 1e3) / 1e12
    gemm_src = os.path.join(ROOT, "rotated_w4a8_int8_gb300", "csrc", "gemm.cu")
    traffic = GEMM_TRAFFIC["bytes"] if GEMM_TRAFFIC["sha256_16"] == code_sha16(gemm_src) else None

    def quant_kernel(us, alg, moved):
        gbs = alg / (us / 1e6) / 1e9
        return {"us": us, "alg_bytes": alg, "gbs": gbs, "hbm_frac": gbs / hbm,
                "moved_bytes": moved, "moved_gbs": moved / (us / 1e6) / 1e9,
                "moved_frac": moved / (us / 1e6) / 1e9 / hbm}

    kernels = {
        "prepare_weight": quant_kernel(1e3 * w_ms, sz["w_alg"], sz["w_bytes"]),
        "quant_act": quant_kernel(1e3 * a_ms, sz["act_alg"], sz["act_bytes"]),
        "gemm": {"ms": g_ms, "tflops": achieved},
    }
    # Decode inside the GEMM: a GEMM whose producers decode, rotate and quantise
    # the NVFP4 weight itself has to redo that work for every 256-row strip of
    # tokens that meets a weight tile (no strip can keep a 256 x K_p tile of
    # codes resident).  At the whole-GPU rate the weight kernel measured just
    # now, that work alone takes strips x its time, with perfect overlap and no
    # interference with the MMAs assumed, plus a scales-only pre-pass.
    # Per tile: one CTA pair (2 SMs) would prepare a work item's 256 weight
    # rows itself; at the measured per-SM rate of the weight kernel that
    # takes tile_weight_us, against tile_mma_us of GEMM time per item.
    strips = -(-wl.M // 256)
    items = strips * -(-wl.N // 256)
    pairs = min(sm_count // 2, items)
    tile_weight_us = 1e3 * w_ms * sm_count / wl.N * 256 / 2
    tile_mma_us = 1e3 * g_ms * pairs / items
    decode_in_gemm = {"m_strips": strips, "redone_weight_work_ms": strips * w_ms,
                      "vs_layer_ms": ms_step,
                      "tile_weight_us": tile_weight_us, "tile_mma_us": tile_mma_us,
                      "tile_ratio": tile_weight_us / tile_mma_us,
                      "note": "lower bound on a decode-inside-GEMM layer from this run's weight-kernel time; "
                              "tile_ratio: one CTA pair preparing a work item's 256 weight rows at the weight "
                              "kernel's per-SM rate, over the GEMM's time per work item"}
    if args.decode_probe:
        decode_in_gemm["producer_probe"] = time_decode_probe(layer, strips, g_ms, args.warmup)

    # end-to-end through the public API with host buffers
    e2e_value = e2e_ms = link = intervals = e2e_runs = None
    h2d = layer.in_bytes
    d2h = layer.y.numel() * layer.y.element_size()
    if args.e2e_steps > 0:
        e2e_ms, h2d, d2h, link, intervals, e2e_runs = time_e2e(layer, args.e2e_steps, 3, 1)
        e2e_value = aggregate_tops(sz["ops"], args.e2e_steps, e2e_ms, 1)
    sustained = None
    if args.sustained_s > 0:
        sustained = time_sustained(layer, args.sustained_s, ms_step, bus, sm_count)
        sustained["gemm_frac_of_sustained_peak"] = sustained["gemm_tflops"] / peak_sust
    if layer.cr.device_error() != 0:
        raise SystemExit("device timeout reported by the GEMM")
    library = time_library_controls(layer, flush, args.warmup) if args.library else None
    del layer
    torch.cuda.empty_cache()

    secondary = None
    if args.secondary:
        wl2 = synth.WORKLOADS[args.secondary]
        l2y = Layer(wl2, dev)
        r2 = time_layer(l2y, max(10, args.steps // 4), args.warmup, 1, flush)
        s2 = l2y.sz
        ms2 = r2["total_ms"] / len(r2["step_ms"])
        g2 = statistics.mean(r2["gemm_ms"])
        a2 = 1e3 * statistics.mean(r2["act_ms"])
        w2 = 1e3 * statistics.mean(r2["weight_ms"])
        secondary = {"workload": f"{wl2.name} M={wl2.M} K={wl2.K} (SwiGLU input {wl2.k_in}) N={wl2.N}"
                     if wl2.swiglu else f"{wl2.name} M={wl2.M} K={wl2.K} N={wl2.N}",
                     "ms_per_layer": ms2, "eff_tops": s2["ops"] / (ms2 / 1e3) / 1e12,
                     "gemm_ms": g2, "gemm_tflops": s2["gemm_flops"] / (g2 / 1e3) / 1e12,
                     "quant_act": quant_kernel(a2, s2["act_alg"], s2["act_bytes"]),
                     "prepare_weight": quant_kernel(w2, s2["w_alg"], s2["w_bytes"]),
                     "pages_a40_ms": 19.49}
        del l2y
        torch.cuda.empty_cache()

    others = {}
    for name in [n for n in args.others.split(",") if n]:
        wlo = synth.WORKLOADS[name]
        lo = Layer(wlo, dev)
        ro = time_layer(lo, 20, args.warmup, 1, flush)
        so = lo.sz
        mso = ro["total_ms"] / len(ro["step_ms"])
        ao = 1e3 * statistics.mean(ro["act_ms"])
        wo = 1e3 * statistics.mean(ro["weight_ms"])
        others[name] = {"workload": f"M={wlo.M} K={wlo.K} N={wlo.N} {wlo.x_dtype}->{wlo.out_dtype}",
                        "ms_per_layer": mso, "eff_tops": so["ops"] / (mso / 1e3) / 1e12,
                        "gemm_tflops": so["gemm_flops"] / (statistics.mean(ro["gemm_ms"]) / 1e3) / 1e12,
                        "quant_act_us": ao, "quant_act_hbm_frac": so["act_alg"] / (ao / 1e6) / 1e9 / hbm,
                        "prepare_weight_us": wo, "prepare_weight_hbm_frac": so["w_alg"] / (wo / 1e6) / 1e9 / hbm}
        del lo
        torch.cuda.empty_cache()

    ffn = None
    if args.ffn_block:
        ffn = time_ffn_block(dev, 1, flush, args.warmup)
    controls = None
    if args.controls:
        controls = time_controls(wl, dev, 1, flush, args.warmup)

    cpu = None
    if args.cpu_budget > 0:
        cpu = cpu_baseline(wl, args.cpu_budget)

    mhz = (clocks or {}).get("sm_mhz")
    roofline = {"bound": "tensor", "achieved": achieved, "peak": peak_burst, "unit": "TFLOP/s",
                "frac": achieved / peak_burst, "traffic": traffic,
                "kernel": "gemm_kernel (tcgen05 kind::f16)",
                "peak_source": f"{peaks_src} bf16_tflops (burst: the GEMM is timed in short steps; "
                               f"FP16 runs at the BF16 rate)",
                "work_per_launch": f"2*M*N*K_p = {sz['gemm_flops']:.4e} FLOP",
                "traffic_source": "ncu dram__bytes_read.sum + dram__bytes_write.sum, one full-size launch"}
    if mhz:
        pipe = tensor_pipe_peak(sm_count, mhz)
        roofline["tensor_pipe_peak_at_clock"] = pipe
        roofline["tensor_pipe_frac"] = achieved / pipe
    if library and "tflops" in library.get("cublas_fp16", {}):
        roofline["vs_cublas_fp16_same_shape"] = achieved / library["cublas_fp16"]["tflops"]
    if library and "tops" in library.get("int8_mm", {}):
        roofline["int8_library_tops_same_shape"] = library["int8_mm"]["tops"]
        roofline["vs_int8_library_same_shape"] = achieved / library["int8_mm"]["tops"]
    if library and "tops" in library.get("int8_mma_sync", {}):
        # the INT8 tensor rate of this GPU measured on the warp-level instruction
        roofline["int8_mma_sync_tops"] = library["int8_mma_sync"]["tops"]
        roofline["vs_int8_mma_sync"] = achieved / library["int8_mma_sync"]["tops"]

    line = {
        "metric": METRIC, "value": value, "unit": "TOPS", "n_gpus": 1, "steps": args.steps,
        "warmup": args.warmup, "ms_per_step": ms_step, "higher_is_better": True,
        "scaling": "weak", "vs_baseline": value / (sz["ops"] / (PAGES_QKV_MS / 1e3) / 1e12),
        "dtype": "s8", "data": "synthetic",
        "config": bench_config(wl, args.overlap),
        "ms_per_layer": ms_step,
        "ms_per_layer_serial": serial_ms,
        "kernels": kernels,
        "decode_inside_gemm_bound": decode_in_gemm,
        "roofline": roofline,
        "hbm_peak_gbs": hbm,
        "hbm_note": ("quant kernels: hbm_frac on algorithmic bytes with 1-byte S8 codes; moved_* on the bytes "
                     "actually moved (codes held as FP16 for the GEMM)"),
        "e2e": {"value": e2e_value, "unit": "TOPS", "h2d_bytes_per_step": h2d,
                "d2h_bytes_per_step": d2h, "pipelined": "streams: copy-in, kernels, copy-out split over 2 copy streams",
                "ms_per_step": e2e_ms / args.e2e_steps if e2e_ms else None,
                "statistic": f"median of {E2E_RUNS} timed runs of e2e_steps pipelined steps",
                "runs_ms_per_step": e2e_runs,
                "host_link_gbs": link,
                # time between consecutive steps' output completions: a slow box shows here
                # whether every step or a few are slow
                "step_interval_ms": intervals},
        "gpu_launches": 3 * args.steps,
        "clocks": clocks,
        "sustained": sustained,
        "library": library,
        "cpu_baseline": cpu,
        "secondary": secondary,
        "others": others,
        "ffn_block": ffn,
        "controls": controls,
        "vs_baseline_note": "value / the pages' A40 QKV layer (25.08 ms = 184.3 TOPS): context only",
    }
    print(json.dumps(line), flush=True)


if __name__ == "__main__":
    main()
