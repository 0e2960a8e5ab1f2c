#!/usr/bin/env python
"""Benchmark of the POP pruned gated-MLP FFN on GB300.

One step = one full inference session of an FFN stack: prefill of every layer's prompt (dense
FFN on the tensor cores, sum of z^2, R/C/P partition), then T decode steps that run every layer
(gate/up over R u C, candidate top-k, down over R and the selected candidates). Default workload:
LLaMA-2-7B FFN shape (D=4096, D_FF=11008), B=1, 2048 prompt tokens, r=0.299, gamma=0.1, 256
decode steps, on 4 independent layer copies (1.08 GB of weights, more than 3x the 129 MB L2, so
consecutive decode steps stream weights from HBM).

value = decode tokens per second per FFN layer = B * T * layers / (session time, prefill
included). Inputs are already in HBM when timing starts; `e2e` repeats the session through the
same public API with inputs in pinned host memory and outputs copied back inside the timed region.

`--impl reference` times the CPU oracle (float64 numpy) on the host cores instead, on a bounded
sample of the same workload, extrapolated to the same unit.

Multi-GPU (`torchrun --nproc-per-node N bench.py --gpus N`): the path has no exchange step, so
every rank runs an independent replica; the time is the maximum over ranks and the value the
sum of all ranks' tokens over that time (weak scaling).
"""
from __future__ import annotations

import argparse
import csv
import io
import json
import os
import statistics
import subprocess
import sys
import threading
import time

ROOT = os.path.dirname(os.path.abspath(__file__))
if ROOT not in sys.path:
    sys.path.insert(0, ROOT)

WORKLOADS = {
    # D, D_FF, rate, gamma, batch, prompt tokens (all sequences), decode steps, period, layers, prefill chunk
    "llama2-7b-ffn-b1": dict(D=4096, N=11008, r=0.299, gamma=0.1, B=1, M=2048, T=256, period=1, layers=4,
                             chunk=2048),
    "llama2-7b-ffn-b16": dict(D=4096, N=11008, r=0.5, gamma=0.1, B=16, M=16 * 1024, T=512, period=1, layers=4,
                              chunk=4096),
    "llama-70b-ffn-b64-p16": dict(D=8192, N=28672, r=0.5, gamma=0.1, B=64, M=64 * 512, T=1024, period=16,
                                  layers=1, chunk=8192),
    # the same with the periodic skip variant: between updates gate/up only over R and the held selection
    "llama-70b-ffn-b64-p16-skip": dict(D=8192, N=28672, r=0.5, gamma=0.1, B=64, M=64 * 512, T=1024, period=16,
                                       layers=1, chunk=8192, skip=True),
    # the POP notes' ablation comparators on the 7B B=1 workload: a static mask (gamma = 0: no
    # candidates, the prefill's top-keep every step) and full per-step re-evaluation (gamma >=
    # max(r, 1 - r): every channel a candidate, a top-keep over all of them every step)
    "llama2-7b-ffn-b1-static": dict(D=4096, N=11008, r=0.299, gamma=0.0, B=1, M=2048, T=256, period=1, layers=4,
                                    chunk=2048),
    "llama2-7b-ffn-b1-fulldyn": dict(D=4096, N=11008, r=0.299, gamma=0.701, B=1, M=2048, T=256, period=1,
                                     layers=4, chunk=2048),
    # MoE layer: 8 experts of D=4096, D_FF=14336, top-2 routing, prompt of 8 sequences x 512 tokens
    "moe-8x4096x14336-b32": dict(D=4096, N=14336, r=0.3, gamma=0.1, B=32, M=8 * 512, T=128, period=1, layers=1,
                                 chunk=2048, experts=8),
}
METRIC = "pruned-FFN decode tokens/s and HBM GB/s vs GB300 peak, LLaMA-7B FFN, B=1/16"
# Per-kernel durations come from a separate pass after the timed region in which every decode step
# records CUDA events between its kernels. An event between two kernels ends the programmatic
# overlap of the next kernel's launch with the previous one's tail, so the timed region itself
# records none; the profiled pass gives each kernel's isolated duration.
PROFILE_SESSIONS = 1
UNIT = "tokens/s"


def measured_peaks():
    try:
        with open(os.path.join(ROOT, "MEASURED_PEAKS.json")) as f:
            p = json.load(f)
        return float(p["hbm_gbs"]), "measured"
    except Exception:
        return 6800.0, "fallback"


def touched_bytes(c, D, wl=None):
    """Algorithmic weight bytes of one decode step: gate+up rows over R u C, down columns over R u S.
    With the periodic skip variant the gate/up rows are R u C on update steps and R u S in between:
    the average over a period."""
    rows = c.n_R + c.n_C
    if wl is not None and wl.get("skip") and wl["period"] > 1 and c.n_C > 0:
        P = wl["period"]
        rows = ((c.n_R + c.n_C) + (P - 1) * (c.n_R + c.k)) / P
    gateup = 2 * rows * D * 2
    down = c.keep * D * 2
    return gateup, down


# ------------------------------------------------------------------ distributed helpers

def dist_info():
    return int(os.environ.get("RANK", "0")), int(os.environ.get("WORLD_SIZE", "1")), \
        int(os.environ.get("LOCAL_RANK", "0"))


def aggregate(elapsed_s: float, units: float, device=None):
    """Max of the elapsed times and sum of the units over all ranks (no-op with one process)."""
    import torch
    import torch.distributed as dist
    if not (dist.is_available() and dist.is_initialized()):
        return elapsed_s, units
    t = torch.tensor([elapsed_s], dtype=torch.float64, device=device)
    u = torch.tensor([units], dtype=torch.float64, device=device)
    dist.all_reduce(t, op=dist.ReduceOp.MAX)
    dist.all_reduce(u, op=dist.ReduceOp.SUM)
    return float(t.item()), float(u.item())


def barrier():
    import torch.distributed as dist
    if dist.is_available() and dist.is_initialized():
        dist.barrier()


# ------------------------------------------------------------------ clocks

CLOCK_FIELDS = ("index,clocks.sm,clocks.max.sm,power.draw,clocks_event_reasons.active,"
                "clocks_event_reasons.hw_slowdown,clocks_event_reasons.hw_thermal_slowdown,"
                "clocks_event_reasons.sw_thermal_slowdown,clocks_event_reasons.sw_power_cap")


class ClockSampler:
    """Samples SM clocks and throttle reasons with nvidia-smi while the timed region runs."""

    def __init__(self, device_index: int):
        import torch
        try:
            self.gpu = "GPU-" + str(torch.cuda.get_device_properties(device_index).uuid)
        except Exception:
            self.gpu = str(device_index)
        self.proc = None
        self.out = b""

    def __enter__(self):
        try:
            self.proc = subprocess.Popen(["nvidia-smi", f"--id={self.gpu}", f"--query-gpu={CLOCK_FIELDS}",
                                          "--format=csv,noheader,nounits", "-lms", "200"],
                                         stdout=subprocess.PIPE, stderr=subprocess.DEVNULL)
            self._t = threading.Thread(target=self._read, daemon=True)
            self._t.start()
        except Exception:
            self.proc = None
        return self

    def _read(self):
        self.out = self.proc.stdout.read()

    def __exit__(self, *a):
        if self.proc is not None:
            self.proc.terminate()
            try:
                self.proc.wait(timeout=5)
            except Exception:
                self.proc.kill()
            self._t.join(timeout=5)

    def summary(self):
        rows = list(csv.reader(io.StringIO(self.out.decode(errors="replace"))))
        sm, smax, reasons = [], None, set()
        names = ["hw_slowdown", "hw_thermal_slowdown", "sw_thermal_slowdown", "sw_power_cap"]
        for r in rows:
            if len(r) < 9:
                continue
            try:
                sm.append(float(r[1]))
                smax = float(r[2])
            except ValueError:
                continue
            for n, v in zip(names, r[5:9]):
                if v.strip().lower().startswith("active"):
                    reasons.add(n)
        if not sm:
            return {"sm_mhz": None, "sm_max_mhz": None, "reasons": [], "samples": 0}
        return {"sm_mhz": statistics.median(sm), "sm_max_mhz": smax, "reasons": sorted(reasons),
                "samples": len(sm)}


# ------------------------------------------------------------------ GPU arm

def prefill_launches(chunks, max_batch):
    return 3 * chunks + 1 + (2 if max_batch > 1 else 0)


def decode_launches(c, B):
    return (2 + (1 if c.n_C > 8192 else 0)) if B == 1 else 2


class Stack:
    """`layers` independent POP FFN layers of one workload, with their inputs resident in HBM."""

    def __init__(self, wl, seed=0):
        import numpy as np
        import torch

        import online_structured_ffn_gb300 as pop
        import synth
        self.wl, self.pop, self.torch = wl, pop, torch
        dev = torch.device("cuda", torch.cuda.current_device())
        self.dev = dev
        D, N, B, M, T, Lyr = wl["D"], wl["N"], wl["B"], wl["M"], wl["T"], wl["layers"]

        def up(a):
            return torch.from_numpy(np.ascontiguousarray(a).view(np.int16)).to(dev).view(torch.bfloat16)

        self.ffn = []
        sc = synth.dim_scales(seed, D)
        self.X, self.Y = [], []
        for l in range(Lyr):
            Wg, W1, W2 = synth.ffn_weights(seed, D, N, layer=l)
            tg, t1, t2 = up(Wg), up(W1), up(W2)
            del Wg, W1, W2
            f = pop.PopFFN(tg, t1, t2, r=wl["r"], gamma=wl["gamma"], period=wl["period"], max_batch=B,
                           max_prefill_tokens=wl["chunk"], out_f32=True, skip=wl.get("skip", False))
            torch.cuda.synchronize()
            del tg, t1, t2
            self.ffn.append(f)
            self.X.append(up(synth.prompt(seed, M, sc, layer=l)))
            self.Y.append(torch.empty((M, D), dtype=torch.float32, device=dev))
        xs = np.stack([np.stack([synth.decode_input(seed, t, B, sc, layer=l) for l in range(Lyr)])
                       for t in range(T)])
        self.x = up(xs)  # [T, layers, B, D]
        self.y = torch.empty((T, Lyr, B, D), dtype=torch.float32, device=dev)
        self.counts = self.ffn[0].counts
        self.chunks = (M + wl["chunk"] - 1) // wl["chunk"]

    def launches_per_session(self):
        # prefill: per chunk gate/up GEMM + sum fold + down GEMM, then the partition kernel (and at
        # B > 1 the two slab builders); decode at B = 1: gate/up with the top-k inside (+ a separate
        # top-k when |C| > 8192) and the tiled down projection; at B > 1: the gate/up GEMM, then the
        # down GEMM with the selection inside
        wl, c = self.wl, self.counts
        T, B = wl["T"], wl["B"]
        decode = decode_launches(c, B) * T
        if wl.get("skip") and wl["period"] > 1 and c.n_C > 0:
            updates = (T + wl["period"] - 1) // wl["period"]
            if B > 1:
                decode += updates  # the slab of [C[S] | R] rebuilt after each update
            elif c.n_C > 8192:
                decode -= T - updates  # steps between updates need no separate top-k
        per_layer = prefill_launches(self.chunks, B) + decode
        return per_layer * wl["layers"]

    def session(self, dec_events=None):
        pop, torch = self.pop, self.torch
        st = torch.cuda.current_stream().cuda_stream
        B, T = self.wl["B"], self.wl["T"]
        for l, f in enumerate(self.ffn):
            pop.pop_prefill_partition(f.handle, self.X[l].data_ptr(), self.X[l].shape[0], self.Y[l].data_ptr(), st)
        if dec_events is not None:
            dec_events[0].record()
        handles = [f.handle for f in self.ffn]
        lib = pop.load_library()
        xp, yp = self.x.data_ptr(), self.y.data_ptr()
        xstride = B * self.wl["D"] * 2
        ystride = B * self.wl["D"] * 4
        i = 0
        for t in range(T):
            for h in handles:
                s = lib.pop_decode_step(h, xp + i * xstride, B, yp + i * ystride, st)
                if s:
                    pop._check(s, h)
                i += 1
        if dec_events is not None:
            dec_events[1].record()

    def session_e2e(self, hX, hx, hY, hy):
        """The same session with inputs in pinned host memory and every output copied back, all
        timed (see overlapped_copies)."""
        pop, torch = self.pop, self.torch
        cs = torch.cuda.current_stream()
        st = cs.cuda_stream
        B, T = self.wl["B"], self.wl["T"]
        lib = pop.load_library()
        with OverlappedCopies(torch, cs) as oc:
            ready = [oc.up(self.X[l], hX[l]) for l in range(len(self.ffn))]
            for l, f in enumerate(self.ffn):
                cs.wait_event(ready[l])
                pop.pop_prefill_partition(f.handle, self.X[l].data_ptr(), self.X[l].shape[0], self.Y[l].data_ptr(), st)
                oc.down(hY[l], self.Y[l])
            for t in range(T):
                self.x[t].copy_(hx[t], non_blocking=True)  # each step's input right before the step
                for l, f in enumerate(self.ffn):
                    s = lib.pop_decode_step(f.handle, self.x[t, l].data_ptr(), B, self.y[t, l].data_ptr(), st)
                    if s:
                        pop._check(s, f.handle)
                oc.down(hy[t], self.y[t])

    def close(self):
        for f in self.ffn:
            f.close()


class MoeStack:
    """One MoE layer (top-2 routing over `experts` POP-pruned experts) with its inputs resident in HBM."""

    def __init__(self, wl, seed=0):
        import numpy as np
        import torch

        import online_structured_ffn_gb300 as pop
        import synth
        self.wl, self.pop, self.torch = wl, pop, torch
        dev = torch.device("cuda", torch.cuda.current_device())
        D, N, B, M, T, E = wl["D"], wl["N"], wl["B"], wl["M"], wl["T"], wl["experts"]

        def up(a):
            return torch.from_numpy(np.ascontiguousarray(a).view(np.int16)).to(dev).view(torch.bfloat16)

        def f32(a):
            return torch.from_numpy(np.ascontiguousarray(a, dtype=np.float32)).to(dev)

        ws = [[], [], []]
        for e in range(E):
            for i, w in enumerate(synth.ffn_weights(seed, D, N, layer=e)):
                ws[i].append(up(w))
        self.moe = pop.PopMoE(ws[0], ws[1], ws[2], r=wl["r"], gamma=wl["gamma"], period=wl["period"], max_batch=B,
                              max_prefill_tokens=wl["chunk"], out_f32=True)
        torch.cuda.synchronize()
        del ws
        self.ffn = self.moe.experts
        self.counts = self.moe.counts
        sc = synth.dim_scales(seed, D)
        self.X = [up(synth.prompt(seed, M, sc))]
        self.Lp = f32(synth.router_logits(seed, M, E))
        self.Y = [torch.empty((M, D), dtype=torch.float32, device=dev)]
        self.x = up(np.stack([synth.decode_input(seed, t, B, sc)[None] for t in range(T)]))  # [T, 1, B, D]
        self.L = f32(np.stack([synth.router_logits(seed, B, E, step=t) for t in range(T)]))  # [T, B, E]
        self.y = torch.empty((T, 1, B, D), dtype=torch.float32, device=dev)
        # route the prompt once, so the experts' token counts (and the launch count) are known
        self.moe.prefill_partition(self.X[0], self.Lp, self.Y[0])
        self.prompt_counts = self.moe.token_counts()

    def launches_per_session(self):
        import numpy as np
        wl = self.wl
        E = wl["experts"]
        n = 3 + 1  # route top-2, token slots, gather; combine
        for c in self.prompt_counts:
            n += prefill_launches(int(np.ceil(c / wl["chunk"])), wl["B"]) if c else 1 + (2 if wl["B"] > 1 else 0)
        n += wl["T"] * (2 + E * decode_launches(self.counts, wl["B"]))
        return n

    def session(self, dec_events=None):
        pop, torch = self.pop, self.torch
        st = torch.cuda.current_stream().cuda_stream
        B, T, D, E = self.wl["B"], self.wl["T"], self.wl["D"], self.wl["experts"]
        lib = pop.load_library()
        h = self.moe.handle
        s = lib.pop_moe_prefill_partition(h, self.X[0].data_ptr(), self.Lp.data_ptr(), self.X[0].shape[0],
                                          self.Y[0].data_ptr(), st)
        if s:
            pop._check_moe(s, h)
        if dec_events is not None:
            dec_events[0].record()
        xp, lp, yp = self.x.data_ptr(), self.L.data_ptr(), self.y.data_ptr()
        for t in range(T):
            s = lib.pop_moe_decode_step(h, xp + t * B * D * 2, lp + t * B * E * 4, B, yp + t * B * D * 4, st)
            if s:
                pop._check_moe(s, h)
        if dec_events is not None:
            dec_events[1].record()

    def session_e2e(self, hX, hx, hY, hy):
        pop, torch = self.pop, self.torch
        cs = torch.cuda.current_stream()
        st = cs.cuda_stream
        B, T = self.wl["B"], self.wl["T"]
        lib = pop.load_library()
        with OverlappedCopies(torch, cs) as oc:
            self.X[0].copy_(hX[0], non_blocking=True)
            self.Lp.copy_(self.hLp, non_blocking=True)
            self.moe.prefill_partition(self.X[0], self.Lp, self.Y[0])
            oc.down(hY[0], self.Y[0])
            for t in range(T):
                self.x[t].copy_(hx[t], non_blocking=True)  # each step's input right before the step
                self.L[t].copy_(self.hL[t], non_blocking=True)
                s = lib.pop_moe_decode_step(self.moe.handle, self.x[t].data_ptr(), self.L[t].data_ptr(), B,
                                            self.y[t].data_ptr(), st)
                if s:
                    pop._check_moe(s, self.moe.handle)
                oc.down(hy[t], self.y[t])

    def e2e_extra_h2d(self):
        """Pinned host copies of the router logits; returns their bytes per session."""
        self.hLp = self.Lp.cpu().pin_memory()
        self.hL = self.L.cpu().pin_memory()
        return self.hLp.numel() * 4 + self.hL.numel() * 4

    def check(self):
        self.moe.check()

    def set_profiling(self, on):
        # the experts run one after another while their kernels are timed one by one
        self.moe.set_concurrent(not on)

    def close(self):
        self.moe.close()


class OverlappedCopies:
    """Host<->device copies of an end-to-end session on two side streams, ordered against the
    compute stream by events: inputs known up front (the prompts) go up while earlier work runs,
    and every result goes down once the compute stream has produced it, while later work runs. A
    decode step's input stays on the compute stream right before the step, since in a model it
    depends on the previous step's output. Leaving the block waits for every copy, so the next
    session's kernels never overwrite a buffer that is still being copied out."""

    _streams = {}

    def __init__(self, torch, compute_stream):
        self.torch, self.cs = torch, compute_stream
        dev = compute_stream.device
        if dev not in OverlappedCopies._streams:
            OverlappedCopies._streams[dev] = (torch.cuda.Stream(device=dev), torch.cuda.Stream(device=dev))
        self.up_s, self.down_s = OverlappedCopies._streams[dev]

    def __enter__(self):
        # the side streams start after the work already queued on the compute stream
        ev = self.torch.cuda.Event()
        ev.record(self.cs)
        self.up_s.wait_event(ev)
        self.down_s.wait_event(ev)
        return self

    def up(self, dst, src):
        """Copies src (pinned host) to dst on the upload stream; returns the event that marks it."""
        with self.torch.cuda.stream(self.up_s):
            dst.copy_(src, non_blocking=True)
        ev = self.torch.cuda.Event()
        ev.record(self.up_s)
        return ev

    def down(self, dst, src):
        """Copies src to dst (pinned host) on the download stream once the compute stream's work so
        far is done."""
        ev = self.torch.cuda.Event()
        ev.record(self.cs)
        self.down_s.wait_event(ev)
        with self.torch.cuda.stream(self.down_s):
            dst.copy_(src, non_blocking=True)

    def __exit__(self, *exc):
        self.cs.synchronize()
        self.up_s.synchronize()
        self.down_s.synchronize()
        return False


def make_stack(wl):
    return MoeStack(wl) if wl.get("experts") else Stack(wl)


def run_gpu(wl_name, steps, warmup, with_e2e=True, with_clocks=True):
    import torch
    wl = WORKLOADS[wl_name]
    rank, world, local = dist_info()
    stack = make_stack(wl)
    for f in stack.ffn:
        f.check()
    for _ in range(warmup):
        stack.session()
    torch.cuda.synchronize()
    ev0, ev1 = torch.cuda.Event(enable_timing=True), torch.cuda.Event(enable_timing=True)
    dec = [(torch.cuda.Event(enable_timing=True), torch.cuda.Event(enable_timing=True)) for _ in range(steps)]
    sampler = ClockSampler(torch.cuda.current_device()) if with_clocks else None
    barrier()
    torch.cuda.synchronize()
    if sampler:
        sampler.__enter__()
    ev0.record()
    for k in range(steps):
        stack.session(dec[k])
    ev1.record()
    torch.cuda.synchronize()
    if sampler:
        sampler.__exit__()
    barrier()
    elapsed = ev0.elapsed_time(ev1) / 1e3
    dec_s = sum(a.elapsed_time(b) for a, b in dec) / 1e3
    if hasattr(stack, "check"):
        stack.check()
    for f in stack.ffn:
        f.check()
    # profiled pass: the same sessions with events between the kernels of every decode step
    if hasattr(stack, "set_profiling"):
        stack.set_profiling(True)
    for f in stack.ffn:
        f.profile(1)
    for _ in range(PROFILE_SESSIONS):
        stack.session()
    torch.cuda.synchronize()
    prof = [f.profile_read() for f in stack.ffn]
    for f in stack.ffn:
        f.profile(False)
        f.check()
    if hasattr(stack, "set_profiling"):
        stack.set_profiling(False)
    B, T, Lyr = wl["B"], wl["T"], wl["layers"]
    dense_us = dense_step_us(stack) if not wl.get("experts") else None
    units = B * T * Lyr * steps
    g_elapsed, g_units = aggregate(elapsed, units, device=torch.device("cuda", torch.cuda.current_device()))
    ksum = [sum(p[0][i] for p in prof) for i in range(4)]
    nsteps = sum(p[1] for p in prof)
    c = stack.counts
    gu_bytes, dn_bytes = touched_bytes(c, wl["D"], wl)
    nexp = wl.get("experts", 1)  # every expert streams its weights every step
    peak, peak_kind = measured_peaks()
    gu_ms = ksum[0] / max(nsteps, 1)
    roof_bytes = gu_bytes
    dec_step_s = dec_s / (T * Lyr * steps)
    res = dict(
        value=g_units / g_elapsed, elapsed=g_elapsed, units=g_units, ms_per_step=1e3 * g_elapsed / steps,
        decode_only_tokens_per_s=B * T * Lyr * steps / dec_s,
        decode_step_us=1e6 * dec_step_s, dense_step_us=dense_us,
        prefill_ms_per_layer=1e3 * (elapsed - dec_s) / (steps * Lyr),
        kernel_us={n: 1e3 * ksum[i] / max(nsteps, 1) for i, n in enumerate(("gateup", "select", "down", "reduce"))},
        roof_bytes=roof_bytes,
        gateup_gbs=roof_bytes / (gu_ms * 1e-3) / 1e9,
        peak=peak, peak_kind=peak_kind,
        step_gbs=nexp * (gu_bytes + dn_bytes) / dec_step_s / 1e9, experts=nexp,
        gu_bytes=gu_bytes, dn_bytes=dn_bytes, counts=c.as_dict(),
        launches=stack.launches_per_session() * steps,
        clocks=sampler.summary() if sampler else None,
    )
    if with_e2e:
        res["e2e"] = run_e2e(stack, max(1, min(steps, 5)))
    stack.close()
    del stack
    torch.cuda.empty_cache()
    return res


def dense_step_us(stack, reps=2):
    """The dense FFN (pop_ffn_dense_ref: every channel, the same kernels' dense path) on the same
    decode inputs, through every layer: microseconds per decode step, for comparison."""
    import torch
    pop, wl = stack.pop, stack.wl
    lib = pop.load_library()
    st = torch.cuda.current_stream().cuda_stream
    B, T, D = wl["B"], wl["T"], wl["D"]
    xs, ys = stack.x.view(-1, D), stack.y.view(-1, D)

    def one():
        i = 0
        for _ in range(T):
            for f in stack.ffn:
                s = lib.pop_ffn_dense_ref(f.handle, xs[i * B].data_ptr(), B, ys[i * B].data_ptr(), st)
                if s:
                    pop._check(s, f.handle)
                i += 1
    one()  # warm
    torch.cuda.synchronize()
    e0, e1 = torch.cuda.Event(enable_timing=True), torch.cuda.Event(enable_timing=True)
    e0.record()
    for _ in range(reps):
        one()
    e1.record()
    torch.cuda.synchronize()
    return 1e3 * e0.elapsed_time(e1) / (reps * T * len(stack.ffn))


def run_e2e(stack, steps):
    import torch
    wl = stack.wl
    hX = [x.cpu().pin_memory() for x in stack.X]
    hY = [torch.empty(y.shape, dtype=y.dtype).pin_memory() for y in stack.Y]
    hx = stack.x.cpu().pin_memory()
    hy = torch.empty(stack.y.shape, dtype=stack.y.dtype).pin_memory()
    extra = stack.e2e_extra_h2d() if hasattr(stack, "e2e_extra_h2d") else 0
    stack.session_e2e(hX, hx, hY, hy)  # warm
    barrier()
    torch.cuda.synchronize()
    t0 = time.perf_counter()
    for _ in range(steps):
        stack.session_e2e(hX, hx, hY, hy)
    torch.cuda.synchronize()
    el = time.perf_counter() - t0
    barrier()
    units = wl["B"] * wl["T"] * wl["layers"] * steps
    g_el, g_units = aggregate(el, units, device=torch.device("cuda", torch.cuda.current_device()))
    h2d = sum(x.numel() * x.element_size() for x in hX) + hx.numel() * hx.element_size() + extra
    d2h = sum(y.numel() * y.element_size() for y in hY) + hy.numel() * hy.element_size()
    return {"value": g_units / g_el, "unit": UNIT, "h2d_bytes_per_step": int(h2d), "d2h_bytes_per_step": int(d2h),
            "steps": steps}


# ------------------------------------------------------------------ CPU oracle arm

# A prompt whose float64 prefill exceeds this many flops is timed at two sizes and fitted (a
# fixed cost plus a cost per token) instead of in full.
PREFILL_FULL_FLOP_LIMIT = 2.0e12
PREFILL_FIT_SIZES = (256, 512)


class OracleSample:
    """The CPU oracle on one layer of a workload (one expert of an MoE layer, with its expected
    share of the tokens). `run` times, on the host cores:

    * the prefill of the layer's whole prompt (all its prompt tokens), or, where that exceeds
      PREFILL_FULL_FLOP_LIMIT, the prefill at two prompt lengths, fitted as a fixed cost plus a
      cost per token and evaluated at the whole prompt;
    * `decode_steps` decode steps, whose mean stands for each of the session's T steps (every
      step does the same work);

    and returns the session time these give, the wall time the sample itself took, and a
    description. One layer's session is what the metric's unit (tokens/s per FFN layer) counts."""

    def __init__(self, wl, seed=0, decode_steps=4):
        import oracle
        import synth
        self.wl, self.oracle = wl, oracle
        f64 = synth.bf16_to_f64
        D, N, B = wl["D"], wl["N"], wl["B"]
        self.E = wl.get("experts", 1)
        self.share = 2.0 / self.E if self.E > 1 else 1.0  # top-2 routing: 2 of E experts per token
        self.Bs = max(1, int(round(B * self.share)))
        self.m_full = max(1, int(round(wl["M"] * self.share)))
        self.fit = 6.0 * self.m_full * D * N > PREFILL_FULL_FLOP_LIMIT
        self.sizes = PREFILL_FIT_SIZES if self.fit else (self.m_full,)
        self.d = decode_steps
        self.W = tuple(f64(w) for w in synth.ffn_weights(seed, D, N))
        sc = synth.dim_scales(seed, D)
        self.X = f64(synth.prompt(seed, max(self.sizes), sc))
        self.xs = [f64(synth.decode_input(seed, t, self.Bs, sc)) for t in range(decode_steps)]

    def run(self):
        wl, oracle = self.wl, self.oracle
        Wg, W1, W2 = self.W
        t_start = time.perf_counter()
        t_at = {}
        pre = None
        for m in self.sizes:
            t0 = time.perf_counter()
            pre = oracle.prefill(Wg, W1, W2, self.X[:m], wl["r"], wl["gamma"])
            t_at[m] = time.perf_counter() - t0
        if self.fit:
            m1, m2 = self.sizes
            per_tok = (t_at[m2] - t_at[m1]) / (m2 - m1)
            fixed = t_at[m1] - per_tok * m1
            t_pre = fixed + per_tok * self.m_full
            pre_info = (f"prefill timed at {m1} and {m2} prompt tokens ({t_at[m1]:.2f} s, {t_at[m2]:.2f} s) and "
                        f"fitted as {fixed:.3f} s + {1e3 * per_tok:.3f} ms per token, evaluated at its "
                        f"{self.m_full} prompt tokens ({t_pre:.2f} s)")
        else:
            t_pre = t_at[self.m_full]
            pre_info = f"prefill of all its {self.m_full} prompt tokens timed ({t_pre:.2f} s)"
        sess = oracle.PopSession(Wg, W1, W2, pre["R"], pre["C"], pre["counts"].k, period=wl["period"])
        t0 = time.perf_counter()
        for x in self.xs:
            sess.step(x)
        t_dec = (time.perf_counter() - t0) / len(self.xs)
        wall = time.perf_counter() - t_start
        session = t_pre + t_dec * wl["T"]
        what = (f"one expert ({wl['D']}x{wl['N']}) of the {self.E}-expert MoE layer with its expected share of "
                f"the tokens" if self.E > 1 else f"one layer of the {wl['D']}x{wl['N']} FFN")
        info = (f"{what}: {pre_info}; {self.d} decode steps at B={self.Bs} timed ({t_dec:.3f} s each), "
                f"their mean taken for each of the session's {wl['T']} steps; float64 numpy with its default "
                f"BLAS threading")
        if self.E > 1:
            # the layer's session: every expert runs its share (the metric counts tokens per layer)
            session *= self.E
        return session, wall, info


def host_threads():
    try:
        return len(os.sched_getaffinity(0))
    except Exception:
        return os.cpu_count() or 1


def cpu_baseline(wl, repeats=3):
    """The oracle's sample (OracleSample), run `repeats` times; the median session time."""
    sample = OracleSample(wl)
    runs = [sample.run() for _ in range(repeats)]
    session = statistics.median(r[0] for r in runs)
    return {"value": wl["B"] * wl["T"] / session, "unit": UNIT, "cores": host_threads(), "kind": "oracle",
            "sample": runs[-1][2] + f"; median of {repeats} runs"}


# ------------------------------------------------------------------ main

def code_hash(path: str) -> str:
    """First 16 hex digits of the SHA-256 of a source file's code: comments and blank lines are
    dropped, so that editing a comment does not retire a profile of unchanged code."""
    import hashlib
    import re
    text = open(path).read()
    text = re.sub(r"/\*.*?\*/", "", text, flags=re.S)
    text = re.sub(r"//[^\n]*", "", text)
    lines = [ln.rstrip() for ln in text.splitlines() if ln.strip()]
    return hashlib.sha256("\n".join(lines).encode()).hexdigest()[:16]


def traffic_from_profiles(kernel: str, workload: str):
    """DRAM bytes per launch from the committed ncu summary, if it was taken on the current code."""
    path = os.path.join(ROOT, "profiles", f"{kernel}_{workload}.md")
    try:
        text = open(path).read()
    except OSError:
        return None
    src_name = "pop_decode1.cu" if workload.endswith("-b1") else "pop_decode_tc.cu"
    sha = code_hash(os.path.join(ROOT, "online_structured_ffn_gb300", "csrc", src_name))
    vals = {}
    for line in text.splitlines():
        line = line.strip().lstrip("-* ")
        if ":" in line and line.startswith(("traffic_bytes_per_launch", "source_sha256_16")):
            k, v = line.split(":", 1)
            vals[k.strip().strip("`")] = v.strip().split()[0].strip("`")
    if vals.get("source_sha256_16") != sha:
        return None
    try:
        return float(vals["traffic_bytes_per_launch"])
    except (KeyError, ValueError):
        return None


def main():
    ap = argparse.ArgumentParser()
    ap.add_argument("--gpus", type=int, default=1)
    ap.add_argument("--steps", type=int, default=20)
    ap.add_argument("--warmup", type=int, default=3)
    ap.add_argument("--impl", choices=["pop", "reference"], default="pop")
    ap.add_argument("--workload", default="llama2-7b-ffn-b1", choices=sorted(WORKLOADS))
    ap.add_argument("--no-secondary", action="store_true",
                    help="skip the B=16, 70B-shape and MoE lines inside the default workload's JSON")
    ap.add_argument("--no-cpu-baseline", action="store_true")
    ap.add_argument("--decode-steps", type=int, default=0,
                    help="override the workload's decode steps per session (short runs for profiler captures)")
    args = ap.parse_args()
    rank, world, local = dist_info()
    if args.decode_steps > 0:
        WORKLOADS[args.workload] = dict(WORKLOADS[args.workload], T=args.decode_steps)
    wl = WORKLOADS[args.workload]
    moe_keys = {"experts": wl["experts"], "routing": "top-2"} if wl.get("experts") else {}
    config = {"workload": args.workload, **moe_keys, **({"skip": True} if wl.get("skip") else {}),
              "D": wl["D"], "D_FF": wl["N"], "r": wl["r"], "gamma": wl["gamma"],
              "B": wl["B"], "prompt_tokens": wl["M"], "decode_steps": wl["T"], "period": wl["period"],
              "layers": wl["layers"],
              "l2": ("inputs larger than L2: each decode step streams every expert's weights "
                     f"({wl['experts']} experts x {3 * wl['D'] * wl['N'] * 2 / 1e6:.0f} MB)" if wl.get("experts") else
                     "inputs larger than L2: each decode step reads another layer's weights "
                     f"({wl['layers']} layers x {3 * wl['D'] * wl['N'] * 2 / 1e6:.0f} MB)"),
              "parallelism": "replicas" if world > 1 else "single-gpu"}

    if args.impl == "reference":
        if rank != 0:
            return
        t0 = time.perf_counter()
        sample = OracleSample(wl)
        for _ in range(args.warmup):
            sample.run()
        sessions, walls, info = [], [], ""
        for _ in range(args.steps):
            sess_s, wall_s, info = sample.run()
            sessions.append(sess_s)
            walls.append(wall_s)
        # each step is one timed sample; its value is the session those timings give (one layer)
        value = wl["B"] * wl["T"] * len(sessions) / sum(sessions)
        line = {"impl": "reference", "metric": METRIC, "value": value, "unit": UNIT, "n_gpus": world,
                "steps": args.steps, "warmup": args.warmup, "ms_per_step": 1e3 * sum(walls) / len(walls),
                "higher_is_better": True, "scaling": "weak", "vs_baseline": None, "dtype": "f64",
                "data": "synthetic", "config": config,
                "cpu_baseline": {"value": value, "unit": UNIT, "cores": host_threads(), "kind": "oracle",
                                 "sample": info + " (each step; ms_per_step is the wall time of one sample)"},
                "e2e": {"value": value, "unit": UNIT, "h2d_bytes_per_step": 0, "d2h_bytes_per_step": 0},
                "wall_s": time.perf_counter() - t0}
        print(json.dumps(line), flush=True)
        return

    import torch
    if world > 1:
        import torch.distributed as dist
        torch.cuda.set_device(local)
        dist.init_process_group("nccl", init_method="env://")
    else:
        torch.cuda.set_device(0)
    import __graft_entry__
    __graft_entry__.build()

    res = run_gpu(args.workload, args.steps, args.warmup)

    def side_line(name, sessions):
        s = run_gpu(name, sessions, max(3, args.warmup), with_e2e=False, with_clocks=True)
        return {"workload": name, "value": s["value"], "unit": UNIT, "sessions": sessions,
                "decode_only_tokens_per_s": s["decode_only_tokens_per_s"],
                "decode_step_us": s["decode_step_us"], "kernel_us": s["kernel_us"],
                "gateup_hbm_gbs": s["gateup_gbs"], "gateup_frac": s["gateup_gbs"] / s["peak"],
                "step_hbm_gbs": s["step_gbs"], "step_frac": s["step_gbs"] / s["peak"],
                "touched_bytes_per_step": s["experts"] * (s["gu_bytes"] + s["dn_bytes"]),
                "dense_step_us": s["dense_step_us"], "prefill_ms_per_layer": s["prefill_ms_per_layer"],
                "clocks": s["clocks"]}

    secondary, others = None, []
    if not args.no_secondary and args.workload == "llama2-7b-ffn-b1":
        # the batched 7B workload, and the 70B-shape and MoE workloads, each timed over 3 sessions
        secondary = side_line("llama2-7b-ffn-b16", max(3, args.steps // 4))
        others = [side_line(n, 3) for n in ("llama-70b-ffn-b64-p16", "moe-8x4096x14336-b32")]
    cpu = None
    if rank == 0 and world == 1 and not args.no_cpu_baseline:
        cpu = cpu_baseline(wl)
    if rank != 0:
        return
    traffic = traffic_from_profiles("gateup_decode", args.workload)
    line = {
        "metric": METRIC, "value": res["value"], "unit": UNIT, "n_gpus": world, "steps": args.steps,
        "warmup": args.warmup, "ms_per_step": res["ms_per_step"], "higher_is_better": True, "scaling": "weak",
        "vs_baseline": None, "dtype": "bf16", "data": "synthetic (seeded counter-based generator)",
        "config": config,
        "roofline": {"bound": "hbm",
                     "kernel": ("k_gateup_sel_b1 (decode gate/up over R u C, top-k inside)" if wl["B"] == 1
                                else "k_gateup_slab (decode gate/up over R u C on tcgen05 from the partition's "
                                     "weight slab, B > 1)"),
                     "achieved": res["gateup_gbs"], "peak": res["peak"], "unit": "GB/s",
                     "frac": res["gateup_gbs"] / res["peak"], "traffic": traffic,
                     "algorithmic_bytes_per_launch": res["roof_bytes"], "peak_source": res["peak_kind"]},
        "decode_step": {"us": res["decode_step_us"], "hbm_gbs": res["step_gbs"], "frac": res["step_gbs"] / res["peak"],
                        "dense_us": res["dense_step_us"],
                        "speedup_vs_dense": (res["dense_step_us"] / res["decode_step_us"]
                                             if res["dense_step_us"] else None),
                        "touched_bytes": res["experts"] * (res["gu_bytes"] + res["dn_bytes"]),
                        "kernel_us": res["kernel_us"],
                        "tokens_per_s": res["decode_only_tokens_per_s"]},
        "prefill_ms_per_layer": res["prefill_ms_per_layer"],
        "counts": res["counts"],
        "e2e": res.get("e2e"),
        "gpu_launches": res["launches"],
        "clocks": res["clocks"],
        "cpu_baseline": cpu,
    }
    if secondary:
        line["secondary"] = secondary
    if others:
        line["other_workloads"] = others
    print(json.dumps(line), flush=True)


if __name__ == "__main__":
    main()
