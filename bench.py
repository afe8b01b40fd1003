#!/usr/bin/env python
"""Decode/verify-step benchmark of the NVFP4 W4A16 skinny path on GB300.

One *step* is one pass of the whole hot path over one batch of M tokens:

  * dense skinny GEMMs K=4096, N=4096 and N=14336,
  * the MoE layer: router top-8 of 128 + grouping, grouped gate+up with the
    GELU-tanh gate, grouped down, combine with the shared expert (d=2816,
    expert intermediate 704),
  * the 262,144 x 2,816 lm_head with the fused per-row argmax.

The metric is weight-GB/s: the algorithmic NVFP4 bytes the step must read
(N*K/2 nibbles + N*K/16 scales per matrix; for the MoE only the experts the
seeded routing touches plus the shared expert) divided by the step time, and
tokens/s = M / step time.  Both M = 15 (the verify block of 14 drafted + 1
token; the headline) and M = 1 are measured in one run: the line's `value` is
M = 15, `per_m` holds both.  A step reads 0.5-0.7 GB of weights, several times
the 126 MB L2, so no flush is needed between steps.  Step times are the median
over 20 batches of back-to-back steps (CUDA events at the batch boundaries).

    python bench.py [--gpus N] [--steps K] [--warmup W] [--impl ours|reference]
    python bench.py --profile-case {lm_head,dense4096,dense14336,moe,router,step} --m M [--reps R]

Under torchrun (N > 1) every rank runs its own replica (the path needs no
exchange between GPUs); rank 0 prints one JSON line.  `--impl reference` times
the FP64 CPU oracle on a bounded sample of the same workload.  `--profile-case`
launches one product R times at one shape (the small case a profiler capture
wants) and prints nothing but a status line.
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

import numpy as np

ROOT = os.path.dirname(os.path.abspath(__file__))
if ROOT not in sys.path:
    sys.path.insert(0, ROOT)

METRIC = "NVFP4 decode weight-GB/s and tokens/s at M=1/15, % of GB300 HBM peak (1 GPU)"
FALLBACK_HBM_GBS = 6800.0


def peaks():
    path = os.path.join(ROOT, "MEASURED_PEAKS.json")
    if os.path.exists(path):
        with open(path) as f:
            p = json.load(f)
        return float(p["hbm_gbs"]), "measured"
    return FALLBACK_HBM_GBS, "fallback"


def max_over_ranks(values, dist, device):
    """Each rank's timings -> their maximum over all ranks (the slowest replica sets
    the job's time).  dist is torch.distributed or None (one process)."""
    if dist is None:
        return [float(v) for v in values]
    import torch
    t = torch.tensor([float(v) for v in values], dtype=torch.float64, device=device)
    dist.all_reduce(t, op=dist.ReduceOp.MAX)
    return t.tolist()


def job_gbs(bytes_per_step, ms_per_step, world):
    """Whole-job weight-GB/s: every replica streams bytes_per_step per step."""
    return world * bytes_per_step / (ms_per_step * 1e-3) / 1e9


def dense_bytes(n, k):
    return n * k // 2 + n * k // 16


class ClockSampler:
    """nvidia-smi clocks/throttle sampling (every 50 ms) while the benchmark runs;
    summary() keeps the samples taken inside the timed windows (window()), with
    50 ms of margin, or, if no sample fell in them, every sample taken under load."""

    FIELDS = ("index,clocks.sm,clocks.max.sm,power.draw,clocks_event_reasons.active,"
              "clocks_event_reasons.hw_slowdown,clocks_event_reasons.hw_thermal_slowdown,"
              "clocks_event_reasons.sw_thermal_slowdown,clocks_event_reasons.sw_power_cap")

    def __init__(self, gpu_index: int):
        self.gpu = gpu_index
        self.proc = None
        self.lines = []      # (time, line)
        self.windows = []    # (start, end)

    def __enter__(self):
        try:
            self.proc = subprocess.Popen(
                ["nvidia-smi", "-i", str(self.gpu), f"--query-gpu={self.FIELDS}", "--format=csv,noheader,nounits",
                 "-lms", "50"], stdout=subprocess.PIPE, stderr=subprocess.DEVNULL, text=True)
            self.thread = threading.Thread(target=self._read, daemon=True)
            self.thread.start()
            time.sleep(0.3)
        except OSError:
            self.proc = None
        return self

    def _read(self):
        for line in self.proc.stdout:
            self.lines.append((time.perf_counter(), line.strip()))

    def __exit__(self, *exc):
        if self.proc is not None:
            time.sleep(0.15)
            self.proc.terminate()
            try:
                self.proc.wait(timeout=5)
            except subprocess.TimeoutExpired:
                self.proc.kill()

    class _Window:
        def __init__(self, owner):
            self.owner = owner

        def __enter__(self):
            self.t0 = time.perf_counter()

        def __exit__(self, *exc):
            self.owner.windows.append((self.t0, time.perf_counter()))

    def window(self):
        return ClockSampler._Window(self)

    def summary(self):
        def inside(t):
            return any(a - 0.05 <= t <= b + 0.05 for a, b in self.windows)
        chosen = [ln for t, ln in self.lines if inside(t)]
        where = "timed windows"
        if not chosen:
            chosen = [ln for _, ln in self.lines]
            where = "whole run (no sample fell inside the short timed windows)"
        sm, mx, reasons = [], [], set()
        names = ["hw_slowdown", "hw_thermal_slowdown", "sw_thermal_slowdown", "sw_power_cap"]
        for line in chosen:
            parts = [p.strip() for p in line.split(",")]
            if len(parts) < 9:
                continue
            try:
                sm.append(float(parts[1]))
                mx.append(float(parts[2]))
            except ValueError:
                continue
            for nm, v in zip(names, parts[5:9]):
                if v.lower() == "active":
                    reasons.add(nm)
        if not sm:
            return {"sm_mhz": None, "sm_max_mhz": None, "reasons": [], "samples": 0, "where": where}
        return {"sm_mhz": statistics.median(sm), "sm_max_mhz": max(mx), "reasons": sorted(reasons),
                "samples": len(sm), "where": where}


# ---------------------------------------------------------------------------------- our arm

MEASURE_M = (15, 1)      # the headline M first
BATCHES = 20


def build_weights(lib, dev):
    """Every weight of the step, quantized and repacked on the GPU (the weights do not depend on M)."""
    import torch
    from nvfp4_w4a16_moe_skinny_gb300 import workloads as W

    def up(a):
        return torch.from_numpy(np.ascontiguousarray(a)).to(dev)

    wl = {"dense": [(n, lib.prepare(up(W.DenseCase.sweep(1, n).w()))) for n in W.DENSE_N]}
    mc = W.MoECase(m=1)
    gu = np.stack([mc.gate_up(e) for e in range(mc.n_experts)])
    wl["gate_up"] = lib.prepare(up(gu), gated=True)
    del gu
    dn = np.stack([mc.down(e) for e in range(mc.n_experts)])
    wl["down"] = lib.prepare(up(dn))
    del dn
    wl["sh_gate_up"] = lib.prepare(up(mc.gate_up(-1)), gated=True)
    wl["sh_down"] = lib.prepare(up(mc.down(-1)))
    lc = W.LMHeadCase(m=1)
    step = 32768
    # quantize needs the whole matrix for its global scale: upload in slices into one buffer
    wfull = torch.empty((lc.vocab, lc.d), dtype=torch.float32, device=dev)
    for lo in range(0, lc.vocab, step):
        wfull[lo:lo + step] = up(lc.w_rows(lo, min(lc.vocab, lo + step)))
    wl["lm_head"] = lib.prepare(wfull)
    del wfull
    torch.cuda.synchronize()
    return wl


def step_bytes(active_experts):
    """Algorithmic weight bytes of one step; the MoE reads the experts the routing touched + the shared one."""
    from nvfp4_w4a16_moe_skinny_gb300 import workloads as W
    per_expert = dense_bytes(2 * W.INTER, W.HIDDEN) + dense_bytes(W.HIDDEN, W.INTER)
    return {
        "dense_4096": dense_bytes(4096, W.DENSE_K),
        "dense_14336": dense_bytes(14336, W.DENSE_K),
        "moe": (active_experts + 1) * per_expert,
        "lm_head": dense_bytes(W.VOCAB, W.HIDDEN),
    }


def make_step(lib, wl, m, dev, stream):
    """Device buffers, pinned host copies of the step's inputs and outputs, and the
    step's calls (zero-argument callables through the C ABI) for batch size m."""
    import torch
    from nvfp4_w4a16_moe_skinny_gb300 import workloads as W

    mc, lc = W.MoECase(m=m), W.LMHeadCase(m=m)
    xd, _ = W.DenseCase.sweep(m, W.DENSE_N[0]).x()
    xm, _ = mc.x()
    xl, _ = lc.x()
    bufs = {
        "x_dense": torch.empty((m, W.DENSE_K), dtype=torch.bfloat16, device=dev),
        "x_moe": torch.empty((m, W.HIDDEN), dtype=torch.bfloat16, device=dev),
        "logits": torch.empty((m, W.N_EXPERTS), dtype=torch.float32, device=dev),
        "x_lm": torch.empty((m, W.HIDDEN), dtype=torch.bfloat16, device=dev),
        "y_4096": torch.empty((m, 4096), dtype=torch.bfloat16, device=dev),
        "y_14336": torch.empty((m, 14336), dtype=torch.bfloat16, device=dev),
        "moe_out": torch.empty((m, W.HIDDEN), dtype=torch.bfloat16, device=dev),
        "max": torch.empty((m,), dtype=torch.float32, device=dev),
        "argmax": torch.empty((m,), dtype=torch.int32, device=dev),
    }
    route = (torch.empty((m, W.TOP_K), dtype=torch.int32, device=dev),
             torch.empty((m, W.TOP_K), dtype=torch.float32, device=dev),
             torch.empty((W.N_EXPERTS + 1,), dtype=torch.int32, device=dev),
             torch.empty((m * W.TOP_K,), dtype=torch.int32, device=dev))
    host = {
        "x_dense": torch.from_numpy(xd.view(np.int16)).view(torch.bfloat16).pin_memory(),
        "x_moe": torch.from_numpy(xm.view(np.int16)).view(torch.bfloat16).pin_memory(),
        "logits": torch.from_numpy(mc.logits()).pin_memory(),
        "x_lm": torch.from_numpy(xl.view(np.int16)).view(torch.bfloat16).pin_memory(),
    }
    outs_host = {k: torch.empty(bufs[k].shape, dtype=bufs[k].dtype).pin_memory()
                 for k in ("y_4096", "y_14336", "moe_out", "max", "argmax")}
    with torch.cuda.stream(stream):
        for k in host:
            bufs[k].copy_(host[k], non_blocking=True)
    stream.synchronize()
    (n0, w0), (n1, w1) = wl["dense"]
    calls = [
        ("dense_4096", lib.plan_gemm(w0, bufs["x_dense"], bufs["y_4096"], stream)),
        ("dense_14336", lib.plan_gemm(w1, bufs["x_dense"], bufs["y_14336"], stream)),
        ("moe", lib.plan_moe(bufs["x_moe"], bufs["logits"], W.TOP_K, wl["gate_up"], wl["down"], wl["sh_gate_up"],
                             wl["sh_down"], route, bufs["moe_out"], stream)),
        ("lm_head", lib.plan_lm_head(wl["lm_head"], bufs["x_lm"], bufs["max"], bufs["argmax"], stream)),
    ]
    return bufs, host, outs_host, calls, route


def time_batches(run_step, steps, stream):
    """Run `steps` steps back to back; CUDA events at BATCHES batch boundaries only (no
    event between the kernels of a batch).  Returns (total ms, median ms per step)."""
    import torch
    nb = max(1, min(BATCHES, steps))
    bounds = [steps * i // nb for i in range(nb + 1)]
    ev = [torch.cuda.Event(enable_timing=True) for _ in range(nb + 1)]
    with torch.cuda.stream(stream):
        ev[0].record(stream)
        for i in range(nb):
            for _ in range(bounds[i + 1] - bounds[i]):
                run_step()
            ev[i + 1].record(stream)
    stream.synchronize()
    per = [ev[i].elapsed_time(ev[i + 1]) / (bounds[i + 1] - bounds[i]) for i in range(nb)]
    return ev[0].elapsed_time(ev[-1]), statistics.median(per)


def time_isolated(lib, wl, calls_m, m, dev, stream, reps=40):
    """Each product of the step alone: `reps` launches back to back (programmatic
    dependent launch overlapping each launch with the previous one), rotating over
    copies of its weights that together exceed 4x L2 so that no launch reads weights
    from L2; events around the whole run.  Returns us per launch (median of 3 runs)."""
    import torch
    from nvfp4_w4a16_moe_skinny_gb300 import binding

    l2 = torch.cuda.get_device_properties(dev).L2_cache_size
    out = {}
    bufs, route = calls_m["bufs"], calls_m["route"]

    def copies(w, nbytes):
        n = max(1, -(-4 * l2 // nbytes))
        return [w] + [binding.Weight(w.data.clone(), w.global_scale.clone(), w.n, w.k, w.num_matrices, w.flags)
                      for _ in range(n - 1)]

    from nvfp4_w4a16_moe_skinny_gb300 import workloads as W
    variants = {}
    for name, (n, w) in zip(("dense_4096", "dense_14336"), wl["dense"]):
        ws = copies(w, w.data.numel())
        y = bufs["y_4096"] if n == 4096 else bufs["y_14336"]
        variants[name] = [lib.plan_gemm(c, bufs["x_dense"], y, stream) for c in ws]
    gus = copies(wl["gate_up"], wl["gate_up"].data.numel() + wl["down"].data.numel())
    dns = [wl["down"]] + [binding.Weight(wl["down"].data.clone(), wl["down"].global_scale.clone(), wl["down"].n,
                                         wl["down"].k, wl["down"].num_matrices, 0) for _ in range(len(gus) - 1)]
    variants["moe"] = [lib.plan_moe(bufs["x_moe"], bufs["logits"], W.TOP_K, g, d, wl["sh_gate_up"], wl["sh_down"],
                                    route, bufs["moe_out"], stream) for g, d in zip(gus, dns)]
    variants["lm_head"] = [lib.plan_lm_head(wl["lm_head"], bufs["x_lm"], bufs["max"], bufs["argmax"], stream)]
    out = time_variants(variants, stream, reps)
    variants.clear()
    torch.cuda.empty_cache()
    return out


def time_variants(variants, stream, reps):
    """us per launch of each named list of callables, cycled `reps` times back to back
    with events around the run on the launching stream (median of 3 runs)."""
    import torch
    out = {}
    for name, fns in variants.items():
        with torch.cuda.stream(stream):
            for i in range(4):
                fns[i % len(fns)]()
        stream.synchronize()
        runs = []
        for _ in range(3):
            e0, e1 = torch.cuda.Event(enable_timing=True), torch.cuda.Event(enable_timing=True)
            with torch.cuda.stream(stream):
                e0.record(stream)
                for i in range(reps):
                    fns[i % len(fns)]()
                e1.record(stream)
            stream.synchronize()
            runs.append(1e3 * e0.elapsed_time(e1) / reps)
        out[name] = statistics.median(runs)
    return out


def time_m_sweep(lib, wl, dev, stream, reps=40):
    """The lm_head and the N=4096 dense GEMM alone at every M = 1..16 (back to back,
    dense weights rotating over copies that exceed 4x L2): us per launch."""
    import torch
    from nvfp4_w4a16_moe_skinny_gb300 import binding
    from nvfp4_w4a16_moe_skinny_gb300 import workloads as W
    l2 = torch.cuda.get_device_properties(dev).L2_cache_size
    (n0, w0), _ = wl["dense"]
    copies = [w0] + [binding.Weight(w0.data.clone(), w0.global_scale.clone(), w0.n, w0.k, 1, 0)
                     for _ in range(max(1, -(-4 * l2 // w0.data.numel())) - 1)]
    out = {}
    for m in range(1, 17):
        xl = torch.from_numpy(W.LMHeadCase(m=m).x()[0].view(np.int16)).to(dev).view(torch.bfloat16)
        xd = torch.from_numpy(W.DenseCase.sweep(m, n0).x()[0].view(np.int16)).to(dev).view(torch.bfloat16)
        mx = torch.empty((m,), dtype=torch.float32, device=dev)
        am = torch.empty((m,), dtype=torch.int32, device=dev)
        y = torch.empty((m, n0), dtype=torch.bfloat16, device=dev)
        us = time_variants({"lm_head": [lib.plan_lm_head(wl["lm_head"], xl, mx, am, stream)],
                            "dense_4096": [lib.plan_gemm(c, xd, y, stream) for c in copies]}, stream, reps)
        out[str(m)] = {k: round(v, 2) for k, v in us.items()}
    del copies
    torch.cuda.empty_cache()
    if lib.device_error() != 0:
        raise RuntimeError("device error flag set during the M sweep")
    return out


def time_w4a4(lib, wl, bufs, m, dev, stream, reps=40):
    """The W4A4 products (activations quantized to NVFP4 per token row) at the step's
    M: the activation quantizer, the dense GEMMs (rotating over weight copies that
    together exceed 4x L2) and the lm_head argmax, each alone, back to back."""
    import torch
    from nvfp4_w4a16_moe_skinny_gb300 import binding
    l2 = torch.cuda.get_device_properties(dev).L2_cache_size
    xq_d, xq_l = lib.quantize_act(bufs["x_dense"]), lib.quantize_act(bufs["x_lm"])
    variants = {"quantize_act_4096": [lib.plan_quantize_act(bufs["x_dense"], xq_d, stream)],
                "quantize_act_2816": [lib.plan_quantize_act(bufs["x_lm"], xq_l, stream)]}
    for name, (n, w) in zip(("dense_4096", "dense_14336"), wl["dense"]):
        copies = [w] + [binding.Weight(w.data.clone(), w.global_scale.clone(), w.n, w.k, 1, 0)
                        for _ in range(max(1, -(-4 * l2 // w.data.numel())) - 1)]
        y = bufs["y_4096"] if n == 4096 else bufs["y_14336"]
        variants[name] = [lib.plan_gemm_w4a4(c, xq_d, y, stream) for c in copies]
    variants["lm_head"] = [lib.plan_lm_head_w4a4(wl["lm_head"], xq_l, bufs["max"], bufs["argmax"], stream)]
    us = time_variants(variants, stream, reps)
    variants.clear()
    torch.cuda.empty_cache()
    if lib.device_error() != 0:
        raise RuntimeError("device error flag set during the W4A4 timing")
    peak, _ = peaks()
    b = step_bytes(0)
    gbs = {k: round(b[k] / (v * 1e-6) / 1e9, 1) for k, v in us.items() if k in b}
    return {"m": m, "kernels_us": {k: round(v, 2) for k, v in us.items()}, "kernels_gbs": gbs,
            "kernels_hbm_frac": {k: round(v / peak, 4) for k, v in gbs.items()}}


def measure_m(lib, wl, m, args, dev, stream, dist, world, clocks):
    """Every figure of one batch size: the step (median of batches), the lm_head's
    launch time inside the steps, each product alone, the end-to-end step through the
    C ABI with host buffers."""
    import torch
    bufs, host, outs_host, calls, route = make_step(lib, wl, m, dev, stream)

    def step():
        for _, fn in calls:
            fn()

    def barrier():
        if dist is not None:
            dist.barrier()

    with torch.cuda.stream(stream):
        for _ in range(args.warmup):
            step()
    stream.synchronize()
    if lib.device_error() != 0:
        raise RuntimeError("device error flag set during warm-up")
    counts = (route[2][1:] - route[2][:-1]).cpu()
    active = int((counts > 0).sum())
    nbytes = step_bytes(active)

    # ---- device-resident timing: steps back to back, events only at batch boundaries
    barrier()
    torch.cuda.synchronize()
    with clocks.window():
        total_ms, med_ms = time_batches(step, args.steps, stream)
    torch.cuda.synchronize()
    barrier()

    # ---- the lm_head (the roofline kernel) timed live inside the same steps: events
    # around it on its stream, a second pass over the steps
    ev_lm = [(torch.cuda.Event(enable_timing=True), torch.cuda.Event(enable_timing=True)) for _ in range(args.steps)]
    with torch.cuda.stream(stream):
        for s in range(args.steps):
            for name, fn in calls:
                if name == "lm_head":
                    ev_lm[s][0].record(stream)
                    fn()
                    ev_lm[s][1].record(stream)
                else:
                    fn()
    stream.synchronize()
    lm_us = 1e3 * statistics.median(a.elapsed_time(b) for a, b in ev_lm)

    # ---- the same steps replayed from a CUDA graph (one step captured)
    graph_ms = None
    try:
        graph = torch.cuda.CUDAGraph()
        with torch.cuda.graph(graph, stream=stream):
            step()
        for _ in range(2):
            graph.replay()
        stream.synchronize()
        _, graph_ms = time_batches(graph.replay, args.steps, stream)
    except Exception as exc:  # capture can be unavailable; the eager number stands
        print(f"graph replay skipped: {exc}", file=sys.stderr)

    kernel_us = time_isolated(lib, wl, {"bufs": bufs, "route": route}, m, dev, stream)

    # ---- end to end through the public API with host buffers (copies inside the timed region)
    h2d = sum(t.numel() * t.element_size() for t in host.values())
    d2h = sum(t.numel() * t.element_size() for t in outs_host.values())
    e0, e1 = torch.cuda.Event(enable_timing=True), torch.cuda.Event(enable_timing=True)
    barrier()
    torch.cuda.synchronize()
    wall0 = time.perf_counter()
    with torch.cuda.stream(stream):
        e0.record(stream)
        for _ in range(args.steps):
            for k, t in host.items():
                bufs[k].copy_(t, non_blocking=True)
            step()
            for k, t in outs_host.items():
                t.copy_(bufs[k], non_blocking=True)
        e1.record(stream)
    stream.synchronize()
    wall_ms = (time.perf_counter() - wall0) * 1e3
    barrier()
    e2e_ms = max(e0.elapsed_time(e1), wall_ms)
    if lib.device_error() != 0:
        raise RuntimeError("device error flag set during the timed region")
    total_ms, med_ms, e2e_ms = max_over_ranks([total_ms, med_ms, e2e_ms], dist, dev)
    bytes_step = sum(nbytes.values())
    peak, _ = peaks()
    return {
        "m": m,
        "ms_per_step": round(med_ms, 4),
        "ms_per_step_mean": round(total_ms / args.steps, 4),
        "weight_gbs": round(job_gbs(bytes_step, med_ms, world), 1),
        "tokens_per_s": round(world * m / (med_ms * 1e-3), 1),
        "hbm_frac": round(bytes_step / (med_ms * 1e-3) / 1e9 / peak, 4),
        "weight_bytes_per_step": bytes_step,
        "bytes": nbytes,
        "active_experts": active,
        "kernels_us": {k: round(v, 2) for k, v in kernel_us.items()},
        "kernels_gbs": {k: round(nbytes[k] / (kernel_us[k] * 1e-6) / 1e9, 1) for k in kernel_us},
        "kernels_hbm_frac": {k: round(nbytes[k] / (kernel_us[k] * 1e-6) / 1e9 / peak, 4) for k in kernel_us},
        "lm_head_us_in_step": round(lm_us, 2),
        "graph_ms_per_step": round(graph_ms, 4) if graph_ms else None,
        "e2e_gbs": round(job_gbs(bytes_step, e2e_ms / args.steps, world), 1),
        "h2d_bytes_per_step": h2d,
        "d2h_bytes_per_step": d2h,
        "launches_per_step": 7,
    }


def run_ours(args, rank, world, dist):
    import torch
    from nvfp4_w4a16_moe_skinny_gb300 import binding

    local = int(os.environ.get("LOCAL_RANK", "0"))
    torch.cuda.set_device(local)
    dev = torch.device("cuda", local)
    lib = binding.load()
    wl = build_weights(lib, dev)
    stream = torch.cuda.Stream(device=dev)
    clocks = ClockSampler(local)
    with clocks:
        per_m = {m: measure_m(lib, wl, m, args, dev, stream, dist, world, clocks) for m in MEASURE_M}
        prefill = time_prefill(lib, wl, args, dev, stream) if args.prefill_m > 0 else None
        bufs, _, _, _, _ = make_step(lib, wl, MEASURE_M[0], dev, stream)
        sampling = time_sampling(lib, wl, bufs, MEASURE_M[0], args, dev, stream)
        w4a4 = time_w4a4(lib, wl, bufs, MEASURE_M[0], dev, stream)
        m_sweep = time_m_sweep(lib, wl, dev, stream)
    head = per_m[MEASURE_M[0]]
    peak, peak_kind = peaks()
    lm_bytes = head["bytes"]["lm_head"]
    achieved = lm_bytes / (head["lm_head_us_in_step"] * 1e-6) / 1e9
    traffic = load_traffic("lm_head", MEASURE_M[0])
    result = {
        "metric": METRIC,
        "value": head["weight_gbs"],
        "unit": "GB/s",
        "n_gpus": world,
        "steps": args.steps,
        "warmup": args.warmup,
        "ms_per_step": head["ms_per_step"],
        "higher_is_better": True,
        "scaling": "weak",
        "vs_baseline": None,
        "dtype": "nvfp4 weights (e2m1 + e4m3 scales), bf16 activations (f16 x 2^s on the tensor cores), fp32 accumulate",
        "data": "synthetic: seeded N(0,0.02) fp32 weights quantized to NVFP4 on the GPU; N(0,1) bf16 activations",
        "config": {
            "workload": f"decode/verify step at M={MEASURE_M[0]} (and M=1 in per_m): dense K=4096 N=4096+14336, "
                        f"MoE d=2816 128 experts (I=704) top-8 + shared, lm_head 262144x2816 with argmax",
            "m": MEASURE_M[0],
            "weight_bytes_per_step": head["weight_bytes_per_step"],
            "bytes": head["bytes"],
            "active_experts": head["active_experts"],
            "l2": "inputs larger than L2: each step reads 0.5-0.7 GB of weights (L2 126 MB); no flush. "
                  "kernels_us rotates weight copies totalling >= 4x L2",
            "parallelism": f"replicas x{world}" if world > 1 else "single GPU",
        },
        "tokens_per_s": head["tokens_per_s"],
        "hbm_frac": head["hbm_frac"],
        "per_m": {str(m): v for m, v in per_m.items()},
        "roofline": {"bound": "hbm", "kernel": "lm_head_argmax (stream_kernel, argmax epilogue), M=15",
                     "achieved": round(achieved, 1), "launch_us": head["lm_head_us_in_step"],
                     "peak": peak, "peak_kind": f"{peak_kind} (copy)", "unit": "GB/s",
                     "frac": round(achieved / peak, 4), "traffic": traffic},
        "e2e": {"value": head["e2e_gbs"], "unit": "GB/s", "h2d_bytes_per_step": head["h2d_bytes_per_step"],
                "d2h_bytes_per_step": head["d2h_bytes_per_step"]},
        "graph_ms_per_step": head["graph_ms_per_step"],
        "prefill": prefill,
        "lm_head_sample": sampling,
        "w4a4": w4a4,
        "m_sweep_us": m_sweep,
        "gpu_launches": head["launches_per_step"] * args.steps,
        "timing": "ms_per_step: median over 20 batches of back-to-back steps (events at batch boundaries only); "
                  "roofline: events around the lm_head in a second pass over the same steps; kernels_us: each "
                  "product alone, 40 launches back to back over rotating weight copies, median of 3",
        "clocks": clocks.summary(),
    }
    if rank == 0 and not args.no_cpu_baseline and world == 1:
        result["cpu_baseline"] = cpu_baseline(MEASURE_M[0], seconds=args.cpu_seconds)
    return result


def time_sampling(lib, wl, bufs, m, args, dev, stream):
    """The lm_head with fused Gumbel-max temperature sampling (T = 1) at the step's M,
    back to back with events on the launching stream, each launch a new seed."""
    import torch
    key = torch.empty((m,), dtype=torch.float32, device=dev)
    tok = torch.empty((m,), dtype=torch.int32, device=dev)
    fns = [lib.plan_lm_head_sample(wl["lm_head"], bufs["x_lm"], 1.0, 1000 + s, key, tok, stream)
           for s in range(args.steps)]
    with torch.cuda.stream(stream):
        for fn in fns[:args.warmup]:
            fn()
    stream.synchronize()
    e0, e1 = torch.cuda.Event(enable_timing=True), torch.cuda.Event(enable_timing=True)
    with torch.cuda.stream(stream):
        e0.record(stream)
        for fn in fns:
            fn()
        e1.record(stream)
    stream.synchronize()
    if lib.device_error() != 0:
        raise RuntimeError("device error flag set during the sampling timing")
    us = 1e3 * e0.elapsed_time(e1) / len(fns)
    nbytes = step_bytes(0)["lm_head"]
    peak, _ = peaks()
    return {"m": m, "temperature": 1.0, "us_per_launch": round(us, 2),
            "weight_gbs": round(nbytes / (us * 1e-6) / 1e9, 1), "hbm_frac": round(nbytes / (us * 1e-6) / 1e9 / peak, 4)}


def time_prefill(lib, wl, args, dev, stream):
    """The MoE layer on a prefill chunk of `args.prefill_m` tokens (same weights as the
    decode step): router + grouped gate+up + grouped down + combine, timed back to back
    with events on the launching stream.  Weight-GB/s counts every expert the routing
    touches once, plus the shared expert."""
    import torch
    from nvfp4_w4a16_moe_skinny_gb300 import workloads as W

    m = args.prefill_m
    mc = W.MoECase(m=m)
    xb, _ = mc.x()
    x = torch.from_numpy(xb.view(np.int16)).to(dev).view(torch.bfloat16)
    logits = torch.from_numpy(mc.logits()).to(dev)
    route = (torch.empty((m, W.TOP_K), dtype=torch.int32, device=dev),
             torch.empty((m, W.TOP_K), dtype=torch.float32, device=dev),
             torch.empty((W.N_EXPERTS + 1,), dtype=torch.int32, device=dev),
             torch.empty((m * W.TOP_K,), dtype=torch.int32, device=dev))
    out = torch.empty((m, W.HIDDEN), dtype=torch.bfloat16, device=dev)
    fn = lib.plan_moe(x, logits, W.TOP_K, wl["gate_up"], wl["down"], wl["sh_gate_up"], wl["sh_down"], route, out,
                      stream)
    with torch.cuda.stream(stream):
        for _ in range(args.warmup):
            fn()
    stream.synchronize()
    counts = (route[2][1:] - route[2][:-1]).cpu()
    active = int((counts > 0).sum())
    nbytes = step_bytes(active)["moe"]
    steps = max(args.steps, 10)
    e0, e1 = torch.cuda.Event(enable_timing=True), torch.cuda.Event(enable_timing=True)
    with torch.cuda.stream(stream):
        e0.record(stream)
        for _ in range(steps):
            fn()
        e1.record(stream)
    stream.synchronize()
    if lib.device_error() != 0:
        raise RuntimeError("device error flag set during the prefill timing")
    ms = e0.elapsed_time(e1) / steps
    peak, _ = peaks()
    gbs = nbytes / (ms * 1e-3) / 1e9
    return {"m": m, "ms_per_layer": round(ms, 4), "tokens_per_s": round(m / (ms * 1e-3), 1),
            "weight_bytes": nbytes, "active_experts": active, "max_pairs_per_expert": int(counts.max()),
            "weight_gbs": round(gbs, 1), "hbm_frac": round(gbs / peak, 4),
            # router (top-k grid + grouping grid above 32 tokens), gate+up, down, combine
            "launches_per_layer": 5 if m > 32 else 4}


def load_traffic(kernel, m):
    """DRAM bytes per launch from the committed ncu summary, if it covers this kernel and M."""
    path = os.path.join(ROOT, "profiles", "traffic.json")
    if not os.path.exists(path):
        return None
    with open(path) as f:
        data = json.load(f)
    entry = data.get(f"{kernel}_m{m}")
    return entry.get("dram_bytes_per_launch") if entry else None


# ---------------------------------------------------------------------------------- oracle arm

def oracle_sample(m):
    """A bounded sample of the same workload for the FP64 CPU oracle: the N=4096 dense GEMM,
    2 experts of the MoE layer (x routed to them) and 16384 lm_head rows.  Quantization is
    offline and not timed; returns (timed callable, weight bytes it reads, description)."""
    from nvfp4_w4a16_moe_skinny_gb300 import workloads as W
    from oracle import formats as F, gemm as OG, lm_head as OLM, moe as OM

    dc = W.DenseCase.sweep(m, 4096)
    dq = F.quantize_matrix(dc.w())
    _, xd = dc.x()
    mc = W.MoECase(m=m)
    experts = [F.quantize_matrix(mc.gate_up(e)) for e in (0, 1)], [F.quantize_matrix(mc.down(e)) for e in (0, 1)]
    _, xm = mc.x()
    lc = W.LMHeadCase(m=m)
    rows = 16384
    lq = F.quantize_matrix(lc.w_rows(0, rows))
    _, xl = lc.x()
    nbytes = dense_bytes(4096, 4096) + 2 * (dense_bytes(2 * W.INTER, W.HIDDEN) + dense_bytes(W.HIDDEN, W.INTER)) + \
        dense_bytes(rows, W.HIDDEN)

    def run():
        OG.nvfp4_gemm(*dq, xd.astype(np.float64))
        for (gn, gs, gg), (dn_, ds, dg) in zip(*experts):
            OM.expert_ffn(F.dequantize_matrix(gn, gs, gg), F.dequantize_matrix(dn_, ds, dg), xm.astype(np.float64))
        OLM.lm_head_argmax(*lq, xl.astype(np.float64), chunk_rows=8192)

    desc = (f"FP64 numpy oracle at M={m}: dense 4096x4096 GEMM + 2 of the MoE experts (gate_up + GELU + down) "
            f"+ {rows} of 262144 lm_head rows with argmax ({nbytes} NVFP4 weight bytes per sample)")
    return run, nbytes, desc


def cpu_threads():
    try:
        return len(os.sched_getaffinity(0))
    except AttributeError:
        return os.cpu_count() or 1


def cpu_baseline(m, seconds=10.0):
    run, nbytes, desc = oracle_sample(m)
    times = []
    t_end = time.perf_counter() + seconds
    while True:
        t = time.perf_counter()
        run()
        times.append(time.perf_counter() - t)
        if time.perf_counter() > t_end or len(times) >= 20:
            break
    med = statistics.median(times)
    return {"value": round(nbytes / med / 1e9, 4), "unit": "GB/s", "cores": cpu_threads(), "kind": "oracle",
            "sample": f"{desc}; median of {len(times)} runs ({med:.2f} s each)"}


def run_reference(args, rank, world):
    if rank != 0:
        return None
    run, nbytes, desc = oracle_sample(args.m)
    for _ in range(args.warmup):
        run()
    t0 = time.perf_counter()
    for _ in range(args.steps):
        run()
    ms = (time.perf_counter() - t0) * 1e3
    value = nbytes * args.steps / (ms * 1e-3) / 1e9
    return {
        "impl": "reference",
        "metric": METRIC,
        "value": round(value, 4),
        "unit": "GB/s",
        "n_gpus": world,
        "steps": args.steps,
        "warmup": args.warmup,
        "ms_per_step": round(ms / args.steps, 2),
        "higher_is_better": True,
        "scaling": "weak",
        "vs_baseline": None,
        "dtype": "f64",
        "data": "synthetic: seeded, same generators as the GPU arm",
        "config": {"workload": f"bounded sample of the decode/verify step at M={args.m}", "m": args.m,
                   "sample_weight_bytes": nbytes},
        "cpu_baseline": {"value": round(value, 4), "unit": "GB/s", "cores": cpu_threads(), "kind": "oracle",
                         "sample": desc},
        "e2e": {"value": round(value, 4), "unit": "GB/s", "h2d_bytes_per_step": 0, "d2h_bytes_per_step": 0},
    }


def profile_case(kind, m, reps):
    """Launch one product `reps` times at one shape: the small single-kernel case a
    profiler capture wants (``ncu -k regex:tc_kernel -s <skip> -c <n> ...``).  Weights
    are seeded N(0, 0.02) fp32 quantized on the GPU, activations N(0, 1) bf16; each
    repetition launches one kernel (lm_head, dense), four (moe: route, gate+up,
    down, combine) or four (router: the NVFP4 router GEMM with fp32 output, the
    RMSNorm + scale, the top-k + grouping); `step` runs the whole decode/verify step
    of the bench (seven launches per repetition, the bench's weights and inputs).
    Exits non-zero if the library's device error flag is set."""
    import torch
    from nvfp4_w4a16_moe_skinny_gb300 import binding

    lib = binding.load()
    dev = torch.device("cuda", 0)
    g = torch.Generator(device=dev).manual_seed(0)

    def randn(*shape):
        return torch.randn(shape, generator=g, device=dev)

    if kind == "step":
        stream = torch.cuda.Stream(device=dev)
        wl = build_weights(lib, dev)
        _, _, _, calls, _ = make_step(lib, wl, m, dev, stream)
        torch.cuda.synchronize()
        for _ in range(reps):
            for _, fn in calls:
                fn()
        stream.synchronize()
    elif kind == "moe":
        e, d, inter = 128, 2816, 704
        gu = lib.prepare(randn(e, 2 * inter, d) * 0.02, gated=True)
        dn = lib.prepare(randn(e, d, inter) * 0.02)
        sgu = lib.prepare(randn(2 * inter, d) * 0.02, gated=True)
        sdn = lib.prepare(randn(d, inter) * 0.02)
        x = randn(m, d).to(torch.bfloat16)
        logits = randn(m, e)
        torch.cuda.synchronize()
        for _ in range(reps):
            _, probs, offs, pairs = lib.route_topk(logits, 8)
            lib.moe_ffn(x, 8, probs, offs, pairs, gu, dn, sgu, sdn)
    elif kind == "router":
        e, d = 128, 2816
        wr = lib.prepare(randn(e, d) * 0.02)
        scale = 1.0 + 0.1 * randn(e)
        x = randn(m, d).to(torch.bfloat16)
        torch.cuda.synchronize()
        for _ in range(reps):
            logits = lib.router_logits(wr, x, scale)
            lib.route_topk(logits, 8)
    else:
        shapes = {"lm_head": (262144, 2816), "dense4096": (4096, 4096), "dense14336": (14336, 4096)}
        n, k = shapes[kind]
        w = lib.prepare(randn(n, k) * 0.02)
        x = randn(m, k).to(torch.bfloat16)
        torch.cuda.synchronize()
        for _ in range(reps):
            if kind == "lm_head":
                lib.lm_head_argmax(w, x)
            else:
                lib.gemm(w, x)
    torch.cuda.synchronize()
    if lib.device_error() != 0:
        raise SystemExit("device error flag set")
    print(f"ok {kind} m={m} reps={reps}")


def main():
    ap = argparse.ArgumentParser(description=__doc__, formatter_class=argparse.RawDescriptionHelpFormatter)
    ap.add_argument("--gpus", type=int, default=1)
    ap.add_argument("--steps", type=int, default=100)
    ap.add_argument("--warmup", type=int, default=5)
    ap.add_argument("--m", type=int, default=15, help="batch size of the reference arm and of --profile-case")
    ap.add_argument("--impl", choices=("ours", "reference"), default="ours")
    ap.add_argument("--cpu-seconds", type=float, default=10.0)
    ap.add_argument("--prefill-m", type=int, default=512,
                    help="also time the MoE layer on a prefill chunk of this many tokens (0: skip)")
    ap.add_argument("--no-cpu-baseline", action="store_true")
    ap.add_argument("--profile-case", choices=("lm_head", "dense4096", "dense14336", "moe", "router", "step"),
                    default=None)
    ap.add_argument("--reps", type=int, default=3)
    args = ap.parse_args()
    if args.profile_case:
        profile_case(args.profile_case, args.m, args.reps)
        return
    if args.warmup < 3:
        ap.error("--warmup must be >= 3")
    world = int(os.environ.get("WORLD_SIZE", "1"))
    rank = int(os.environ.get("RANK", "0"))
    dist = None
    if args.impl == "reference":
        res = run_reference(args, rank, world)
    else:
        if world > 1:
            import torch
            import torch.distributed as tdist
            torch.cuda.set_device(int(os.environ.get("LOCAL_RANK", "0")))
            tdist.init_process_group("nccl")
            dist = tdist
        res = run_ours(args, rank, world, dist)
        if dist is not None:
            dist.destroy_process_group()
    if rank == 0 and res is not None:
        print(json.dumps(res), flush=True)


if __name__ == "__main__":
    main()
