#!/usr/bin/env python
"""Decode/verify-step benchmark of the NVFP4 W4A16 skinny path on GB300.

One *step* is one pass of the whole hot path over one batch of M tokens
(default M = 15, the verify block of 14 drafted + 1 token):

  * dense skinny GEMMs K=4096, N=4096 and N=14336,
  * the MoE layer: router top-8 of 128 + grouping, grouped gate+up with the
    GELU-tanh gate, grouped down, combine with the shared expert (d=2816,
    expert intermediate 704),
  * the 262,144 x 2,816 lm_head with the fused per-row argmax.

The metric is weight-GB/s: the algorithmic NVFP4 bytes the step must read
(N*K/2 nibbles + N*K/16 scales per matrix; for the MoE only the experts the
seeded routing touches plus the shared expert) divided by the step time.
tokens/s = M / step time.  A step reads ~0.7 GB of weights, several times the
126 MB L2, so no L2 flush is needed between steps.

    python bench.py [--gpus N] [--steps K] [--warmup W] [--m M] [--impl ours|reference]

Under torchrun (N > 1) every rank runs its own replica (the path needs no
exchange between GPUs); rank 0 prints one JSON line.  `--impl reference` times
the FP64 CPU oracle on a bounded sample of the same workload.
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
    """nvidia-smi clocks/throttle sampling during the timed region."""

    FIELDS = ("index,clocks.sm,clocks.max.sm,power.draw,clocks_event_reasons.active,"
              "clocks_event_reasons.hw_slowdown,clocks_event_reasons.hw_thermal_slowdown,"
              "clocks_event_reasons.sw_thermal_slowdown,clocks_event_reasons.sw_power_cap")

    def __init__(self, gpu_index: int):
        self.gpu = gpu_index
        self.proc = None
        self.lines = []

    def __enter__(self):
        try:
            self.proc = subprocess.Popen(
                ["nvidia-smi", "-i", str(self.gpu), f"--query-gpu={self.FIELDS}", "--format=csv,noheader,nounits",
                 "-lms", "100"], stdout=subprocess.PIPE, stderr=subprocess.DEVNULL, text=True)
            self.thread = threading.Thread(target=self._read, daemon=True)
            self.thread.start()
            time.sleep(0.3)
        except OSError:
            self.proc = None
        return self

    def _read(self):
        for line in self.proc.stdout:
            self.lines.append(line.strip())

    def __exit__(self, *exc):
        if self.proc is not None:
            time.sleep(0.15)
            self.proc.terminate()
            try:
                self.proc.wait(timeout=5)
            except subprocess.TimeoutExpired:
                self.proc.kill()

    def summary(self):
        sm, mx, reasons = [], [], set()
        names = ["hw_slowdown", "hw_thermal_slowdown", "sw_thermal_slowdown", "sw_power_cap"]
        for line in self.lines:
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
            return {"sm_mhz": None, "sm_max_mhz": None, "reasons": [], "samples": 0}
        return {"sm_mhz": statistics.median(sm), "sm_max_mhz": max(mx), "reasons": sorted(reasons),
                "samples": len(sm)}


# ---------------------------------------------------------------------------------- our arm

def build_workload(lib, m, dev):
    import torch
    from nvfp4_w4a16_moe_skinny_gb300 import workloads as W

    def up(a):
        return torch.from_numpy(np.ascontiguousarray(a)).to(dev)

    def up_bf16(bits):
        return torch.from_numpy(bits.view(np.int16)).to(dev).view(torch.bfloat16)

    wl = {}
    dense = []
    for n in W.DENSE_N:
        case = W.DenseCase.sweep(m, n)
        dense.append((n, lib.prepare(up(case.w()))))
    wl["dense"] = dense
    xd, _ = W.DenseCase.sweep(m, W.DENSE_N[0]).x()
    wl["x_dense_host"] = xd

    mc = W.MoECase(m=m)
    gu = np.stack([mc.gate_up(e) for e in range(mc.n_experts)])
    wl["gate_up"] = lib.prepare(up(gu), gated=True)
    del gu
    dn = np.stack([mc.down(e) for e in range(mc.n_experts)])
    wl["down"] = lib.prepare(up(dn))
    del dn
    wl["sh_gate_up"] = lib.prepare(up(mc.gate_up(-1)), gated=True)
    wl["sh_down"] = lib.prepare(up(mc.down(-1)))
    xm, _ = mc.x()
    wl["x_moe_host"] = xm
    wl["logits_host"] = mc.logits()

    lc = W.LMHeadCase(m=m)
    chunks = []
    step = 32768
    # quantize needs the whole matrix for its global scale: upload in slices into one buffer
    wfull = torch.empty((lc.vocab, lc.d), dtype=torch.float32, device=dev)
    for lo in range(0, lc.vocab, step):
        wfull[lo:lo + step] = up(lc.w_rows(lo, min(lc.vocab, lo + step)))
    wl["lm_head"] = lib.prepare(wfull)
    del wfull, chunks
    xl, _ = lc.x()
    wl["x_lm_host"] = xl

    torch.cuda.synchronize()
    return wl


def step_bytes(wl, active_experts):
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
    import torch
    from nvfp4_w4a16_moe_skinny_gb300 import workloads as W

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
        "x_dense": torch.from_numpy(wl["x_dense_host"].view(np.int16)).view(torch.bfloat16).pin_memory(),
        "x_moe": torch.from_numpy(wl["x_moe_host"].view(np.int16)).view(torch.bfloat16).pin_memory(),
        "logits": torch.from_numpy(wl["logits_host"]).pin_memory(),
        "x_lm": torch.from_numpy(wl["x_lm_host"].view(np.int16)).view(torch.bfloat16).pin_memory(),
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


def run_ours(args, rank, world, dist):
    import torch
    from nvfp4_w4a16_moe_skinny_gb300 import binding

    local = int(os.environ.get("LOCAL_RANK", "0"))
    torch.cuda.set_device(local)
    dev = torch.device("cuda", local)
    lib = binding.load()
    m = args.m
    wl = build_workload(lib, m, dev)
    stream = torch.cuda.Stream(device=dev)
    bufs, host, outs_host, calls, route = make_step(lib, wl, m, dev, stream)
    launches_per_step = 1 + 1 + 4 + 1   # gemm, gemm, route + gate_up + down + combine, lm_head

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
    wl["active_experts"] = int((counts > 0).sum())
    wl["bytes"] = step_bytes(wl, wl["active_experts"])

    def timed_events():
        return [(torch.cuda.Event(enable_timing=True), torch.cuda.Event(enable_timing=True))
                for _ in range(args.steps)]

    # ---- device-resident timing of the steps back to back (each launch may start
    # its weight copies while the previous one finishes); events around the whole
    # region and around the lm_head, the dominant kernel, inside it
    ev_lm = timed_events()
    t0, t1 = torch.cuda.Event(enable_timing=True), torch.cuda.Event(enable_timing=True)
    barrier()
    torch.cuda.synchronize()
    with ClockSampler(local) as clocks:
        with torch.cuda.stream(stream):
            t0.record(stream)
            for s in range(args.steps):
                for name, fn in calls:
                    if name == "lm_head":
                        ev_lm[s][0].record(stream)
                        fn()
                        ev_lm[s][1].record(stream)
                    else:
                        fn()
            t1.record(stream)
        stream.synchronize()
    torch.cuda.synchronize()
    barrier()
    total_ms = t0.elapsed_time(t1)
    lm_us = 1e3 * statistics.mean(a.elapsed_time(b) for a, b in ev_lm)

    # ---- the same steps replayed from a CUDA graph (one step captured; launch costs off the host)
    graph_ms = None
    try:
        graph = torch.cuda.CUDAGraph()
        with torch.cuda.graph(graph, stream=stream):
            step()
        for _ in range(2):
            graph.replay()
        stream.synchronize()
        g0, g1 = torch.cuda.Event(enable_timing=True), torch.cuda.Event(enable_timing=True)
        with torch.cuda.stream(stream):
            g0.record(stream)
            for _ in range(args.steps):
                graph.replay()
            g1.record(stream)
        stream.synchronize()
        graph_ms = g0.elapsed_time(g1) / args.steps
    except Exception as exc:  # capture can be unavailable; the eager number stands
        print(f"graph replay skipped: {exc}", file=sys.stderr)

    # ---- per-call attribution: events around every call (no overlap across calls)
    ev = {name: timed_events() for name, _ in calls}
    with torch.cuda.stream(stream):
        for s in range(args.steps):
            for name, fn in calls:
                a, b = ev[name][s]
                a.record(stream)
                fn()
                b.record(stream)
    stream.synchronize()
    kernel_us = {name: 1e3 * statistics.mean(a.elapsed_time(b) for a, b in ev[name]) for name, _ in calls}

    prefill = time_prefill(lib, wl, args, dev, stream) if args.prefill_m > 0 else None
    sampling = time_sampling(lib, wl, bufs, m, args, dev, stream)

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

    bytes_step = sum(wl["bytes"].values())
    total_ms, e2e_ms = max_over_ranks([total_ms, e2e_ms], dist, dev)
    ms_step = total_ms / args.steps
    value = job_gbs(bytes_step, ms_step, world)
    e2e_value = job_gbs(bytes_step, e2e_ms / args.steps, world)
    peak, peak_kind = peaks()
    lm_bytes = wl["bytes"]["lm_head"]
    achieved = lm_bytes / (lm_us * 1e-6) / 1e9
    traffic = load_traffic("lm_head", m)
    result = {
        "metric": METRIC,
        "value": round(value, 1),
        "unit": "GB/s",
        "n_gpus": world,
        "steps": args.steps,
        "warmup": args.warmup,
        "ms_per_step": round(ms_step, 4),
        "higher_is_better": True,
        "scaling": "weak",
        "vs_baseline": None,
        "dtype": "nvfp4 weights (e2m1 + e4m3 scales), bf16 activations, fp32 accumulate",
        "data": "synthetic: seeded N(0,0.02) fp32 weights quantized to NVFP4 on the GPU; N(0,1) bf16 activations",
        "config": {
            "workload": f"decode/verify step at M={m}: dense K=4096 N=4096+14336, MoE d=2816 128 experts "
                        f"(I=704) top-8 + shared, lm_head 262144x2816 with argmax",
            "m": m,
            "weight_bytes_per_step": bytes_step,
            "bytes": wl["bytes"],
            "active_experts": wl["active_experts"],
            "l2": "inputs larger than L2: each step reads ~0.7 GB of weights (L2 126 MB); no flush",
            "parallelism": f"replicas x{world}" if world > 1 else "single GPU",
        },
        "tokens_per_s": round(world * m / (ms_step * 1e-3), 1),
        "hbm_frac": round(value / world / peak, 4),
        "kernels_us": {k: round(v, 2) for k, v in kernel_us.items()},
        "kernels_gbs": {k: round(wl["bytes"][k] / (kernel_us[k] * 1e-6) / 1e9, 1) for k in kernel_us},
        "roofline": {"bound": "hbm", "kernel": "lm_head_argmax (stream_kernel, argmax epilogue)",
                     "achieved": round(achieved, 1), "launch_us": round(lm_us, 2),
                     "peak": peak, "peak_kind": f"{peak_kind} (copy)", "unit": "GB/s",
                     "frac": round(achieved / peak, 4), "traffic": traffic},
        "e2e": {"value": round(e2e_value, 1), "unit": "GB/s", "h2d_bytes_per_step": h2d, "d2h_bytes_per_step": d2h},
        "graph_ms_per_step": round(graph_ms, 4) if graph_ms else None,
        "prefill": prefill,
        "lm_head_sample": sampling,
        "gpu_launches": launches_per_step * args.steps,
        "timing": "value: steps back to back, events around the region; kernels_us: a second pass with events "
                  "around every call",
        "clocks": clocks.summary(),
    }
    if rank == 0 and not args.no_cpu_baseline and world == 1:
        result["cpu_baseline"] = cpu_baseline(m, seconds=args.cpu_seconds)
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
    nbytes = step_bytes(wl, 0)["lm_head"]
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
    nbytes = step_bytes(wl, active)["moe"]
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


def main():
    ap = argparse.ArgumentParser(description=__doc__, formatter_class=argparse.RawDescriptionHelpFormatter)
    ap.add_argument("--gpus", type=int, default=1)
    ap.add_argument("--steps", type=int, default=50)
    ap.add_argument("--warmup", type=int, default=5)
    ap.add_argument("--m", type=int, default=15)
    ap.add_argument("--impl", choices=("ours", "reference"), default="ours")
    ap.add_argument("--cpu-seconds", type=float, default=10.0)
    ap.add_argument("--prefill-m", type=int, default=512,
                    help="also time the MoE layer on a prefill chunk of this many tokens (0: skip)")
    ap.add_argument("--no-cpu-baseline", action="store_true")
    args = ap.parse_args()
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
