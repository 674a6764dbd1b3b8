#!/usr/bin/env python
"""Benchmark of the MoE decode layer step on GB300 (one JSON line on rank 0).

    python bench.py [--gpus N] [--steps K] [--warmup W] [--workload ling_m1]
                    [--impl ours|reference] [--sched persistent|...]
                    [--extra tiny_m1,ling_m6,stack_m6,nvfp4_m1,nvfp4_m6]

A step is one MoE layer step (router, top-k, expert gate/up, down, combine with
the shared expert into the residual) over one batch of M token rows; for the
``stack_m6`` workload a step is the 12-layer stack. Weights stay cold: steps
rotate over several distinct full-size layer copies (far more bytes than the
129 MB L2) and over 64 distinct inputs, so the routed experts change every step.

Timed region: exactly K steps, replayed from CUDA graphs that hold them (a graph
of P = min(K, 64) steps replayed K // P times, then a graph of the K % P rest),
bracketed by CUDA events on the launching stream. ``value`` is algorithmic HBM
GB/s over the whole job: the bytes the K steps must read (router + each distinct
routed expert + shared experts) summed over ranks, divided by the max-over-ranks
time. ``step_latency_us`` adds p10 / p50 / p90 over at least 200 single steps,
each launched directly and bracketed by its own events.

The headline workload fills the top-level keys; every other configuration of the
layer step (tiny, Ling M=6, the 12-layer stack, NVFP4 M=1 and M=6) gets a block
of the same fields under ``workloads``, each with its roofline, its CPU-oracle
baseline (1 thread and all cores) and its end-to-end figure.

Multi-GPU: the layer step does not shard (one GPU, no collectives); N processes
run N independent replicas, the timed region is bracketed by barriers and the
max over ranks is taken (weak scaling).

``--impl reference`` times the C++ float64 CPU oracle on the host cores instead
(the only reference that exists for this layer step), on the same workload.
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
import time

ROOT = os.path.dirname(os.path.abspath(__file__))
sys.path.insert(0, ROOT)

METRIC = "MoE decode layer-step µs and achieved HBM GB/s (% of roofline), M=1 and M=6"
NOMINAL_HBM_GBS = 8000.0
FALLBACK_HBM_GBS = 6800.0
CPU_BASELINE_EXTRAS = {"tiny_m1", "ling_m6", "stack_m6", "nvfp4_m1", "nvfp4_m6"}
DEFAULT_EXTRA = ("tiny_m1,ling_m6,ling_m16,stack_m6,nvfp4_m1,nvfp4_m6,ling_fp8_m1,ling_fp8_m6,"
                 "ling_m1_seq,ling_m1_seq_off,ling_m6_seq,ling_m6_seq_off")

from moe_decode_layer_gb300.synth import WORKLOADS  # noqa: E402


# ----------------------------------------------------------------------------- helpers


def measured_peak():
    path = os.path.join(ROOT, "MEASURED_PEAKS.json")
    try:
        with open(path) as f:
            return float(json.load(f)["hbm_gbs"]), "measured"
    except Exception:
        return FALLBACK_HBM_GBS, "fallback"


def sources_digest() -> str:
    """Digest of the CUDA sources: a traffic record holds only for the sources it
    was captured with."""
    import hashlib
    csrc = os.path.join(ROOT, "moe_decode_layer_gb300", "csrc")
    h = hashlib.sha256()
    for name in sorted(os.listdir(csrc)):
        with open(os.path.join(csrc, name), "rb") as f:
            h.update(f.read())
    return h.hexdigest()[:16]


def traffic_record(kernel: str, workload: str):
    """dram read+write bytes per launch from profiles/, if recorded for the
    current kernel sources (a changed kernel invalidates the number)."""
    digest = sources_digest()
    path = os.path.join(ROOT, "profiles", f"{kernel}_{workload}.md")
    if not os.path.exists(path):
        return None, digest
    sha, traffic = None, None
    with open(path) as f:
        for line in f:
            if line.startswith("sources_sha256_16:"):
                sha = line.split(":", 1)[1].strip()
            if line.startswith("traffic_bytes_per_launch:"):
                traffic = float(line.split(":", 1)[1].strip())
    return (traffic if sha == digest else None), digest


class ClockSampler:
    """nvidia-smi clock / throttle samples every 200 ms while running."""

    QUERY = ("index,clocks.sm,clocks.max.sm,power.draw,clocks_event_reasons.active,"
             "clocks_event_reasons.hw_slowdown,clocks_event_reasons.hw_thermal_slowdown,"
             "clocks_event_reasons.sw_thermal_slowdown,clocks_event_reasons.sw_power_cap")

    def __init__(self, gpu_index: int):
        self.gpu = gpu_index
        self.proc = None

    def start(self):
        try:
            self.proc = subprocess.Popen(
                ["nvidia-smi", "-i", str(self.gpu), f"--query-gpu={self.QUERY}", "--format=csv,noheader,nounits",
                 "-lms", "200"], stdout=subprocess.PIPE, stderr=subprocess.DEVNULL, text=True)
        except Exception:
            self.proc = None

    def stop(self):
        if self.proc is None:
            return {"sm_mhz": None, "sm_max_mhz": None, "reasons": ["nvidia-smi unavailable"], "samples": 0}
        self.proc.terminate()
        try:
            out, _ = self.proc.communicate(timeout=5)
        except Exception:
            self.proc.kill()
            out, _ = self.proc.communicate()
        rows = [r for r in csv.reader(io.StringIO(out)) if len(r) >= 9]
        sm, smax, reasons = [], [], set()
        names = ["hw_slowdown", "hw_thermal_slowdown", "sw_thermal_slowdown", "sw_power_cap"]
        for r in rows:
            try:
                sm.append(float(r[1]))
                smax.append(float(r[2]))
            except ValueError:
                continue
            for n, v in zip(names, r[5:9]):
                if v.strip().lower() == "active":
                    reasons.add(n)
        return {"sm_mhz": statistics.median(sm) if sm else None,
                "sm_max_mhz": max(smax) if smax else None,
                "reasons": sorted(reasons), "samples": len(sm)}


def reduce_over_ranks(dist, maxes, sums, device):
    """Max over ranks of `maxes` (times) and sum over ranks of `sums` (work)."""
    import torch
    t = torch.tensor(maxes, dtype=torch.float64, device=device)
    dist.all_reduce(t, op=dist.ReduceOp.MAX)
    b = torch.tensor(sums, dtype=torch.float64, device=device)
    dist.all_reduce(b, op=dist.ReduceOp.SUM)
    return t.tolist(), b.tolist()


def percentiles(v):
    v = sorted(v)
    q = lambda f: v[min(len(v) - 1, int(f * len(v)))]  # noqa: E731
    return {"p10": round(q(0.10), 3), "p50": round(statistics.median(v), 3), "p90": round(q(0.90), 3),
            "n": len(v)}


# ----------------------------------------------------------------------------- our arm


class LayerPool:
    """Distinct full-size layer copies on the device, shared by the workloads that
    use the same layer shape (the stack's 12 layers also serve as the cold copies
    of the single-layer Ling workloads)."""

    def __init__(self, rank: int):
        self.rank = rank
        self.layers = {}

    def get(self, shape_name: str, shape, n: int, w2_layout: str = "h_i"):
        from moe_decode_layer_gb300 import synth
        have = self.layers.setdefault((shape_name, w2_layout), [])
        while len(have) < n:
            have.append(synth.make_layer(shape, seed=1000 + 97 * self.rank + len(have), device="cuda",
                                         w2_layout=w2_layout))
        return have[:n]

    def drop(self, shape_name: str):
        for key in [k for k in self.layers if k[0] == shape_name]:
            self.layers.pop(key, None)


def w2_layout_for(args, shape) -> str:
    """The down-matrix layout the layer copies are built with: "i_h" (transposed,
    the split-K kernel) where --w2-layout asks for it and the format allows it."""
    if args.w2_layout == "i_h" and shape.wdtype != "nvfp4" and args.sched == "persistent":
        return "i_h"
    return "h_i"


def run_workload(name, args, rank, world, dist, pool, steps, warmup, lat_steps, e2e_steps, cpu_seconds):
    """Measure one workload: timed graph replay, latency distribution, e2e, roofline."""
    import torch
    from moe_decode_layer_gb300 import _lib, synth
    from moe_decode_layer_gb300.layer import MoEDecodeLayer

    wl = WORKLOADS[name]
    shape = synth.workload_shape(name)
    m, nl = wl["m"], wl["layers"]
    copies = nl if nl > 1 else args.copies
    layers = pool.get(wl["shape"], shape, copies, w2_layout_for(args, shape))
    mods = [MoEDecodeLayer(shape, layers[i], m, sched=args.sched, pre_rmsnorm=nl > 1) for i in range(copies)]
    n_in = args.inputs
    seq_rho = wl.get("seq_rho")
    if seq_rho is None:
        xs = [synth.hidden_rows(m, shape.hidden, seed=50_000 + 1000 * rank + j, rho=wl["rho"]).cuda()
              for j in range(n_in)]
    else:
        # step j runs layer copy j % copies on the next step of that copy's sequence
        per = max(1, n_in // copies)
        seqs = [synth.decode_sequence(per, m, shape.hidden, seed=60_000 + 1000 * rank + c, rho=wl["rho"],
                                      seq_rho=seq_rho) for c in range(copies)]
        xs = [seqs[j % copies][j // copies].cuda() for j in range(n_in)]
    prefetch = wl.get("prefetch", 0) if args.prefetch is None else args.prefetch
    for md in mods:
        md.set_option(_lib.MOE_OPT_PREFETCH_EXPERTS, prefetch)
    out = torch.empty_like(xs[0])
    stream = torch.cuda.current_stream()

    def step(s):
        if nl == 1:
            mods[s % copies].run(xs[s % n_in], xs[s % n_in], out)
        else:
            out.copy_(xs[s % n_in])
            for layer in mods:
                layer.run(out, out, out)  # pre-norm, residual and output in place

    # algorithmic bytes of each distinct step of the rotation (from the routing)
    period = n_in
    step_bytes = []
    idx = torch.empty((m, shape.top_k), dtype=torch.int32, device="cuda")
    chosen = []
    for s in range(period):
        if nl == 1:
            mods[s % copies].run(xs[s % n_in], xs[s % n_in], out, topk_idx=idx)
            chosen.append(idx.cpu())
            step_bytes.append(synth.algorithmic_bytes(shape, len(set(idx.cpu().flatten().tolist()))))
        else:
            h = xs[s % n_in].clone()
            tot = 0
            for layer in mods:
                layer.run(h, h, h, topk_idx=idx)
                tot += synth.algorithmic_bytes(shape, len(set(idx.cpu().flatten().tolist())))
            step_bytes.append(tot)
    for md in mods:
        st = md.status()
        if st != _lib.MOE_OK:
            raise RuntimeError(f"device status {_lib.status_string(st)}")
    # speculative prefetch: how many of the experts each step prefetched (the
    # previous visit of its layer copy, by the kernel's rule) it then selected
    pf_stats = None
    if prefetch and nl == 1 and period >= 2 * copies:
        hit = tot = sel = 0
        for s in range(copies, period):
            prev, cur = chosen[s - copies], set(chosen[s].flatten().tolist())
            if m == 1:
                pred = prev[0].tolist()[:prefetch]
            else:
                cnt = {}
                for e in prev.flatten().tolist():
                    cnt[e] = cnt.get(e, 0) + 1
                pred = sorted(cnt, key=lambda e: (-cnt[e], e))[:prefetch]
            hit += len(set(pred) & cur)
            tot += len(pred)
            sel += len(cur)
        pf_stats = {"experts": prefetch, "prefetched_then_selected": round(hit / max(tot, 1), 3),
                    "selected_that_were_prefetched": round(hit / max(sel, 1), 3)}

    for s in range(warmup):
        step(s)
    torch.cuda.synchronize()

    # The K timed steps replay from CUDA graphs holding exactly those steps, as a
    # decode loop launches them: P = min(K, period) steps per graph, replayed
    # K // P times, then a graph of the remaining K % P steps.
    K = steps
    P = min(K, period)
    R = K % P
    cs = torch.cuda.Stream()
    cs.wait_stream(stream)
    graphs = []
    for count, first in ((P, 0), (R, K - R)):
        if count == 0:
            graphs.append(None)
            continue
        with torch.cuda.stream(cs):
            for s in range(first, first + count):
                step(s)  # warm the capture stream
        torch.cuda.synchronize()
        g = torch.cuda.CUDAGraph()
        with torch.cuda.graph(g, stream=cs):
            for s in range(first, first + count):
                step(s)
        graphs.append(g)
    torch.cuda.synchronize()
    for g in graphs:
        if g is not None:
            g.replay()
    torch.cuda.synchronize()
    t0, t1 = torch.cuda.Event(enable_timing=True), torch.cuda.Event(enable_timing=True)
    if dist is not None:
        dist.barrier()
    torch.cuda.synchronize()
    torch.cuda.nvtx.range_push("timed")  # ncu --nvtx --nvtx-include "timed/" selects these launches
    t0.record(stream)
    for _ in range(K // P):
        graphs[0].replay()
    if graphs[1] is not None:
        graphs[1].replay()
    t1.record(stream)
    torch.cuda.nvtx.range_pop()
    torch.cuda.synchronize()
    if dist is not None:
        dist.barrier()
    elapsed_ms = t0.elapsed_time(t1)
    # the graph replays cover step s = i mod P for i < K - R, then steps K - R .. K - 1
    bytes_total = sum(step_bytes[(i % P) % period] for i in range(K - R)) + \
        sum(step_bytes[s % period] for s in range(K - R, K))

    # per-step latency: single direct launches, each bracketed by its own events
    ev = [torch.cuda.Event(enable_timing=True) for _ in range(2 * lat_steps)]
    for s in range(lat_steps):
        ev[2 * s].record(stream)
        step(s)
        ev[2 * s + 1].record(stream)
    torch.cuda.synchronize()
    lat_us = [ev[2 * s].elapsed_time(ev[2 * s + 1]) * 1e3 / nl for s in range(lat_steps)]
    for md in mods:
        st = md.status()
        if st != _lib.MOE_OK:
            raise RuntimeError(f"device status {_lib.status_string(st)}")

    # end to end through the host-buffer entry point (copies + sync every step)
    xh = [x.cpu().pin_memory() for x in xs]
    oh = torch.empty_like(xh[0]).pin_memory()
    if nl == 1:
        for s in range(min(10, e2e_steps)):
            mods[s % copies].run_host(xh[s % n_in], xh[s % n_in], oh)
        if dist is not None:
            dist.barrier()
        te = time.perf_counter()
        for s in range(e2e_steps):
            mods[s % copies].run_host(xh[s % n_in], xh[s % n_in], oh)
        e2e_s = time.perf_counter() - te
        h2d, d2h = mods[0].host_copy_bytes(m)  # x (also the residual) in; status words and out back
        e2e_path = ("moe_decode_run_host (pinned host buffers; x doubles as the residual; one copy in, "
                    "one copy of status words + outputs back, sync each step)")
    else:
        if dist is not None:
            dist.barrier()
        te = time.perf_counter()
        for s in range(e2e_steps):
            out.copy_(xh[s % n_in], non_blocking=True)
            for layer in mods:
                layer.run(out, out, out)
            oh.copy_(out, non_blocking=True)
            torch.cuda.synchronize()
        e2e_s = time.perf_counter() - te
        h2d, d2h = m * shape.hidden * 2, m * shape.hidden * 2
        e2e_path = "pinned host copy in, 12 x moe_decode_run in place, copy out, sync"
    e2e_bytes = sum(step_bytes[s % period] for s in range(e2e_steps))

    lat_sorted_us = lat_us
    if dist is not None:
        (elapsed_ms, e2e_s), (bytes_total, e2e_bytes) = reduce_over_ranks(
            dist, [elapsed_ms, e2e_s], [bytes_total, e2e_bytes], "cuda")

    kernels_per_layer = mods[0].info(_lib.MOE_INFO_KERNELS_PER_RUN)
    peak, peak_kind = measured_peak()
    if kernels_per_layer > 1:
        kernel_name = "moe_layer_kernel_chain"
    elif mods[0].info(_lib.MOE_INFO_SPLIT_K):
        kernel_name = "moe_sk_kernel"
    elif mods[0].info(_lib.MOE_INFO_FLAT_ROWS) >> (m - 1) & 1:
        kernel_name = "moe_flat_kernel"
    elif mods[0].info(_lib.MOE_INFO_INTERLEAVED_ROWS) >> (m - 1) & 1:
        kernel_name = "moe_ilv_kernel"
    else:
        kernel_name = "moe_layer_kernel"
    traffic, digest = traffic_record(kernel_name, name)
    ms_step = elapsed_ms / K
    launches_per_step = kernels_per_layer * nl
    # the dominant (single-kernel schedules: only) kernel's mean launch duration
    # over the timed region, and the algorithmic bytes one launch streams
    launch_us = ms_step * 1e3 / launches_per_step
    bytes_per_launch = bytes_total / K / nl / world
    achieved = bytes_per_launch / (launch_us * 1e-6) / 1e9 if kernels_per_layer == 1 else None
    gbs = bytes_total / (elapsed_ms * 1e-3) / 1e9
    res = {
        "metric": METRIC,
        "value": round(gbs, 1),
        "unit": "GB/s",
        "n_gpus": world,
        "steps": K,
        "warmup": warmup,
        "ms_per_step": round(ms_step, 6),
        "higher_is_better": True,
        "scaling": "weak",
        "vs_baseline": None,
        "dtype": shape.wdtype,
        "data": "synthetic",
        "config": {
            "workload": f"{name}: {wl['desc']}",
            "rows_M": m,
            "layers_per_step": nl,
            "sched": args.sched,
            "w2_layout": w2_layout_for(args, shape),
            "expert_prefetch": pf_stats if pf_stats else prefetch,
            "parallelism": f"replicas x{world}" if world > 1 else "single GPU",
            "launch": (f"CUDA graph replay of exactly {K} steps (a {P}-step graph x {K // P}"
                       + (f" + a {R}-step graph" if R else "") + ")"),
            "l2": (f"no flush; inputs larger than L2: weights cold, {copies} distinct full layer copies "
                   f"({copies * (shape.router_bytes() + (shape.num_experts + shape.num_shared) * shape.expert_bytes()) / 1e9:.1f} GB) "
                   f"and {n_in} distinct inputs rotate, far above the 129 MB L2"),
        },
        "us_per_layer_step": round(ms_step * 1e3 / nl, 3),
        "step_latency_us": dict(percentiles(lat_sorted_us),
                                note="single steps launched directly, each bracketed by CUDA events "
                                     "(per layer for the stack)"),
        "tokens_per_s_equiv": round(world * m / (ms_step * 1e-3), 1),
        "bytes_per_step_avg": round(bytes_total / K / world),
        "roofline": {
            "bound": "hbm",
            "achieved": None if achieved is None else round(achieved, 1),
            "peak": peak,
            "unit": "GB/s",
            "frac": None if achieved is None else round(achieved / peak, 4),
            "peak_kind": f"{peak_kind} (STREAM-style copy, MEASURED_PEAKS.json hbm_gbs)",
            "frac_of_nominal_8TBs": None if achieved is None else round(achieved / NOMINAL_HBM_GBS, 4),
            "kernel": kernel_name,
            "kernel_us_per_launch": round(launch_us, 3),
            "algorithmic_bytes_per_launch": round(bytes_per_launch),
            "timing": "launch duration = timed-region time / launches (one launch per layer step)",
            "traffic": traffic,
            "traffic_note": f"ncu dram read+write per launch for kernel sources {digest}" if traffic
            else "no ncu record for the current kernel sources",
        },
        "e2e": {"value": round(e2e_bytes / e2e_s / 1e9, 2), "unit": "GB/s",
                "us_per_step": round(e2e_s / e2e_steps * 1e6, 2), "steps": e2e_steps,
                "h2d_bytes_per_step": h2d, "d2h_bytes_per_step": d2h, "path": e2e_path},
        "gpu_launches": K * launches_per_step,
    }
    if rank == 0 and world == 1 and cpu_seconds > 0:
        res["cpu_baseline"] = cpu_baseline(name, cpu_seconds)
    for md in mods:
        md.close()
    del mods, xs, graphs
    return res


# ----------------------------------------------------------------------------- oracle (CPU) arm


class OracleWorkload:
    """A layer of the workload's shape for the C++ oracle on the host.

    Ling-sized layers are not materialised: the router is drawn once and each
    expert's weights are drawn when a step first selects it (same N(0, 0.02^2)
    recipe as the device layers, from a CPU generator, so not the GPU's values;
    the oracle's cost does not depend on them)."""

    def __init__(self, name: str, seed: int = 7):
        import numpy as np
        import torch
        from moe_decode_layer_gb300 import synth
        self.np, self.torch, self.synth = np, torch, synth
        self.wl = WORKLOADS[name]
        self.shape = synth.workload_shape(name)
        self.seed = seed
        g = torch.Generator().manual_seed(seed)
        r = (torch.randn((self.shape.num_experts, self.shape.hidden), generator=g) * 0.02).to(torch.bfloat16)
        self.router = r.view(torch.int16).numpy().view(np.uint16)
        self.cache = {}

    def expert(self, e, shared=False):
        from oracle import cpp
        key = (shared, e)
        if key not in self.cache:
            torch, np, sh = self.torch, self.np, self.shape
            gg = torch.Generator().manual_seed(self.seed * 1009 + e + (100_003 if shared else 0))
            w13 = torch.randn((2 * sh.inter, sh.hidden), generator=gg) * 0.02
            w2 = torch.randn((sh.hidden, sh.inter), generator=gg) * 0.02
            if sh.wdtype == "bf16":
                bits = lambda t: t.to(torch.bfloat16).view(torch.int16).numpy().view(np.uint16)  # noqa: E731
                self.cache[key] = (bits(w13), bits(w2))
            else:
                qg, sg, tg = self.synth.quantize_nvfp4(w13[:sh.inter])
                qu, su, tu = self.synth.quantize_nvfp4(w13[sh.inter:])
                q2, s2, t2 = self.synth.quantize_nvfp4(w2)
                self.cache[key] = cpp.NVFP4Expert(torch.cat([qg, qu]).numpy(), torch.cat([sg, su]).numpy(),
                                                  np.array([float(tg), float(tu)], np.float32), q2.numpy(),
                                                  s2.numpy(), np.float32(t2))
            if len(self.cache) > 192:
                self.cache.pop(next(iter(self.cache)))
        return self.cache[key]

    def prepare(self, step: int):
        from oracle import cpp
        x = self.synth.hidden_rows(self.wl["m"], self.shape.hidden, seed=90_000 + step, rho=self.wl["rho"])
        xb = x.view(self.torch.int16).numpy().view(self.np.uint16)
        xf = cpp.bf16_bits_to_f64(xb)
        shared = [self.expert(s, True) for s in range(self.shape.num_shared)]
        return cpp.Prepared(xf, xf, self.router, self.expert, shared, self.shape.top_k)


def oracle_timing(name: str, target_s: float, threads: int):
    """Time the C++ oracle on layer steps of the workload for about target_s of
    oracle time (weights gathered outside the timed calls). Returns (s per layer
    step, algorithmic bytes per layer step, steps)."""
    from moe_decode_layer_gb300 import synth
    ow = OracleWorkload(name)
    t_total, b_total, n = 0.0, 0, 0
    wall0 = time.perf_counter()
    while True:
        prep = ow.prepare(n)
        t = time.perf_counter()
        prep.run(threads)
        t_total += time.perf_counter() - t
        b_total += synth.algorithmic_bytes(ow.shape, len(prep.needed))
        n += 1
        if (t_total >= target_s and n >= 2) or time.perf_counter() - wall0 > 4 * target_s + 10:
            break
    return t_total / n, b_total / n, n


def cores_used():
    try:
        return len(os.sched_getaffinity(0))
    except Exception:
        return os.cpu_count()


def cpu_baseline(workload, target_s):
    """The oracle, as it stands, on the host cores: one thread and all cores."""
    from oracle import cpp
    wl = WORKLOADS[workload]
    nl = wl["layers"]
    cores = min(cores_used(), cpp.max_threads())
    t1, b1, n1 = oracle_timing(workload, target_s / 2, 1)
    tn, bn, nn = oracle_timing(workload, target_s / 2, cores)
    return {"value": round(bn / tn / 1e9, 4), "unit": "GB/s", "us_per_step": round(tn * nl * 1e6, 1),
            "cores": cores, "kind": "oracle",
            "one_thread": {"value": round(b1 / t1 / 1e9, 4), "unit": "GB/s", "us_per_step": round(t1 * nl * 1e6, 1),
                           "cores": 1, "steps": n1},
            "sample": f"{nn} (all cores) and {n1} (one thread) layer steps of the {workload} workload through "
                      f"the C++ float64 oracle (router over all experts + the selected and shared experts, "
                      f"OpenMP over output elements), ~{target_s / 2:.1f} s each"
                      + (f"; a step of the {nl}-layer stack is timed as {nl} such layer steps" if nl > 1 else "")
                      + "; expert weights drawn on the CPU with the device recipe, not the GPU's values"}


def run_reference(args, rank, world):
    """The oracle as the reference arm: rank 0 only."""
    if rank != 0:
        return None
    from oracle import cpp
    wl = WORKLOADS[args.workload]
    nl = wl["layers"]
    budget = getattr(args, "ref_seconds", None)
    if budget is None:
        budget = max(1.0, min(10.0, 120.0 / max(1, args.steps + args.warmup))) * (args.steps + args.warmup)
    cores = min(cores_used(), cpp.max_threads())
    t_step, b_step, n = oracle_timing(args.workload, budget, cores)
    t_step *= nl
    b_step *= nl
    v = b_step / t_step / 1e9
    base = {"value": round(v, 4), "unit": "GB/s", "cores": cores, "kind": "oracle",
            "sample": f"{n} layer steps of the {args.workload} workload through the C++ float64 oracle on "
                      f"{cores} host cores (OpenMP)"}
    return {
        "impl": "reference", "metric": METRIC, "value": round(v, 4), "unit": "GB/s", "n_gpus": world,
        "steps": args.steps, "warmup": args.warmup, "ms_per_step": round(t_step * 1e3, 3),
        "higher_is_better": True, "scaling": "weak", "vs_baseline": None,
        "dtype": "f64", "data": "synthetic",
        "config": {"workload": f"{args.workload}: {wl['desc']}", "rows_M": wl["m"], "layers_per_step": nl},
        "cpu_baseline": base,
        "e2e": {"value": round(v, 4), "unit": "GB/s", "h2d_bytes_per_step": 0, "d2h_bytes_per_step": 0},
    }


# ----------------------------------------------------------------------------- main


def main(argv=None):
    ap = argparse.ArgumentParser(description=__doc__, formatter_class=argparse.RawDescriptionHelpFormatter)
    ap.add_argument("--gpus", type=int, default=1)
    ap.add_argument("--steps", type=int, default=2000)
    ap.add_argument("--warmup", type=int, default=50)
    ap.add_argument("--workload", default="ling_m1", choices=sorted(WORKLOADS))
    ap.add_argument("--impl", default="ours", choices=["ours", "reference"])
    ap.add_argument("--sched", default="persistent",
                    choices=["persistent", "phased", "interleaved", "flat", "pdl_chain", "chain"])
    ap.add_argument("--w2-layout", default="h_i", choices=["h_i", "i_h"],
                    help="down matrices [E,H,I] (row-block kernels) or transposed [E,I,H] (split-K kernel; "
                         "bf16 and fp8 workloads under --sched persistent)")
    ap.add_argument("--copies", type=int, default=8, help="distinct layer copies (single-layer workloads)")
    ap.add_argument("--inputs", type=int, default=64,
                    help="distinct input batches the steps rotate over (1: every step routes alike, for "
                         "comparing one launch's DRAM traffic with its algorithmic bytes)")
    ap.add_argument("--prefetch", type=int, default=None,
                    help="experts of the previous step prefetched into L2 while routing (default: the workload's)")
    ap.add_argument("--lat-steps", type=int, default=256, help="single steps for the latency percentiles (>= 200)")
    ap.add_argument("--e2e-steps", type=int, default=500)
    ap.add_argument("--cpu-seconds", type=float, default=6.0, help="oracle CPU baseline sample per workload")
    ap.add_argument("--ref-seconds", type=float, default=None,
                    help="--impl reference: total oracle time (default: ~10 s per step, <= 2 min)")
    ap.add_argument("--extra", default=DEFAULT_EXTRA,
                    help="other workloads measured in the same run (comma list, '' to skip)")
    ap.add_argument("--extra-steps", type=int, default=400, help="timed steps of each extra workload")
    args = ap.parse_args(argv)
    if args.warmup < 3:
        ap.error("--warmup must be >= 3")

    world = int(os.environ.get("WORLD_SIZE", "1"))
    rank = int(os.environ.get("RANK", "0"))
    dist = None
    if world > 1:
        import torch
        import torch.distributed as tdist
        torch.cuda.set_device(int(os.environ.get("LOCAL_RANK", "0")))
        tdist.init_process_group("nccl" if args.impl == "ours" else "gloo")
        dist = tdist

    if args.impl == "reference":
        res = run_reference(args, rank, world)
        if res is not None:
            print(json.dumps(res), flush=True)
        if dist is not None:
            dist.destroy_process_group()
        return 0

    import torch
    dev = int(os.environ.get("LOCAL_RANK", "0"))
    torch.cuda.set_device(dev)
    clocks = ClockSampler(dev)
    clocks.start()
    pool = LayerPool(rank)
    lat = max(200, args.lat_steps)
    res = run_workload(args.workload, args, rank, world, dist, pool, args.steps, args.warmup, lat,
                       min(args.e2e_steps, max(args.steps, 50)), args.cpu_seconds)
    extras = [w for w in args.extra.split(",") if w and w != args.workload] if world == 1 else []
    blocks = {}
    order = sorted(extras, key=lambda w: WORKLOADS[w]["shape"] != WORKLOADS[args.workload]["shape"])
    for name in order:
        shape_name = WORKLOADS[name]["shape"]
        # the oracle's CPU timing for the configurations the pages name; the FP8,
        # M = 16 and decode-sequence extras repeat known shapes
        cpu_s = args.cpu_seconds if name in CPU_BASELINE_EXTRAS else 0.0
        blk = run_workload(name, args, rank, world, None, pool, max(args.extra_steps, 64), max(args.warmup, 10),
                           lat, min(args.e2e_steps, 200), cpu_s)
        blocks[name] = {k: blk[k] for k in ("value", "unit", "ms_per_step", "us_per_layer_step", "step_latency_us",
                                           "tokens_per_s_equiv", "bytes_per_step_avg", "roofline", "e2e",
                                           "cpu_baseline", "config", "steps", "gpu_launches", "dtype")
                        if k in blk}
        if not any(WORKLOADS[w]["shape"] == shape_name for w in order[order.index(name) + 1:]):
            pool.drop(shape_name)
            torch.cuda.empty_cache()
    if blocks:
        res["workloads"] = {k: blocks[k] for k in extras if k in blocks}
    res["clocks"] = clocks.stop()
    if rank == 0:
        print(json.dumps(res), flush=True)
    if dist is not None:
        dist.destroy_process_group()
    return 0


if __name__ == "__main__":
    sys.exit(main())
