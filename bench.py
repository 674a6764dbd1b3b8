#!/usr/bin/env python
"""Benchmark of the MoE decode layer step on GB300 (one JSON line on rank 0).

    python bench.py [--gpus N] [--steps K] [--warmup W] [--workload ling_m1]
                    [--impl ours|reference] [--sched persistent|pdl_chain|chain]

A step is one MoE layer step (router, top-k, expert gate/up, down, combine with
the shared expert into the residual) over one batch of M token rows; for the
``stack_m6`` workload a step is the 12-layer stack. Weights stay cold: steps
rotate over several distinct full-size layer copies (far more bytes than the
129 MB L2) and over 64 distinct inputs, so the routed experts change every step.

``value`` is algorithmic HBM GB/s over the whole job: the bytes a step must read
(router + each distinct routed expert + shared experts) summed over all steps
and ranks, divided by the max-over-ranks device time of the timed region.

Multi-GPU: the layer step does not shard (one GPU, no collectives); N processes
run N independent replicas, the timed region is bracketed by barriers and the
max over ranks is taken (weak scaling).

``--impl reference`` times the float64 CPU oracle on the host cores instead
(the only reference that exists for this layer step), on the same workload.
"""

from __future__ import annotations

import argparse
import csv
import io
import json
import math
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

from moe_decode_layer_gb300.synth import WORKLOADS  # noqa: E402


# ----------------------------------------------------------------------------- helpers


def measured_peak():
    path = os.path.join(ROOT, "MEASURED_PEAKS.json")
    try:
        with open(path) as f:
            return float(json.load(f)["hbm_gbs"]), "measured"
    except Exception:
        return FALLBACK_HBM_GBS, "fallback"


def traffic_record(kernel: str, workload: str):
    """dram read+write bytes per launch from profiles/, if recorded for the
    current kernel sources (a changed kernel invalidates the number)."""
    import hashlib
    csrc = os.path.join(ROOT, "moe_decode_layer_gb300", "csrc")
    h = hashlib.sha256()
    for name in sorted(os.listdir(csrc)):
        with open(os.path.join(csrc, name), "rb") as f:
            h.update(f.read())
    digest = h.hexdigest()[:16]
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


# ----------------------------------------------------------------------------- our arm


def run_ours(args, rank, world, dist):
    import torch
    from moe_decode_layer_gb300 import _lib, synth
    from moe_decode_layer_gb300.layer import MoEDecodeLayer

    wl = WORKLOADS[args.workload]
    shape = synth.workload_shape(args.workload)
    m, nl = wl["m"], wl["layers"]
    dev = int(os.environ.get("LOCAL_RANK", "0"))
    torch.cuda.set_device(dev)
    clocks = ClockSampler(dev)
    clocks.start()

    # distinct layer copies: enough bytes that no weight stays in L2 between uses
    copies = nl if nl > 1 else args.copies
    layers = [synth.make_layer(shape, seed=1000 + 97 * rank + i, device="cuda") for i in range(copies)]
    mods = [MoEDecodeLayer(shape, layers[i], m, sched=args.sched, pre_rmsnorm=nl > 1) for i in range(copies)]
    if args.ring_slots:
        for md in mods:
            md.set_option(_lib.MOE_OPT_RING_SLOTS, min(args.ring_slots, md.info(_lib.MOE_INFO_RING_SLOTS)))
    n_in = 64
    xs = [synth.hidden_rows(m, shape.hidden, seed=50_000 + 1000 * rank + j, rho=wl["rho"]).cuda()
          for j in range(n_in)]
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
    period = n_in if nl == 1 else n_in
    step_bytes = []
    idx = torch.empty((m, shape.top_k), dtype=torch.int32, device="cuda")
    for s in range(period):
        if nl == 1:
            mods[s % copies].run(xs[s % n_in], xs[s % n_in], out, topk_idx=idx)
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

    for s in range(args.warmup):
        step(s)
    torch.cuda.synchronize()

    # The timed steps are replayed from a CUDA graph of one rotation period (as a
    # decode loop launches them); the remainder of K steps launches directly.
    K = args.steps
    graph = torch.cuda.CUDAGraph()
    cs = torch.cuda.Stream()
    cs.wait_stream(stream)
    with torch.cuda.stream(cs):
        for s in range(period):
            step(s)
    torch.cuda.synchronize()
    with torch.cuda.graph(graph, stream=cs):
        for s in range(period):
            step(s)
    torch.cuda.synchronize()
    for _ in range(2):
        graph.replay()
    torch.cuda.synchronize()
    t0, t1 = torch.cuda.Event(enable_timing=True), torch.cuda.Event(enable_timing=True)
    if dist is not None:
        dist.barrier()
    torch.cuda.synchronize()
    torch.cuda.nvtx.range_push("timed")  # ncu --nvtx --nvtx-include "timed/" selects these launches
    t0.record(stream)
    for _ in range(K // period):
        graph.replay()
    for s in range(K - K % period, K):
        step(s)
    t1.record(stream)
    torch.cuda.nvtx.range_pop()
    torch.cuda.synchronize()
    if dist is not None:
        dist.barrier()
    elapsed_ms = t0.elapsed_time(t1)

    # kernel time per launch (CUDA events around sampled direct launches) and the
    # same steps launched one by one from the host
    K2 = min(K, 4000)
    stride = max(1, K2 // 1000)
    ev_a = [torch.cuda.Event(enable_timing=True) for _ in range(0, K2, stride)]
    ev_b = [torch.cuda.Event(enable_timing=True) for _ in range(0, K2, stride)]
    d0, d1 = torch.cuda.Event(enable_timing=True), torch.cuda.Event(enable_timing=True)
    d0.record(stream)
    for s in range(K2):
        if s % stride == 0:
            ev_a[s // stride].record(stream)
            step(s)
            ev_b[s // stride].record(stream)
        else:
            step(s)
    d1.record(stream)
    torch.cuda.synchronize()
    direct_ms = d0.elapsed_time(d1)
    launch_ms = statistics.mean(a.elapsed_time(b) for a, b in zip(ev_a, ev_b))
    for md in mods:
        st = md.status()
        if st != _lib.MOE_OK:
            raise RuntimeError(f"device status {_lib.status_string(st)}")
    clk = clocks.stop()

    bytes_total = sum(step_bytes[s % period] for s in range(K))
    sampled_bytes = statistics.mean(step_bytes[s % period] for s in range(0, K2, stride))

    # end to end through the host-buffer entry point (copies + sync every step)
    k_e2e = min(K, args.e2e_steps)
    if nl == 1:
        xh = [x.cpu().pin_memory() for x in xs]
        oh = torch.empty_like(xh[0]).pin_memory()
        for s in range(min(10, k_e2e)):
            mods[s % copies].run_host(xh[s % n_in], xh[s % n_in], oh)
        if dist is not None:
            dist.barrier()
        te = time.perf_counter()
        for s in range(k_e2e):
            mods[s % copies].run_host(xh[s % n_in], xh[s % n_in], oh)
        e2e_s = time.perf_counter() - te
        h2d, d2h = 2 * m * shape.hidden * 2, m * shape.hidden * 2
    else:
        xh = [x.cpu().pin_memory() for x in xs]
        oh = torch.empty_like(xh[0]).pin_memory()
        if dist is not None:
            dist.barrier()
        te = time.perf_counter()
        for s in range(k_e2e):
            out.copy_(xh[s % n_in], non_blocking=True)
            for layer in mods:
                layer.run(out, out, out)
            oh.copy_(out, non_blocking=True)
            torch.cuda.synchronize()
        e2e_s = time.perf_counter() - te
        h2d, d2h = m * shape.hidden * 2, m * shape.hidden * 2
    e2e_bytes = sum(step_bytes[s % period] for s in range(k_e2e))

    direct_bytes = sum(step_bytes[s % period] for s in range(K2))
    # max over ranks of the times, sum over ranks of the bytes
    if dist is not None:
        (elapsed_ms, e2e_s, launch_ms, direct_ms), (bytes_total, e2e_bytes, direct_bytes) = reduce_over_ranks(
            dist, [elapsed_ms, e2e_s, launch_ms, direct_ms], [bytes_total, e2e_bytes, direct_bytes], "cuda")

    kernels_per_run = mods[0].info(_lib.MOE_INFO_KERNELS_PER_RUN)
    peak, peak_kind = measured_peak()
    if mods[0].info(_lib.MOE_INFO_INTERLEAVED_ROWS) >> (m - 1) & 1:
        kernel_name = "moe_ilv_kernel"
    else:
        kernel_name = "moe_layer_kernel" if args.sched in ("persistent", "phased", "interleaved") else "moe_layer_kernel_chain"
    traffic, digest = traffic_record(kernel_name, args.workload)
    ms_step = elapsed_ms / K
    gbs = bytes_total / (elapsed_ms * 1e-3) / 1e9
    launch_gbs = sampled_bytes / (launch_ms * 1e-3) / 1e9 / (nl if False else 1)
    res = {
        "metric": METRIC,
        "value": round(gbs, 1),
        "unit": "GB/s",
        "n_gpus": world,
        "steps": K,
        "warmup": args.warmup,
        "ms_per_step": round(ms_step, 6),
        "higher_is_better": True,
        "scaling": "weak",
        "vs_baseline": None,
        "dtype": "bf16" if shape.wdtype == "bf16" else "nvfp4",
        "data": "synthetic",
        "config": {
            "workload": f"{args.workload}: {wl['desc']}",
            "rows_M": m,
            "layers_per_step": nl,
            "sched": args.sched,
            "parallelism": f"replicas x{world}" if world > 1 else "single GPU",
            "launch": f"CUDA graph of {period} captured steps, replayed (remainder launched directly)",
            "l2": (f"no flush; weights cold: {copies} distinct full layer copies "
                   f"({copies * (shape.router_bytes() + (shape.num_experts + shape.num_shared) * shape.expert_bytes()) / 1e9:.1f} GB) "
                   f"and {n_in} distinct inputs rotate, far above the 129 MB L2"),
        },
        "us_per_layer_step": round(ms_step * 1e3 / nl, 3),
        "direct_launch": {"value": round(direct_bytes / (direct_ms * 1e-3) / 1e9, 1), "unit": "GB/s",
                          "us_per_layer_step": round(direct_ms * 1e3 / K2 / nl, 3), "steps": K2,
                          "note": "the same steps launched one by one from the host"},
        "tokens_per_s_equiv": round(world * m / (ms_step * 1e-3), 1),
        "bytes_per_step_avg": round(bytes_total / K / world),
        "roofline": {
            "bound": "hbm",
            "achieved": round(launch_gbs, 1),
            "peak": peak,
            "unit": "GB/s",
            "frac": round(launch_gbs / peak, 4),
            "peak_kind": f"{peak_kind} (STREAM-style copy)",
            "frac_of_nominal_8TBs": round(launch_gbs / NOMINAL_HBM_GBS, 4),
            "kernel": kernel_name,
            "kernel_us_per_launch": round(launch_ms * 1e3 / (nl * (1 if args.sched == "persistent" else 1)), 3),
            "traffic": traffic,
            "traffic_note": f"ncu dram read+write per launch for kernel sources {digest}" if traffic
            else "no ncu record for the current kernel sources",
        },
        "e2e": {"value": round(e2e_bytes / e2e_s / 1e9, 2), "unit": "GB/s",
                "us_per_step": round(e2e_s / k_e2e * 1e6, 2), "steps": k_e2e,
                "h2d_bytes_per_step": h2d, "d2h_bytes_per_step": d2h,
                "path": "moe_decode_run_host (pinned host buffers, copies + sync each step)" if nl == 1
                else "host copy in, 12 x moe_decode_run, copy out, sync"},
        "gpu_launches": K * kernels_per_run * nl,
        "clocks": clk,
    }
    return res, (layers, mods, xs, shape, m, nl)


# ----------------------------------------------------------------------------- oracle (CPU) arm


def oracle_step_time(shape, m, rho, target_s, seed=7):
    """Time the float64 oracle on one layer step, repeated for about target_s."""
    import numpy as np
    import torch
    import oracle
    from moe_decode_layer_gb300 import synth

    layer = synth.make_layer(shape, seed=seed, device="cpu") if shape.num_experts <= 64 else None
    rng_experts = {}

    # Ling-sized layers are not materialised on the CPU: each step reads the
    # router and only the experts it selects, drawn lazily (same distribution).
    if layer is None:
        g = torch.Generator().manual_seed(seed)
        router = (torch.randn((shape.num_experts, shape.hidden), generator=g) * 0.02).to(torch.bfloat16)
    else:
        router = layer["router_w"]

    def bits(t):
        return t.contiguous().view(torch.int16).numpy().view(np.uint16) if t.dtype == torch.bfloat16 \
            else t.contiguous().numpy()

    def expert_bits(e, prefix=""):
        key = (prefix, e)
        if key not in rng_experts:
            if layer is not None:
                rng_experts[key] = (bits(layer[prefix + "w13"][e]), bits(layer[prefix + "w2"][e]))
            else:
                gg = torch.Generator().manual_seed(seed * 1009 + e + (7 if prefix else 0))
                if shape.wdtype == "bf16":
                    w13 = (torch.randn((2 * shape.inter, shape.hidden), generator=gg) * 0.02).to(torch.bfloat16)
                    w2 = (torch.randn((shape.hidden, shape.inter), generator=gg) * 0.02).to(torch.bfloat16)
                    rng_experts[key] = (bits(w13), bits(w2))
                else:
                    w13 = torch.randn((2 * shape.inter, shape.hidden), generator=gg) * 0.02
                    w2 = torch.randn((shape.hidden, shape.inter), generator=gg) * 0.02
                    q13, s13, t13 = synth.quantize_nvfp4(w13)
                    q2, s2, t2 = synth.quantize_nvfp4(w2)
                    rng_experts[key] = ((bits(q13), bits(s13), float(t13)), (bits(q2), bits(s2), float(t2)))
        return rng_experts[key]

    def accessor(prefix=""):
        def get(e):
            a, b = expert_bits(e, prefix)
            if shape.wdtype == "bf16":
                return oracle.bf16_bits_to_f64(a), oracle.bf16_bits_to_f64(b)
            return (oracle.dequant_nvfp4_rows(a[0], a[1], a[2]), oracle.dequant_nvfp4_rows(b[0], b[1], b[2]))
        return get

    rbits = bits(router)
    steps, t_total, step_bytes = 0, 0.0, 0
    while True:
        x = synth.hidden_rows(m, shape.hidden, seed=90_000 + steps, rho=rho)
        xb = bits(x)
        # warm the lazily drawn weights outside the timed part
        _, idx, _ = oracle.route(oracle.bf16_bits_to_f64(xb), oracle.bf16_bits_to_f64(rbits), shape.top_k)
        for e in set(idx.ravel().tolist()):
            expert_bits(e)
        for s in range(shape.num_shared):
            expert_bits(s, "sh_")
        t = time.perf_counter()
        xf = oracle.bf16_bits_to_f64(xb)
        shared_get = accessor("sh_")
        oracle.moe_layer(xf, xf, oracle.bf16_bits_to_f64(rbits), accessor(),
                         [shared_get(s) for s in range(shape.num_shared)], shape.top_k)
        t_total += time.perf_counter() - t
        step_bytes += synth.algorithmic_bytes(shape, len(set(idx.ravel().tolist())))
        steps += 1
        rng_experts.clear() if len(rng_experts) > 256 else None
        if t_total >= target_s and steps >= 3:
            break
    return t_total / steps, step_bytes / steps, steps


def cores_used():
    try:
        return len(os.sched_getaffinity(0))
    except Exception:
        return os.cpu_count()


def cpu_baseline(workload, target_s):
    from moe_decode_layer_gb300 import synth
    wl = WORKLOADS[workload]
    shape = synth.workload_shape(workload)
    t_step, b_step, n = oracle_step_time(shape, wl["m"], wl["rho"], target_s)
    t_step *= wl["layers"]  # the stack runs the same layer arithmetic per layer
    b_step *= wl["layers"]
    return {"value": round(b_step / t_step / 1e9, 4), "unit": "GB/s",
            "us_per_step": round(t_step * 1e6, 1), "cores": cores_used(), "kind": "oracle",
            "sample": f"{n} layer steps of the {workload} workload through the float64 numpy oracle "
                      f"(router over all experts + the selected experts), ~{target_s:.0f} s of CPU time; "
                      f"numpy BLAS threads over {cores_used()} cores"}


def run_reference(args, rank, world):
    """The oracle as the reference arm: rank 0 only."""
    if rank != 0:
        return None
    from moe_decode_layer_gb300 import synth
    wl = WORKLOADS[args.workload]
    shape = synth.workload_shape(args.workload)
    # each step is a bounded sample; total CPU time ~ a few minutes at most
    budget = getattr(args, "ref_seconds", None)
    if budget is None:
        budget = max(1.0, min(20.0, 120.0 / max(1, args.steps + args.warmup))) * (args.steps + args.warmup)
    t_step, b_step, n = oracle_step_time(shape, wl["m"], wl["rho"], budget)
    t_step *= wl["layers"]
    b_step *= wl["layers"]
    v = b_step / t_step / 1e9
    base = {"value": round(v, 4), "unit": "GB/s", "cores": cores_used(), "kind": "oracle",
            "sample": f"{n} oracle layer steps on the host cores, workload {args.workload}"}
    return {
        "impl": "reference", "metric": METRIC, "value": round(v, 4), "unit": "GB/s", "n_gpus": world,
        "steps": args.steps, "warmup": args.warmup, "ms_per_step": round(t_step * 1e3, 3),
        "higher_is_better": True, "scaling": "weak", "vs_baseline": None,
        "dtype": "f64", "data": "synthetic",
        "config": {"workload": f"{args.workload}: {wl['desc']}", "rows_M": wl["m"], "layers_per_step": wl["layers"]},
        "cpu_baseline": base,
        "e2e": {"value": round(v, 4), "unit": "GB/s", "h2d_bytes_per_step": 0, "d2h_bytes_per_step": 0},
    }


# ----------------------------------------------------------------------------- main


def main(argv=None):
    ap = argparse.ArgumentParser(description=__doc__, formatter_class=argparse.RawDescriptionHelpFormatter)
    ap.add_argument("--gpus", type=int, default=1)
    ap.add_argument("--steps", type=int, default=20000)
    ap.add_argument("--warmup", type=int, default=2000)
    ap.add_argument("--workload", default="ling_m1", choices=sorted(WORKLOADS))
    ap.add_argument("--impl", default="ours", choices=["ours", "reference"])
    ap.add_argument("--sched", default="persistent", choices=["persistent", "phased", "interleaved", "pdl_chain", "chain"])
    ap.add_argument("--copies", type=int, default=8, help="distinct layer copies (single-layer workloads)")
    ap.add_argument("--e2e-steps", type=int, default=2000)
    ap.add_argument("--ring-slots", type=int, default=0, help="cap on shared-memory ring slots (0 = planned)")
    ap.add_argument("--cpu-seconds", type=float, default=15.0, help="oracle CPU baseline sample length")
    ap.add_argument("--ref-seconds", type=float, default=None,
                    help="--impl reference: total oracle time (default: ~20 s per step, <= 2 min)")
    ap.add_argument("--secondary", default="ling_m6",
                    help="extra workload measured in the same run ('' to skip)")
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

    res, keep = run_ours(args, rank, world, dist)
    del keep
    if args.secondary and args.secondary != args.workload and world == 1:
        import torch
        torch.cuda.empty_cache()
        sec_args = argparse.Namespace(**vars(args))
        sec_args.workload = args.secondary
        sec_args.steps = max(100, args.steps // 4)
        sec_args.warmup = max(10, args.warmup // 4)
        sec, keep = run_ours(sec_args, rank, world, None)
        del keep
        res["secondary"] = {k: sec[k] for k in ("value", "unit", "ms_per_step", "us_per_layer_step",
                                                "tokens_per_s_equiv", "bytes_per_step_avg", "roofline",
                                                "config", "steps", "clocks")}
    if rank == 0 and world == 1 and args.cpu_seconds > 0:
        res["cpu_baseline"] = cpu_baseline(args.workload, args.cpu_seconds)
    if rank == 0:
        print(json.dumps(res), flush=True)
    if dist is not None:
        dist.destroy_process_group()
    return 0


if __name__ == "__main__":
    sys.exit(main())
