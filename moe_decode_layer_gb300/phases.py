"""Phase timeline of the single-kernel MoE decode step from the kernel's own
timestamps (each CTA stores %globaltimer at its phase boundaries).

    python -m moe_decode_layer_gb300.phases --workload ling_m1 [--copies 8]
           [--runs 200] [--ring-slots N]

Prints, per phase boundary, the median / 10th / 90th percentile over CTAs and
runs of the time since the earliest CTA entered the kernel, in microseconds.
Weights rotate over several layer copies so they are cold as in the bench.
"""

from __future__ import annotations

import argparse
import statistics

import torch

from . import _lib, synth
from .layer import MoEDecodeLayer


def timeline(workload: str, copies: int, runs: int, ring_slots: int = 0, sched: str = "persistent",
             n_inputs: int = 64, w2_layout: str = "h_i"):
    wl = synth.WORKLOADS[workload]
    shape = synth.workload_shape(workload)
    m = wl["m"]
    layers = [synth.make_layer(shape, seed=2000 + i, device="cuda", w2_layout=w2_layout) for i in range(copies)]
    mods = [MoEDecodeLayer(shape, layers[i], m, sched=sched) for i in range(copies)]
    grid = mods[0].info(_lib.MOE_INFO_GRID)
    stamps = torch.zeros((grid, _lib.STAMP_SLOTS), dtype=torch.int64, device="cuda")
    for md in mods:
        if ring_slots:
            md.set_option(_lib.MOE_OPT_RING_SLOTS, min(ring_slots, md.info(_lib.MOE_INFO_RING_SLOTS)))
    xs = [synth.hidden_rows(m, shape.hidden, seed=70_000 + j, rho=wl["rho"]).cuda() for j in range(n_inputs)]
    out = torch.empty_like(xs[0])
    per_event = {k: [] for k in _lib.STAMP_NAMES}
    per_count = {k: [] for k in _lib.STAMP_COUNTS}
    totals = []
    derived = {}
    for r in range(runs + 5):
        md = mods[r % copies]
        md.set_option(_lib.MOE_OPT_STAMPS, stamps.data_ptr() if r >= 5 else 0)
        stamps.zero_()
        md.run(xs[r % n_inputs], xs[r % n_inputs], out)
        torch.cuda.synchronize()
        if r < 5:
            continue
        st = stamps.cpu()
        t0 = int(st[:, 0].min())
        for k in _lib.STAMP_NAMES:
            col = st[:, k]
            for v in col.tolist():
                if v:
                    per_event[k].append((v - t0) / 1000.0)
        totals.append((int(st[:, 6].max()) - t0) / 1000.0)
        # per-run derived: the last CTA to store its router logits vs the first
        # CTA to see all logits
        rf = [v for v in st[:, 16].tolist() if v]
        ls = [v for v in st[:, 12].tolist() if v]
        if rf and ls:
            derived.setdefault("last_logits_stored", []).append((max(rf) - t0) / 1000.0)
            derived.setdefault("first_logits_seen", []).append((min(ls) - t0) / 1000.0)
        for k, name in _lib.STAMP_COUNTS.items():
            scale = 1e-3 if "_us" in name else 1.0  # ns sums shown in microseconds
            per_count[k].extend(v * scale for v in st[:, k].tolist() if v)
    for md in mods:
        md.set_option(_lib.MOE_OPT_STAMPS, 0)
        assert md.status() == _lib.MOE_OK
    rows = []
    for k, name in _lib.STAMP_NAMES.items():
        v = sorted(per_event[k])
        if not v:
            continue
        q = lambda f: v[min(len(v) - 1, int(f * len(v)))]  # noqa: E731
        rows.append((name, statistics.median(v), q(0.1), q(0.9), v[-1]))
    for k, name in _lib.STAMP_COUNTS.items():
        v = sorted(per_count[k])
        if v:
            q = lambda f: v[min(len(v) - 1, int(f * len(v)))]  # noqa: E731
            rows.append((name, statistics.median(v), q(0.1), q(0.9), v[-1]))
    for name, v in derived.items():
        v = sorted(v)
        rows.append(("run:" + name, statistics.median(v), v[len(v) // 10], v[(9 * len(v)) // 10], v[-1]))
    return rows, statistics.median(totals), mods[0].info(_lib.MOE_OPT_RING_SLOTS)


def main():
    ap = argparse.ArgumentParser()
    ap.add_argument("--workload", default="ling_m1", choices=sorted(synth.WORKLOADS))
    ap.add_argument("--copies", type=int, default=8)
    ap.add_argument("--runs", type=int, default=200)
    ap.add_argument("--ring-slots", type=int, default=0)
    ap.add_argument("--sweep-ring", default="", help="comma list of ring slot counts to compare")
    ap.add_argument("--hot", action="store_true", help="one layer copy and one input: weights stay in L2")
    ap.add_argument("--sched", default="persistent", help="schedule (see MoEDecodeLayer)")
    ap.add_argument("--w2-layout", default="h_i", choices=["h_i", "i_h"],
                    help="down matrices as stored: i_h (transposed) runs the split-K kernel")
    a = ap.parse_args()
    sweep = [int(v) for v in a.sweep_ring.split(",") if v] or [a.ring_slots]
    for rs in sweep:
        rows, total, used = timeline(a.workload, 1 if a.hot else a.copies, a.runs, rs, sched=a.sched,
                                     n_inputs=1 if a.hot else 64, w2_layout=a.w2_layout)
        print(f"# {a.workload} [{a.sched}]{' (hot: weights in L2)' if a.hot else ''}: ring slots {used}, "
              f"median first-entry -> last-exit {total:.2f} us")
        print(f"{'event':>16} {'median':>8} {'p10':>8} {'p90':>8} {'max':>8}")
        for name, med, p10, p90, mx in rows:
            print(f"{name:>16} {med:8.2f} {p10:8.2f} {p90:8.2f} {mx:8.2f}")


if __name__ == "__main__":
    main()
