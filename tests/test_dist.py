"""The multi-process path of the bench on CPU (gloo, world size 2): replicas time
independently, the job's time is the max over ranks and its work the sum."""

import os
import socket

import torch
import torch.distributed as dist
import torch.multiprocessing as mp


def _free_port():
    s = socket.socket()
    s.bind(("127.0.0.1", 0))
    port = s.getsockname()[1]
    s.close()
    return port


def _worker(rank, world, port, results):
    os.environ.update(MASTER_ADDR="127.0.0.1", MASTER_PORT=str(port))
    dist.init_process_group("gloo", rank=rank, world_size=world)
    import bench
    maxes, sums = bench.reduce_over_ranks(dist, [10.0 + rank, 5.0 - rank], [100.0 * (rank + 1)], "cpu")
    dist.barrier()
    results[rank] = (maxes, sums)
    dist.destroy_process_group()


def test_reduce_over_two_ranks():
    ctx = mp.get_context("spawn")
    mgr = ctx.Manager()
    results = mgr.dict()
    port = _free_port()
    procs = [ctx.Process(target=_worker, args=(r, 2, port, results)) for r in range(2)]
    for p in procs:
        p.start()
    for p in procs:
        p.join(120)
        assert p.exitcode == 0
    for r in range(2):
        maxes, sums = results[r]
        assert maxes == [11.0, 5.0]
        assert sums == [300.0]


def test_reference_arm_runs_on_rank_zero_only(monkeypatch, capsys):
    import bench
    import argparse
    args = argparse.Namespace(workload="tiny_m1", steps=1, warmup=3, ref_seconds=0.2)
    assert bench.run_reference(args, rank=1, world=2) is None
    res = bench.run_reference(args, rank=0, world=1)
    assert res["impl"] == "reference" and res["unit"] == "GB/s" and res["value"] > 0
    assert res["e2e"]["h2d_bytes_per_step"] == 0 and res["cpu_baseline"]["kind"] == "oracle"
