"""The multi-rank host logic of bench.py on CPU ranks (gloo, world size 2).

The path shards by independent heads: every rank runs its own replica of the
workload (no collective touches the data), the timed region's duration is the
maximum over ranks, and the whole-job value counts every rank's steps. Under
torchrun the reference arm runs on rank 0 only; the other ranks exit without
work. These run two spawned processes on 127.0.0.1.
"""
import io
import os
import socket
import sys
from contextlib import redirect_stdout

import pytest
import torch.multiprocessing as mp

ROOT = os.path.dirname(os.path.dirname(os.path.abspath(__file__)))


def _free_port():
    with socket.socket() as s:
        s.bind(("127.0.0.1", 0))
        return s.getsockname()[1]


def _rank_main(rank, world, port, times, out_q):
    sys.path.insert(0, ROOT)
    os.environ.update({"MASTER_ADDR": "127.0.0.1", "MASTER_PORT": str(port), "RANK": str(rank),
                       "WORLD_SIZE": str(world), "LOCAL_RANK": str(rank)})
    import torch
    import torch.distributed as dist

    import bench
    from mxfp4_precision_attention_gb300 import workloads as W

    dist.init_process_group("gloo", rank=rank, world_size=world)
    try:
        w = W.WORKLOADS["wan_32760"]
        assert bench._dist() == (world, rank, rank)
        slowest = bench.max_over_ranks(times[rank], torch.device("cpu"))
        value = bench.job_value(world, w.flops, 10, slowest)
        # the reference arm: rank 0 alone runs and prints; the others return at once
        printed = ""
        if rank != 0:
            buf = io.StringIO()
            with redirect_stdout(buf):
                bench.run_reference(type("A", (), {"gpus": world, "steps": 1, "warmup": 3, "ref_step_s": 1.0})(), w)
            printed = buf.getvalue()
        dist.barrier()
        out_q.put((rank, slowest, value, bench.rank_seed(w, rank), printed))
    finally:
        dist.destroy_process_group()


def test_two_cpu_ranks_max_over_ranks_and_job_value():
    world, times = 2, [0.75, 1.25]
    ctx = mp.get_context("spawn")
    q = ctx.Queue()
    port = _free_port()
    procs = [ctx.Process(target=_rank_main, args=(r, world, port, times, q)) for r in range(world)]
    for p in procs:
        p.start()
    res = sorted(q.get(timeout=120) for _ in range(world))
    for p in procs:
        p.join(timeout=60)
        assert p.exitcode == 0
    import bench
    from mxfp4_precision_attention_gb300 import workloads as W

    w = W.WORKLOADS["wan_32760"]
    for rank, slowest, value, seed, printed in res:
        assert slowest == max(times)                       # every rank sees the slowest rank's time
        assert value == pytest.approx(world * w.flops * 10 / max(times) / 1e12)
        assert seed == w.seed + rank                       # replicas run on distinct inputs
    assert res[1][4] == ""                                 # rank 1 of the reference arm printed nothing
    assert len({r[3] for r in res}) == world


def test_single_process_has_no_collective():
    import torch

    import bench

    assert bench.max_over_ranks(3.5, torch.device("cpu")) == 3.5
    assert bench.job_value(1, 2e12, 5, 10.0) == pytest.approx(1.0)
