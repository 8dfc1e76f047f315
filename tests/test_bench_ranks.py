"""Multi-rank logic of bench.py on CPU: two gloo ranks, no GPU.

Each rank runs its own problem of the full workload (weak scaling, no
collective on the data path); the reported time is the slowest rank's and the
throughput counts every rank's work.
"""
import os
import socket

import pytest
import torch
import torch.distributed as dist
import torch.multiprocessing as mp

ROOT = os.path.dirname(os.path.dirname(os.path.abspath(__file__)))


def _free_port() -> int:
    with socket.socket() as s:
        s.bind(("127.0.0.1", 0))
        return s.getsockname()[1]


def _rank_main(rank, world, port, out):
    import sys
    sys.path.insert(0, ROOT)
    dist.init_process_group("gloo", init_method=f"tcp://127.0.0.1:{port}", rank=rank, world_size=world)
    import bench
    import synth
    w = synth.WORKLOADS[0]
    # rank r pretends its timed region took 1 + r ms
    ms = bench.max_over_ranks(1.0 + rank, torch.device("cpu"))
    x = synth.make_inputs(w, device="cpu", seed=bench.rank_seed(w, rank))
    out.put((rank, ms, bench.job_throughput(w.flops(), world, ms), float(x["q"].float().sum()),
             bench.runs_reference(rank)))
    dist.barrier()
    dist.destroy_process_group()


def test_two_gloo_ranks_take_the_slowest_time_and_own_problems():
    world = 2
    ctx = mp.get_context("spawn")
    q = ctx.Queue()
    port = _free_port()
    procs = [ctx.Process(target=_rank_main, args=(r, world, port, q)) for r in range(world)]
    for p in procs:
        p.start()
    res = sorted(q.get(timeout=120) for _ in range(world))
    for p in procs:
        p.join(timeout=60)
        assert p.exitcode == 0
    import sys
    sys.path.insert(0, ROOT)
    import synth
    flops = synth.WORKLOADS[0].flops()
    for rank, ms, value, _, _ in res:
        assert ms == pytest.approx(2.0)                       # max over ranks
        assert value == pytest.approx(flops * world / 2e-3 / 1e12)
    assert res[0][3] != res[1][3]                             # independent inputs per rank
    assert [r[4] for r in res] == [True, False]               # reference arm on rank 0 only


def test_single_process_needs_no_group():
    import sys
    sys.path.insert(0, ROOT)
    import bench
    assert bench.max_over_ranks(3.5, torch.device("cpu")) == 3.5
    assert bench.job_throughput(2e12, 1, 1000.0) == pytest.approx(2.0)
