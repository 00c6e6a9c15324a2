"""The multi-process path of bench.py on CPU: two gloo ranks, each timing its
own replica; the job's time is the maximum over ranks and its work the sum."""
import os
import socket

import torch
import torch.distributed as tdist
import torch.multiprocessing as mp


def _free_port():
    with socket.socket() as s:
        s.bind(("127.0.0.1", 0))
        return s.getsockname()[1]


def _worker(rank, world, port, out):
    os.environ.update(MASTER_ADDR="127.0.0.1", MASTER_PORT=str(port))
    tdist.init_process_group("gloo", rank=rank, world_size=world)
    import bench
    mx, sm = bench.reduce_ranks([10.0 + rank, 3.0 * rank], [100.0 * (rank + 1), 1.0], "cpu")
    out[rank] = (mx, sm)
    tdist.barrier()
    tdist.destroy_process_group()


def test_reduce_over_two_gloo_ranks():
    ctx = mp.get_context("spawn")
    mgr = ctx.Manager()
    out = mgr.dict()
    port = _free_port()
    procs = [ctx.Process(target=_worker, args=(r, 2, port, out)) for r in range(2)]
    for p in procs:
        p.start()
    for p in procs:
        p.join(timeout=120)
        assert p.exitcode == 0
    for r in range(2):
        mx, sm = out[r]
        assert mx == [11.0, 3.0]       # slowest rank's time
        assert sm == [300.0, 2.0]      # all ranks' work


def test_reduce_single_process_is_identity():
    import bench
    assert bench.reduce_ranks([1.5, 2.0], [3.0], "cpu") == ([1.5, 2.0], [3.0])


def test_reference_arm_prints_only_on_rank0(monkeypatch):
    import argparse
    import bench
    args = argparse.Namespace(steps=1, warmup=0, workload="mimo")
    assert bench.run_reference(args, rank=1, world=2) is None
