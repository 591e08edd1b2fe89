"""The multi-GPU host logic on CPU: two gloo ranks, as torchrun would start them.

Each rank draws its own shard of heads (weak scaling, no collective on the data
path); the benchmark's only collectives are a barrier and a MAX all-reduce of the
timings, and the whole-job value counts every rank's work over the slowest
rank's time.
"""
import os
import socket

import pytest
import torch
import torch.distributed as dist
import torch.multiprocessing as mp

WORLD = 2


def _free_port():
    with socket.socket() as s:
        s.bind(("127.0.0.1", 0))
        return s.getsockname()[1]


def _rank_main(rank, world, port, queue):
    import sys
    root = os.path.dirname(os.path.dirname(os.path.abspath(__file__)))
    sys.path.insert(0, root)
    import bench
    from fa_inputs import WORKLOADS, make_qkv
    os.environ.update(MASTER_ADDR="127.0.0.1", MASTER_PORT=str(port))
    dist.init_process_group("gloo", rank=rank, world_size=world)
    try:
        w = WORKLOADS["tiny"]
        q, _, _ = make_qkv(w.shape, w.dtype, bench.shard_seed(w, rank))
        mine = torch.tensor([float(q.double().sum()), float(bench.shard_seed(w, rank))], dtype=torch.float64)
        got = [torch.zeros(2, dtype=torch.float64) for _ in range(world)]
        dist.all_gather(got, mine)
        dist.barrier()
        t = torch.tensor([100.0 + 25.0 * rank], dtype=torch.float64)      # this rank's timed ms
        dist.all_reduce(t, op=dist.ReduceOp.MAX)
        value = bench.aggregate_tflops(w.flops(False), 10, world, float(t))
        queue.put((rank, [g.tolist() for g in got], float(t), value))
    finally:
        dist.destroy_process_group()


def test_two_gloo_ranks_shard_and_reduce():
    ctx = mp.get_context("spawn")
    queue = ctx.Queue()
    port = _free_port()
    procs = [ctx.Process(target=_rank_main, args=(r, WORLD, port, queue)) for r in range(WORLD)]
    for p in procs:
        p.start()
    results = [queue.get(timeout=120) for _ in range(WORLD)]
    for p in procs:
        p.join(timeout=60)
        assert p.exitcode == 0
    results.sort()
    gathered = results[0][1]
    assert all(r[1] == gathered for r in results)                 # every rank sees the same shards
    assert gathered[0][1] != gathered[1][1] and gathered[0][0] != gathered[1][0]   # distinct shards
    assert all(r[2] == 125.0 for r in results)                   # slowest rank's time
    from fa_inputs import WORKLOADS
    want = WORLD * WORKLOADS["tiny"].flops(False) * 10 / 0.125 / 1e12
    assert all(abs(r[3] - want) < 1e-12 for r in results)
