"""bench.py's multi-replica host logic on CPU with a world_size-2 gloo group:
each rank gets its own batch over the same expert weights, the step time is
the max over ranks, and the job throughput counts every rank's tokens."""

import multiprocessing as mp
import os
import socket

import numpy as np
import pytest


def _free_port():
    with socket.socket() as s:
        s.bind(("127.0.0.1", 0))
        return s.getsockname()[1]


def _rank_main(rank, world, port, q):
    import sys
    root = os.path.dirname(os.path.dirname(os.path.abspath(__file__)))
    sys.path.insert(0, root)
    os.environ.update(MASTER_ADDR="127.0.0.1", MASTER_PORT=str(port), RANK=str(rank), WORLD_SIZE=str(world))
    import torch.distributed as dist
    import bench
    from bit_quantized_moe_quantize_gb300 import synth
    dist.init_process_group("gloo", rank=rank, world_size=world)
    try:
        wl = synth.WORKLOADS["tiny"]
        w, x, ids = bench.make_inputs(wl, 16, rank)
        local_ms = 1.0 + rank            # rank 1 is the slower one
        ms = bench.max_over_ranks(local_ms)
        q.put((rank, x.tobytes(), ids.tobytes(), w.tobytes(), ms, bench.job_throughput(16, world, ms)))
        dist.barrier()
    finally:
        dist.destroy_process_group()


def test_two_replicas_gloo():
    ctx = mp.get_context("spawn")
    q = ctx.Queue()
    port = _free_port()
    procs = [ctx.Process(target=_rank_main, args=(r, 2, port, q)) for r in range(2)]
    for p in procs:
        p.start()
    res = {}
    for _ in range(2):
        r = q.get(timeout=120)
        res[r[0]] = r
    for p in procs:
        p.join(60)
        assert p.exitcode == 0
    assert res[0][1] != res[1][1], "replicas must process different token batches"
    assert res[0][2] != res[1][2]
    assert res[0][3] == res[1][3], "expert weights are replicated"
    assert res[0][4] == res[1][4] == 2.0            # max over ranks
    assert res[0][5] == pytest.approx(16 * 2 / 0.002)


def test_single_process_identity():
    import bench
    assert bench.max_over_ranks(3.5) == 3.5
    assert bench.job_throughput(8191, 1, 1000.0) == pytest.approx(8191.0)


def _ep_rank_main(rank, world, port, q):
    import sys
    root = os.path.dirname(os.path.dirname(os.path.abspath(__file__)))
    sys.path.insert(0, root)
    os.environ.update(MASTER_ADDR="127.0.0.1", MASTER_PORT=str(port), RANK=str(rank), WORLD_SIZE=str(world))
    import torch
    import torch.distributed as dist
    import oracle as oracle_pkg
    from bit_quantized_moe_quantize_gb300 import synth
    dist.init_process_group("gloo", rank=rank, world_size=world)
    try:
        o = oracle_pkg.get()
        case = synth.make_case("tiny", 16)
        w, ids = case["weights"], case["topk_ids"]
        act = o.quantize_q8_1(case["x"])
        E = w.shape[0]
        lo, hi = rank * E // world, (rank + 1) * E // world      # this rank's experts
        part = o.moe_ep(w[lo:hi], act, ids, E, lo)
        total = torch.from_numpy(part.astype(np.float64))
        dist.all_reduce(total)                                     # the combine: a sum over shards
        q.put((rank, total.numpy().tobytes(), o.moe(w, act, ids).astype(np.float64).tobytes()))
        dist.barrier()
    finally:
        dist.destroy_process_group()


def test_expert_parallel_shards_combine_over_gloo():
    """Two ranks each hold half of the experts; every slot routed to another
    rank's expert is a zero row, so one sum over ranks gives the full matmul."""
    ctx = mp.get_context("spawn")
    q = ctx.Queue()
    port = _free_port()
    procs = [ctx.Process(target=_ep_rank_main, args=(r, 2, port, q)) for r in range(2)]
    for p in procs:
        p.start()
    res = [q.get(timeout=120) for _ in range(2)]
    for p in procs:
        p.join(60)
        assert p.exitcode == 0
    for rank, total, full in res:
        got = np.frombuffer(total)
        want = np.frombuffer(full)
        assert np.allclose(got, want, rtol=0, atol=1e-6 * np.abs(want).max())
