"""The multi-rank host logic of bench.py on CPU: world size 2, gloo backend.

Each rank is an independent replica (tokens are independent); the job time is
the slowest rank's, and the whole-job throughput counts every rank's tokens.
"""
import os
import socket

import numpy as np
import pytest
import torch
import torch.distributed as dist
import torch.multiprocessing as mp


def _free_port():
    with socket.socket() as s:
        s.bind(("127.0.0.1", 0))
        return s.getsockname()[1]


def _worker(rank, world, port, q):
    os.environ.update(MASTER_ADDR="127.0.0.1", MASTER_PORT=str(port), RANK=str(rank), WORLD_SIZE=str(world))
    dist.init_process_group("gloo", rank=rank, world_size=world)
    import bench
    ms = [12.5, 20.0][rank]
    worst = bench.max_over_ranks(dist, ms)
    bench.barrier(dist)
    value = bench.whole_job_tokens_per_s(world, 10, 16, worst)
    # each replica routes its own batch: rank-local oracle rows equal the same rows of a joint batch
    import oracle
    from quantised_moe_expert_gb300 import synth
    shape = synth.TINY_SHAPE
    w = synth.make_weights(shape, 0)
    x_all = synth.make_x(shape, 6, 0)
    mine = x_all[rank * 3:(rank + 1) * 3]
    y_mine = oracle.forward(shape, w, mine)["y"]
    gathered = [torch.zeros((3, shape.hidden), dtype=torch.int32) for _ in range(world)]
    dist.all_gather(gathered, torch.from_numpy(y_mine.astype(np.int32)))
    joint = torch.cat(gathered).numpy().astype(np.uint16)
    ok = bool(np.array_equal(joint, oracle.forward(shape, w, x_all)["y"]))
    q.put((rank, worst, value, ok))
    dist.destroy_process_group()


def test_two_rank_max_time_and_weak_scaling_value():
    import oracle
    oracle.build()
    ctx = mp.get_context("spawn")
    q = ctx.Queue()
    port = _free_port()
    procs = [ctx.Process(target=_worker, args=(r, 2, port, q)) for r in range(2)]
    for p in procs:
        p.start()
    for p in procs:
        p.join(120)
        assert p.exitcode == 0
    res = sorted(q.get(timeout=10) for _ in range(2))
    for rank, worst, value, ok in res:
        assert worst == 20.0
        assert value == pytest.approx(2 * 10 * 16 / 0.020)
        assert ok
