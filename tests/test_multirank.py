"""World-size-2 check of the benchmark's multi-rank host logic on CPU (gloo): every rank
gets its own independent layer (weak scaling, no data-path collective), the step time is
the max over ranks, and the whole-job value counts the work of every rank."""
import os
import socket

import pytest
import torch
import torch.distributed as dist
import torch.multiprocessing as mp


def _free_port():
    with socket.socket() as s:
        s.bind(("127.0.0.1", 0))
        return s.getsockname()[1]


def _worker(rank, world, port, out):
    os.environ.update(MASTER_ADDR="127.0.0.1", MASTER_PORT=str(port), RANK=str(rank),
                      WORLD_SIZE=str(world))
    dist.init_process_group("gloo", rank=rank, world_size=world)
    import bench
    import kvp_inputs
    w = bench.rank_workload(kvp_inputs.QWEN3_4B_LAYER, rank)
    ms = bench.reduce_max(1.0 + 2.0 * rank, world)           # rank 1 is the slow one
    dist.barrier()
    out[rank] = (w.seed, ms, bench.whole_job_tflops(1e12, world, ms))
    dist.destroy_process_group()


def test_two_ranks_gloo():
    world = 2
    port = _free_port()
    with mp.Manager() as man:
        out = man.dict()
        mp.spawn(_worker, args=(world, port, out), nprocs=world, join=True)
        res = dict(out)
    seeds = {res[r][0] for r in range(world)}
    assert len(seeds) == world                      # independent problems per rank
    assert all(res[r][1] == 3.0 for r in range(world))   # max over ranks
    assert all(abs(res[r][2] - 2e12 / 3e-3 / 1e12) < 1e-9 for r in range(world))


def test_single_rank_passthrough():
    import bench
    assert bench.reduce_max(4.5, 1) == 4.5
    assert bench.whole_job_tflops(2e12, 1, 2.0) == pytest.approx(1000.0)
