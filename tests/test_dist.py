"""Multi-process host logic of the benchmark on CPU (gloo, world size 2):
each rank serves its own session (distinct seeded inputs, no data exchange),
and the job time is the maximum over ranks."""
import os
import socket

import pytest
import torch
import torch.distributed as dist
import torch.multiprocessing as mp


def _free_port():
    s = socket.socket()
    s.bind(("127.0.0.1", 0))
    port = s.getsockname()[1]
    s.close()
    return port


def _worker(rank, world, port, out):
    os.environ.update(MASTER_ADDR="127.0.0.1", MASTER_PORT=str(port), RANK=str(rank),
                      WORLD_SIZE=str(world), LOCAL_RANK=str(rank))
    dist.init_process_group("gloo", rank=rank, world_size=world)
    import bench
    from bit_plane_kv_gb300 import synth
    w = bench.rank_workload(synth.WORKLOADS["single_4k"], rank)
    q = synth.unit_query(w, 0, "cpu")
    t = bench.max_over_ranks(float(rank + 1) * 0.5, world)
    bench.barrier(world)
    out[rank] = (w.seed, float(q[0, 0]), t)
    dist.destroy_process_group()


def test_two_ranks_serve_independent_sessions():
    world = 2
    mgr = mp.get_context("spawn").Manager()
    out = mgr.dict()
    mp.start_processes(_worker, args=(world, _free_port(), out), nprocs=world, start_method="spawn")
    seeds = {out[r][0] for r in range(world)}
    assert len(seeds) == world                       # distinct sessions
    assert out[0][1] != out[1][1]                    # distinct inputs
    assert out[0][2] == out[1][2] == 1.0             # max over ranks
