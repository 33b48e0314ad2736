"""Multi-rank host logic of the benchmark on CPU (gloo, world size 2).

The attention path shards by (batch, head) with no collective on the data
path: every rank runs its own independent problem, and only the timing is
reduced (max over ranks). This checks that logic without a GPU."""
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
    os.environ["MASTER_ADDR"] = "127.0.0.1"
    os.environ["MASTER_PORT"] = str(port)
    dist.init_process_group("gloo", rank=rank, world_size=world)
    import bench
    from exact_io_aware_108_b300 import inputs
    # each rank draws a different, independent problem
    w = inputs.WORKLOADS["fwd_b1_h2_n256_d64_f16"]
    t = inputs.make_qkv(w.B, w.H, w.N, w.d, w.dtype, seed=w.seed + bench.rank_seed_offset(rank))
    local_ms = 10.0 + 5.0 * rank          # rank 1 is the slow one
    ms_max = bench.max_over_ranks(local_ms, dist)
    rate = bench.whole_job_rate(1e12, ms_max, world)
    out[rank] = (ms_max, rate, float(t["q"].float().sum()))
    dist.barrier()
    dist.destroy_process_group()


def test_two_ranks_weak_scaling_host_logic():
    world = 2
    port = _free_port()
    mgr = mp.Manager()
    out = mgr.dict()
    mp.spawn(_worker, args=(world, port, out), nprocs=world, join=True)
    (m0, r0, s0), (m1, r1, s1) = out[0], out[1]
    assert m0 == m1 == 15.0                       # max over ranks
    assert r0 == r1 == pytest.approx(2 * 1e12 / 15e-3 / 1e12)
    assert s0 != s1                               # independent problems per rank
