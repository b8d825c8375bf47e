"""Weak-scaling bookkeeping of bench.py across ranks (gloo, world size 2, CPU only).

Each rank owns an independent batch (seed = rank): there is no exchange on the data path, so
the only cross-rank steps are the barrier and the reductions of the timing.  This checks that
the whole-job value is the units of all ranks over the slowest rank's time, and that the
ranks' inputs differ while each rank's oracle result is its own.
"""
import os
import socket

import numpy as np
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
    os.environ.update(MASTER_ADDR="127.0.0.1", MASTER_PORT=str(port))
    dist.init_process_group("gloo", rank=rank, world_size=world)
    import bench
    import oracle
    from gqa_attention_learned_head_gb300 import workloads as W

    inp = W.make_decode(2, 4, 1, (16, 64), seed=rank)
    o, lse = oracle.decode(inp.q, inp.k_pages, inp.v_pages, inp.page_table, inp.kv_lens, inp.sinks, inp.scale)
    units = int(inp.kv_lens.sum())
    ms = 1.0 + rank  # rank 1 is the slower one
    bench.barrier(world)
    value, slowest = bench.weak_scaling_value(units, ms, world)
    all_units = [torch.zeros(1, dtype=torch.float64) for _ in range(world)]
    dist.all_gather(all_units, torch.tensor([float(units)], dtype=torch.float64))
    out[rank] = (value, slowest, [float(u) for u in all_units], float(lse.sum()))
    dist.destroy_process_group()


def test_weak_scaling_reduction_two_ranks():
    ctx = mp.get_context("spawn")
    with ctx.Manager() as mgr:
        out = mgr.dict()
        port = _free_port()
        mp.start_processes(_worker, args=(2, port, out), nprocs=2, join=True, start_method="spawn")
        r0, r1 = out[0], out[1]
    units = r0[2]
    assert r0[1] == r1[1] == 2.0                      # slowest rank's ms
    np.testing.assert_allclose(r0[0], sum(units) / 2e-3)
    assert r0[0] == r1[0]
    assert r0[3] != r1[3]                             # independent batches (seed = rank)
