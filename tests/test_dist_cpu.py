"""CPU, world size 2 over gloo: the multi-rank path of bench.py.

Every rank is an independent replica of the experts forward (the forward has
no exchange step on one GPU), so the only cross-rank step is the timing: the
job's time is the maximum over ranks and the whole-job throughput is
world x per-rank work / that time. Each rank here also runs the fp64 oracle
on its own replica batch to check that replicas stay independent.
"""
import os
import socket

import numpy as np
import pytest
import torch
import torch.distributed as dist
import torch.multiprocessing as mp


def _free_port():
    s = socket.socket()
    s.bind(("127.0.0.1", 0))
    p = s.getsockname()[1]
    s.close()
    return p


def _worker(rank, world, port, q):
    os.environ.update(MASTER_ADDR="127.0.0.1", MASTER_PORT=str(port), RANK=str(rank), WORLD_SIZE=str(world),
                      LOCAL_RANK=str(rank))
    dist.init_process_group("gloo", rank=rank, world_size=world)
    try:
        import bench
        from block_scaled_moe_expert_gb300 import workloads as W
        import oracle.moe as OM
        assert bench.dist_env() == (world, rank, rank)
        t = bench.max_over_ranks(10.0 + rank)
        wl = W.scaled(W.WORKLOADS["tiny_fp8"], T=4)
        hid, idx, w, wt = W.make_all(wl)
        wt = {k: (v.numpy() if torch.is_tensor(v) else v) for k, v in wt.items()}
        out = OM.experts_forward(hid.view(torch.int16).numpy().view(np.uint16), idx.numpy(), w.numpy(), wt)
        gathered = [torch.zeros(4, wl.H, dtype=torch.float64) for _ in range(world)]
        dist.all_gather(gathered, torch.from_numpy(out))
        same = all(torch.equal(g, gathered[0]) for g in gathered)
        q.put((rank, t, bench.replica_throughput(100.0, world, 2.0), same))
    finally:
        dist.destroy_process_group()


def test_two_rank_replicas_over_gloo():
    world = 2
    ctx = mp.get_context("spawn")
    q = ctx.Queue()
    port = _free_port()
    procs = [ctx.Process(target=_worker, args=(r, world, port, q)) for r in range(world)]
    for p in procs:
        p.start()
    for p in procs:
        p.join(timeout=120)
        assert p.exitcode == 0
    res = sorted(q.get(timeout=5) for _ in range(world))
    assert [r[1] for r in res] == [11.0, 11.0]      # max over ranks on every rank
    assert [r[2] for r in res] == [100.0, 100.0]    # 2 ranks x 100 units / 2 s
    assert all(r[3] for r in res)                   # identical replicas
