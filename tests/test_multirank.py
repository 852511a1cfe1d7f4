"""Host logic of the N-rank benchmark, run as two gloo ranks on the CPU: the
replicas are independent problems (distinct seeds, same shapes), the timing
reduction takes the slowest rank, and barriers pair up."""
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


def _rank_main(rank, world, port, out):
    os.environ.update(MASTER_ADDR="127.0.0.1", MASTER_PORT=str(port), RANK=str(rank),
                      WORLD_SIZE=str(world), LOCAL_RANK=str(rank))
    import bench
    from sdpa_workloads import WORKLOADS
    dist.init_process_group("gloo", rank=rank, world_size=world)
    try:
        w_env, r_env, _ = bench.dist_env()
        assert (w_env, r_env) == (world, rank)
        w = WORKLOADS["mha_causal_b4_h16_l4096_d128"]
        rw = bench.replica_workload(w, rank)
        assert (rw.B, rw.H, rw.Lq, rw.d_k, rw.mask_kind) == (w.B, w.H, w.Lq, w.d_k, w.mask_kind)
        seeds = [None] * world
        dist.all_gather_object(seeds, rw.seed)
        bench.barrier(world)
        slowest = bench.max_over_ranks(1.5 + rank, world, device="cpu")
        out[rank] = (seeds, slowest)
    finally:
        dist.destroy_process_group()


def test_two_gloo_ranks():
    world = 2
    port = _free_port()
    mgr = mp.Manager()
    out = mgr.dict()
    mp.spawn(_rank_main, args=(world, port, out), nprocs=world, join=True)
    seeds0, slow0 = out[0]
    seeds1, slow1 = out[1]
    assert seeds0 == seeds1 and len(set(seeds0)) == world   # distinct replicas
    assert slow0 == slow1 == 2.5                              # max over ranks
