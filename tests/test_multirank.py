"""Host logic of the multi-GPU bench (replicas, max over ranks) on gloo, world size 2."""
import os
import socket

import torch
import torch.distributed as dist
import torch.multiprocessing as mp

import bench


def _free_port():
    s = socket.socket()
    s.bind(("127.0.0.1", 0))
    port = s.getsockname()[1]
    s.close()
    return port


def _worker(rank, world, port, out):
    dist.init_process_group("gloo", init_method=f"tcp://127.0.0.1:{port}", rank=rank, world_size=world)
    try:
        ms = [3.0, 7.5][rank]
        got = bench.max_over_ranks(ms, dist, "cpu")
        seed = bench.replica_seed(1, rank)
        seeds = [None] * world
        dist.all_gather_object(seeds, seed)
        out[rank] = (got, seeds)
        dist.barrier()
    finally:
        dist.destroy_process_group()


def test_replicas_and_max_over_ranks():
    world = 2
    port = _free_port()
    mgr = mp.Manager()
    out = mgr.dict()
    mp.spawn(_worker, args=(world, port, out), nprocs=world, join=True)
    for r in range(world):
        got, seeds = out[r]
        assert got == 7.5                      # every rank sees the slowest rank's time
        assert len(set(seeds)) == world        # independent replicas
    assert bench.max_over_ranks(4.0, None) == 4.0


def test_algorithmic_bytes_of_decode_workload():
    from csa2_inputs import workloads
    wl = workloads.decode_128k()
    alg = bench.algorithmic(wl)
    assert alg["scan_bytes"] == 32 * 32768 * 256 == 268435456
    assert alg["gathered_bytes"] == 32 * 512 * 288
    assert alg["scan_bytes"] // 32 + alg["gathered_bytes"] // 32 == 8536064   # per sequence
