"""bench.py's multi-GPU path is N independent replicas (the layer's tensor
parallelism runs as virtual partitions inside one GPU): every rank times its
own replica, the job is timed by the slowest rank and only rank 0 prints.
Checked here with two gloo ranks on the CPU."""
import os
import socket

import pytest
import torch.distributed as dist
import torch.multiprocessing as mp

import bench


def _free_port():
    with socket.socket() as s:
        s.bind(("127.0.0.1", 0))
        return s.getsockname()[1]


def _rank_main(rank, world, port, q):
    os.environ.update(MASTER_ADDR="127.0.0.1", MASTER_PORT=str(port), RANK=str(rank),
                      WORLD_SIZE=str(world), LOCAL_RANK=str(rank))
    dist.init_process_group("gloo", rank=rank, world_size=world)
    try:
        my_ms = 100.0 + 50.0 * rank            # rank 1 is the slower replica
        bench.barrier(world)
        slowest = bench.max_over_ranks(my_ms, world)
        value = bench.replica_throughput(world, 4096, 10, slowest)
        # the reference arm does no work on ranks other than 0
        args = type("A", (), {"workload": "c1", "ref_prefix": 4, "warmup": 0, "steps": 1,
                              "gpus": world})()
        if rank != 0:
            bench.run_reference(args, world, rank)
        q.put((rank, slowest, value))
    finally:
        dist.destroy_process_group()


def test_two_replicas_timed_by_slowest_rank():
    world, port = 2, _free_port()
    ctx = mp.get_context("spawn")
    q = ctx.Queue()
    procs = [ctx.Process(target=_rank_main, args=(r, world, port, q)) for r in range(world)]
    for p in procs:
        p.start()
    for p in procs:
        p.join(timeout=120)
        assert p.exitcode == 0
    results = sorted(q.get(timeout=5) for _ in range(world))
    for rank, slowest, value in results:
        assert slowest == 150.0
        assert value == pytest.approx(2 * 4096 * 10 / 0.150)
