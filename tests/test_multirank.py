"""The multi-process path of bench.py on CPU: two gloo ranks (world size 2)
exchange their timings through the same max-over-ranks reduction the GPU
replicas use over NCCL, and read their rank from the torchrun environment.
The path has no data-path collective (independent replicas, weak scaling), so
this is all the exchange there is."""
import os
import socket
import sys

import torch.multiprocessing as mp

ROOT = os.path.dirname(os.path.dirname(os.path.abspath(__file__)))


def _free_port():
    with socket.socket(socket.AF_INET, socket.SOCK_STREAM) as s:
        s.bind(("127.0.0.1", 0))
        return s.getsockname()[1]


def _rank_main(rank, world, port, q):
    os.environ.update(MASTER_ADDR="127.0.0.1", MASTER_PORT=str(port), RANK=str(rank),
                      WORLD_SIZE=str(world), LOCAL_RANK=str(rank))
    sys.path.insert(0, ROOT)
    import torch
    import torch.distributed as dist
    import bench
    dist.init_process_group("gloo", rank=rank, world_size=world)
    try:
        w, r, local = bench.dist_env()
        # each rank reports its own elapsed time; every rank must get the max
        t = bench.barrier_max(1.5 + rank, w, torch)
        q.put((r, w, local, t))
    finally:
        dist.destroy_process_group()


def test_two_gloo_ranks_agree_on_the_max_time():
    ctx = mp.get_context("spawn")
    q = ctx.Queue()
    port = _free_port()
    procs = [ctx.Process(target=_rank_main, args=(r, 2, port, q)) for r in range(2)]
    for p in procs:
        p.start()
    try:
        got = sorted(q.get(timeout=120) for _ in procs)
    finally:
        for p in procs:
            p.join(timeout=60)
            if p.is_alive():
                p.kill()
    assert got == [(0, 2, 0, 2.5), (1, 2, 1, 2.5)]
    assert all(p.exitcode == 0 for p in procs)
