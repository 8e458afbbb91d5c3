"""The multi-rank host logic of bench.py on CPU: two gloo ranks (the replicas that
`bench.py --gpus N` runs under torchrun), barrier, max over ranks of the timed region, and
the reference arm running on rank 0 only."""
import multiprocessing as mp
import os
import socket
import sys

import pytest

ROOT = os.path.dirname(os.path.dirname(os.path.abspath(__file__)))


def _free_port() -> int:
    with socket.socket(socket.AF_INET, socket.SOCK_STREAM) as s:
        s.bind(("127.0.0.1", 0))
        return s.getsockname()[1]


def _rank_main(rank: int, world: int, port: int, q):
    try:
        sys.path.insert(0, ROOT)
        os.environ.update(MASTER_ADDR="127.0.0.1", MASTER_PORT=str(port), RANK=str(rank),
                          WORLD_SIZE=str(world), LOCAL_RANK=str(rank))
        import torch.distributed as dist
        dist.init_process_group("gloo", rank=rank, world_size=world)
        import bench
        bench.barrier(world)
        slowest = bench.max_over_ranks(10.0 + rank, world)

        class Args:
            steps, warmup = 1, 0
        ran = None
        if rank != 0:  # the reference arm: ranks other than 0 leave at once, without work
            ran = bench.run_reference(Args())
        bench.barrier(world)
        dist.destroy_process_group()
        q.put((rank, slowest, ran))
    except Exception as e:  # report to the parent instead of hanging it
        q.put((rank, repr(e), None))


def test_two_gloo_ranks_barrier_and_max():
    ctx = mp.get_context("spawn")
    q = ctx.Queue()
    port = _free_port()
    procs = [ctx.Process(target=_rank_main, args=(r, 2, port, q)) for r in range(2)]
    for p in procs:
        p.start()
    out = {}
    for _ in range(2):
        rank, slowest, ran = q.get(timeout=120)
        out[rank] = (slowest, ran)
    for p in procs:
        p.join(timeout=60)
        assert p.exitcode == 0
    assert out[0][0] == 11.0 and out[1][0] == 11.0, out
    assert out[1][1] is None
