"""The multi-replica path of bench.py on CPU: two gloo ranks (the driver runs
one rank per GPU over NCCL with the same code), each an independent request;
the whole-job tokens are summed and the times are the slowest rank's."""
import os
import socket

import pytest
import torch.multiprocessing as mp

ROOT = os.path.dirname(os.path.dirname(os.path.abspath(__file__)))


def _free_port():
    with socket.socket() as s:
        s.bind(("127.0.0.1", 0))
        return s.getsockname()[1]


def _rank(rank, world, port, q):
    import sys
    sys.path.insert(0, ROOT)
    import torch.distributed as dist
    import bench
    dist.init_process_group("gloo", init_method=f"tcp://127.0.0.1:{port}", rank=rank, world_size=world)
    tokens, dec, wall = [(255.0, 1.5, 2.0), (255.0, 1.25, 2.5)][rank]
    out = bench.aggregate_replicas(tokens, dec, wall, "cpu")
    q.put((rank, out))
    dist.barrier()
    dist.destroy_process_group()


def test_two_replicas_aggregate_over_gloo():
    ctx = mp.get_context("spawn")
    q = ctx.Queue()
    port = _free_port()
    procs = [ctx.Process(target=_rank, args=(r, 2, port, q)) for r in range(2)]
    for p in procs:
        p.start()
    res = dict(q.get(timeout=120) for _ in range(2))
    for p in procs:
        p.join(timeout=120)
        assert p.exitcode == 0
    for r in range(2):
        tok, dec, wall = res[r]
        assert tok == 510.0 and dec == 1.5 and wall == 2.5


def test_single_process_is_identity():
    import sys
    sys.path.insert(0, ROOT)
    import bench
    assert bench.aggregate_replicas(10, 2.0, 3.0) == (10.0, 2.0, 3.0)
