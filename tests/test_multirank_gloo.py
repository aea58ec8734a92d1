"""The multi-GPU path of bench.py is one independent replica per rank (weak
scaling: the sequences of different ranks never interact), so the only
cross-rank step is the final aggregation: slowest rank's time, all ranks'
tokens.  Checked here with world_size 2 on CPU (gloo)."""
import os
import socket
import sys

import pytest
import torch
import torch.multiprocessing as mp

ROOT = os.path.dirname(os.path.dirname(os.path.abspath(__file__)))


def _free_port():
    s = socket.socket()
    s.bind(("127.0.0.1", 0))
    p = s.getsockname()[1]
    s.close()
    return p


def _worker(rank, world, port, results):
    sys.path.insert(0, ROOT)
    import torch.distributed as dist
    os.environ["MASTER_ADDR"] = "127.0.0.1"
    os.environ["MASTER_PORT"] = str(port)
    dist.init_process_group("gloo", rank=rank, world_size=world)
    import bench
    # rank r: 10 + r seconds, 100 * (r + 1) tokens
    sec, tok = bench.aggregate_over_ranks(10.0 + rank, 100 * (rank + 1), torch.device("cpu"))
    results[rank] = (sec, tok)
    dist.barrier()
    dist.destroy_process_group()


def test_aggregate_over_two_ranks():
    ctx = mp.get_context("spawn")
    manager = ctx.Manager()
    results = manager.dict()
    port = _free_port()
    procs = [ctx.Process(target=_worker, args=(r, 2, port, results)) for r in range(2)]
    for p in procs:
        p.start()
    for p in procs:
        p.join(timeout=120)
        assert p.exitcode == 0
    assert results[0] == results[1] == (11.0, 300)


def test_aggregate_single_process_is_identity():
    sys.path.insert(0, ROOT)
    import bench
    assert bench.aggregate_over_ranks(2.5, 7, torch.device("cpu")) == (2.5, 7)
