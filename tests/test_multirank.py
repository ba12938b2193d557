"""Multi-rank host logic of bench.py on CPU: two gloo ranks, weak scaling.

The decode shards by batch (each rank decodes its own sequences, no data-path
collective); the bench reports the slowest rank's time and the sum of the
ranks' tokens.  This checks that aggregation with real gloo collectives."""
import os
import socket
import sys

import torch.multiprocessing as mp

ROOT = os.path.dirname(os.path.dirname(os.path.abspath(__file__)))


def _free_port():
    with socket.socket() as s:
        s.bind(("127.0.0.1", 0))
        return s.getsockname()[1]


def _rank(rank, world, port, out):
    os.environ.update(MASTER_ADDR="127.0.0.1", MASTER_PORT=str(port), RANK=str(rank),
                      WORLD_SIZE=str(world))
    sys.path.insert(0, ROOT)
    import torch.distributed as dist
    import bench
    dist.init_process_group("gloo", rank=rank, world_size=world)
    el, tok = bench.aggregate_ranks(1.0 + rank, 100.0 * (rank + 1), world, "cpu")
    out[rank] = (el, tok)
    dist.barrier()
    dist.destroy_process_group()


def test_two_rank_aggregation_gloo():
    world = 2
    mgr = mp.get_context("spawn").Manager()
    out = mgr.dict()
    ctx = mp.get_context("spawn")
    port = _free_port()
    procs = [ctx.Process(target=_rank, args=(r, world, port, out)) for r in range(world)]
    for p in procs:
        p.start()
    for p in procs:
        p.join(timeout=120)
        assert p.exitcode == 0
    # slowest rank's time, summed tokens, identical on every rank
    assert out[0] == (2.0, 300.0) and out[1] == (2.0, 300.0)


def test_single_rank_is_identity():
    sys.path.insert(0, ROOT)
    import bench
    assert bench.aggregate_ranks(1.5, 42.0, 1, "cpu") == (1.5, 42.0)
