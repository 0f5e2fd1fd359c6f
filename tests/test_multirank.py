"""The benchmark's multi-rank host logic (barrier, max over ranks), world size 2 over
gloo on CPU; replicas share nothing else, so nothing else crosses ranks."""
import os
import socket

import torch.distributed as dist
import torch.multiprocessing as mp

import bench


def _free_port():
    with socket.socket() as s:
        s.bind(("127.0.0.1", 0))
        return s.getsockname()[1]


def _worker(rank, world, port, results):
    os.environ.update(MASTER_ADDR="127.0.0.1", MASTER_PORT=str(port))
    dist.init_process_group("gloo", rank=rank, world_size=world)
    dist.barrier()
    ms = 10.0 + 5.0 * rank
    results[rank] = bench.max_over_ranks(ms, dist)
    dist.barrier()
    dist.destroy_process_group()


def test_max_over_ranks_world2():
    ctx = mp.get_context("spawn")
    with ctx.Manager() as m:
        results = m.dict()
        port = _free_port()
        procs = [ctx.Process(target=_worker, args=(r, 2, port, results)) for r in range(2)]
        for p in procs:
            p.start()
        for p in procs:
            p.join(120)
            assert p.exitcode == 0
        assert dict(results) == {0: 15.0, 1: 15.0}


def test_single_rank_is_identity():
    assert bench.max_over_ranks(3.5, None) == 3.5
