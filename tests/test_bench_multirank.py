"""The multi-rank path of bench.py on CPU: two gloo ranks, each a replica,
agree on the slowest rank's time (max over ranks), and one rank alone is the
identity.  No GPU needed."""
import os
import socket
import sys

import pytest
import torch.multiprocessing as mp

ROOT = os.path.dirname(os.path.dirname(os.path.abspath(__file__)))


def _free_port():
    with socket.socket() as s:
        s.bind(("127.0.0.1", 0))
        return s.getsockname()[1]


def _worker(rank, world, port, out):
    sys.path.insert(0, ROOT)
    import torch.distributed as dist
    import bench
    os.environ.update(MASTER_ADDR="127.0.0.1", MASTER_PORT=str(port))
    dist.init_process_group("gloo", rank=rank, world_size=world)
    try:
        out[rank] = bench.replica_seconds(1.0 + 0.5 * rank, world)
    finally:
        dist.destroy_process_group()


@pytest.mark.timeout(120)
def test_replica_time_is_max_over_two_gloo_ranks():
    ctx = mp.get_context("spawn")
    with ctx.Manager() as mgr:
        out = mgr.dict()
        port = _free_port()
        procs = [ctx.Process(target=_worker, args=(r, 2, port, out)) for r in range(2)]
        for p in procs:
            p.start()
        for p in procs:
            p.join(90)
            assert p.exitcode == 0
        assert dict(out) == {0: 1.5, 1: 1.5}


def test_single_rank_identity():
    sys.path.insert(0, ROOT)
    import bench
    assert bench.replica_seconds(0.25, 1) == 0.25
