"""CPU test of bench.py's multi-process plumbing (world size 2, gloo): the
barrier and the max-over-ranks reduction that turn per-rank timings into the
whole-job number.  The benchmark path itself has no data-path collective
(replicas only)."""
import os
import socket

import pytest
import torch.multiprocessing as mp


def _free_port():
    s = socket.socket()
    s.bind(("127.0.0.1", 0))
    port = s.getsockname()[1]
    s.close()
    return port


def _worker(rank, world, port, out):
    os.environ.update(MASTER_ADDR="127.0.0.1", MASTER_PORT=str(port), RANK=str(rank), WORLD_SIZE=str(world),
                      LOCAL_RANK=str(rank))
    import bench
    r, w, local = bench.dist_env()
    assert (r, w, local) == (rank, world, rank)
    bench.dist_init(w)
    bench.dist_barrier(w)
    out[rank] = bench.dist_max(10.0 * (rank + 1), w)
    import torch.distributed as dist
    dist.destroy_process_group()


def test_dist_max_over_two_ranks():
    port = _free_port()
    out = mp.Manager().dict()
    mp.spawn(_worker, args=(2, port, out), nprocs=2, join=True)
    assert dict(out) == {0: 20.0, 1: 20.0}


def test_single_process_is_identity(monkeypatch):
    for k in ("RANK", "WORLD_SIZE", "LOCAL_RANK"):
        monkeypatch.delenv(k, raising=False)
    import bench
    assert bench.dist_env() == (0, 1, 0)
    assert bench.dist_max(3.5, 1) == 3.5
