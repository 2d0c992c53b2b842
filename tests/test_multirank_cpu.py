"""The multi-rank host logic of bench.py on CPU (gloo, world size 2): ranks meet
at the barriers that bracket a timed region, the slowest rank's time is the one
reported, and the oracle arm runs on rank 0 only (the other ranks exit without
work).  No GPU and no kernel is involved."""
import os
import socket

import pytest
import torch
import torch.distributed as dist
import torch.multiprocessing as mp


def _free_port():
    with socket.socket() as s:
        s.bind(("127.0.0.1", 0))
        return s.getsockname()[1]


def _worker(rank, world, port, out):
    os.environ.update(MASTER_ADDR="127.0.0.1", MASTER_PORT=str(port), RANK=str(rank),
                      WORLD_SIZE=str(world), LOCAL_RANK=str(rank))
    import bench
    r, w, _ = bench.rank_info()
    assert (r, w) == (rank, world)
    bench.dist_init(w)
    assert dist.get_backend() == "gloo"
    bench.barrier(w)
    slowest = bench.max_over_ranks(1.5 + rank, w)         # rank times 1.5 and 2.5 ms
    ref = None
    if rank != 0:
        ref = bench.run_reference(None, rank, w)           # returns before touching args
    bench.barrier(w)
    out[rank] = (slowest, ref)
    dist.destroy_process_group()


@pytest.mark.timeout(120)
def test_two_ranks_gloo():
    world = 2
    port = _free_port()
    with mp.Manager() as mgr:
        out = mgr.dict()
        mp.spawn(_worker, args=(world, port, out), nprocs=world, join=True)
        res = dict(out)
    assert res[0][0] == pytest.approx(2.5) and res[1][0] == pytest.approx(2.5)
    assert res[1][1] == 0
