"""The N > 1 timing logic of bench.py on CPU ranks (gloo, world size 2).

The layer has no data-path exchange (independent output columns and
independent replicas need none), so the multi-rank path is replicas only:
each rank times its own work, the job's time is the maximum over ranks, and
the job's throughput is the work of all ranks divided by that time.  These
checks run the same helpers bench.py uses, over a real gloo process group.
"""
import os
import socket

import pytest
import torch
import torch.distributed as dist
import torch.multiprocessing as mp

ROOT = os.path.dirname(os.path.dirname(os.path.abspath(__file__)))


def _free_port():
    with socket.socket() as s:
        s.bind(("127.0.0.1", 0))
        return s.getsockname()[1]


def _worker(rank, ws, port, q):
    import sys
    sys.path.insert(0, ROOT)
    os.environ.update(MASTER_ADDR="127.0.0.1", MASTER_PORT=str(port), WORLD_SIZE=str(ws),
                      RANK=str(rank), LOCAL_RANK=str(rank))
    dist.init_process_group("gloo", rank=rank, world_size=ws)
    try:
        import bench
        got_ws, got_rank, got_local = bench.dist_info()
        bench.barrier(got_ws)
        # rank r "took" 1 + r seconds; the job's time is the slowest rank's
        t = bench.max_over_ranks(1.0 + rank, got_ws)
        bench.barrier(got_ws)
        q.put((rank, got_ws, got_rank, got_local, t))
    finally:
        dist.destroy_process_group()


def test_max_over_ranks_and_barrier_gloo_two_ranks():
    ws = 2
    ctx = mp.get_context("spawn")
    q = ctx.Queue()
    port = _free_port()
    procs = [ctx.Process(target=_worker, args=(r, ws, port, q)) for r in range(ws)]
    for p in procs:
        p.start()
    for p in procs:
        p.join(timeout=120)
    codes = [p.exitcode for p in procs]
    assert codes == [0, 0], codes
    res = sorted(q.get(timeout=5) for _ in range(ws))
    for rank, got_ws, got_rank, got_local, t in res:
        assert (got_ws, got_rank, got_local) == (ws, rank, rank)
        assert t == pytest.approx(2.0)      # max over ranks, seen identically by every rank


def test_single_rank_needs_no_process_group():
    import sys
    sys.path.insert(0, ROOT)
    import bench
    assert bench.max_over_ranks(3.5, 1) == 3.5
    bench.barrier(1)                        # no process group: a no-op
