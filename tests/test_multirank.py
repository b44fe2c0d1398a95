"""Replica aggregation of bench.py across ranks (CPU, gloo, world size 2).

The fused-prefill path has no exchange step: every GPU runs independent
requests, and the bench reports all ranks' tokens over the slowest rank's
time.  This checks the host-side barrier and max-over-ranks reduction with two
gloo processes, and that a rank that fails is reported instead of hanging.
"""
import os
import socket

import pytest
import torch.multiprocessing as mp


def _free_port():
    s = socket.socket()
    s.bind(("127.0.0.1", 0))
    p = s.getsockname()[1]
    s.close()
    return p


def _worker(rank, world, port, values, out, fail_rank):
    import datetime
    import torch.distributed as dist
    os.environ.update(MASTER_ADDR="127.0.0.1", MASTER_PORT=str(port), WORLD_SIZE=str(world), RANK=str(rank),
                      LOCAL_RANK=str(rank))
    dist.init_process_group("gloo", rank=rank, world_size=world, timeout=datetime.timedelta(seconds=20))
    import bench
    try:
        if rank == fail_rank:
            raise RuntimeError("injected failure before the timed region")
        bench.barrier(world)
        out[rank] = bench.reduce_max_over_ranks(values[rank], world)
    except RuntimeError as e:
        out[rank] = -1.0 if "injected" in str(e) else -2.0
    finally:
        if rank != fail_rank:
            dist.destroy_process_group()


def _run(values, fail_rank=-1):
    world = len(values)
    port = _free_port()
    ctx = mp.get_context("spawn")
    out = ctx.Manager().dict()
    procs = [ctx.Process(target=_worker, args=(r, world, port, values, out, fail_rank)) for r in range(world)]
    for p in procs:
        p.start()
    for p in procs:
        p.join(60)
        if p.is_alive():
            p.kill()
    return dict(out)


def test_max_over_two_ranks():
    res = _run([12.5, 40.25])
    assert res == {0: 40.25, 1: 40.25}


def test_failed_rank_is_reported_not_hung():
    res = _run([1.0, 2.0], fail_rank=1)
    assert res[1] == -1.0
    # the surviving rank's collective ends with an error (process-group timeout), never a hang
    assert res.get(0, -2.0) == -2.0
