"""The benchmark's N > 1 host path on CPU: two gloo ranks, each timing its own
replica; the reported time is the max over ranks and the token count covers
every rank (weak scaling, no data-path collective).  A rank that leaves makes
the other's timing reduction fail within the process group's timeout."""
import os
import socket
import time

import pytest
import torch.multiprocessing as mp


def _free_port():
    s = socket.socket()
    s.bind(("127.0.0.1", 0))
    port = s.getsockname()[1]
    s.close()
    return port


def _rank_main(rank, world, port, out):
    import torch.distributed as dist
    import bench
    os.environ.update(MASTER_ADDR="127.0.0.1", MASTER_PORT=str(port))
    dist.init_process_group("gloo", rank=rank, world_size=world)
    mine = [1.0 + rank, 10.0 - rank]
    got = bench.max_over_ranks(mine, world)
    out.put((rank, got, bench.replica_tokens(1, 128, 5, world)))
    dist.barrier()
    dist.destroy_process_group()


def test_two_rank_max_and_tokens():
    ctx = mp.get_context("spawn")
    q = ctx.Queue()
    port = _free_port()
    procs = [ctx.Process(target=_rank_main, args=(r, 2, port, q)) for r in range(2)]
    for p in procs:
        p.start()
    res = sorted(q.get(timeout=120) for _ in procs)
    for p in procs:
        p.join(timeout=60)
        assert p.exitcode == 0
    for rank, got, toks in res:
        assert got == [2.0, 10.0]
        assert toks == 1 * 128 * 5 * 2


def _report_and_exit(out, msg):
    out.put(msg)
    out.close()
    out.join_thread()   # the message is sent before the process ends
    os._exit(0)         # no process-group teardown with a peer gone


def _leaving_rank_main(rank, world, port, out):
    import bench
    os.environ.update(MASTER_ADDR="127.0.0.1", MASTER_PORT=str(port), RANK=str(rank),
                      WORLD_SIZE=str(world), C2KV_RANK_TIMEOUT_S="5")
    bench.init_ranks("gloo")
    if rank == 1:   # leaves between steps: nothing of it is in flight
        _report_and_exit(out, (rank, "left", 0.0))
    t0 = time.monotonic()
    try:
        bench.max_over_ranks([1.0, 2.0], world)
        what = "no error"
    except RuntimeError:
        what = "error"
    _report_and_exit(out, (rank, what, time.monotonic() - t0))


def test_a_rank_that_leaves_fails_the_timing_reduction():
    ctx = mp.get_context("spawn")
    q = ctx.Queue()
    port = _free_port()
    procs = [ctx.Process(target=_leaving_rank_main, args=(r, 2, port, q)) for r in range(2)]
    for p in procs:
        p.start()
    res = dict((r, (what, dt)) for r, what, dt in (q.get(timeout=120) for _ in procs))
    for p in procs:
        p.join(timeout=60)
    assert res[1][0] == "left"
    assert res[0][0] == "error" and res[0][1] < 60.0, res[0]


def test_single_rank_is_identity():
    import bench
    assert bench.max_over_ranks([3.0, 4.0], 1) == [3.0, 4.0]
