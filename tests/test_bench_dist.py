"""Multi-process host logic of bench.py on the CPU (gloo, world size 2).

Each GPU process of an N-GPU run steps an independent virtual rank; only the
timing is combined (slowest rank) and the value aggregates every rank's bytes.
"""
import os
import socket

import pytest
import torch.distributed as dist
import torch.multiprocessing as mp

import bench


def _free_port():
    with socket.socket() as s:
        s.bind(("127.0.0.1", 0))
        return s.getsockname()[1]


def _worker(rank, world, port, out):
    os.environ.update(MASTER_ADDR="127.0.0.1", MASTER_PORT=str(port), RANK=str(rank),
                      WORLD_SIZE=str(world), LOCAL_RANK=str(rank))
    dist.init_process_group("gloo", rank=rank, world_size=world)
    r, w, lr = bench.env_rank()
    local_ms = 10.0 + 5.0 * rank
    slowest = bench.max_over_ranks(local_ms, dist)
    value = bench.whole_job_gbs(70 * 842301952, w, slowest)
    agree = (bench.all_ranks_ok(True, dist), bench.all_ranks_ok(rank != 1, dist))
    out.put((r, w, lr, bench.virtual_rank(r, 8), slowest, value, agree))
    dist.barrier()
    dist.destroy_process_group()


def test_two_ranks_take_the_slowest_time_and_aggregate_bytes():
    ctx = mp.get_context("spawn")
    q = ctx.Queue()
    port = _free_port()
    procs = [ctx.Process(target=_worker, args=(r, 2, port, q)) for r in range(2)]
    for p in procs:
        p.start()
    res = sorted(q.get(timeout=120) for _ in procs)
    for p in procs:
        p.join(timeout=60)
        assert p.exitcode == 0
    assert [x[0] for x in res] == [0, 1] and all(x[1] == 2 for x in res)
    assert [x[3] for x in res] == [0, 1]
    assert all(x[4] == 15.0 for x in res)
    want = 70 * 842301952 * 2 / 15e-3 / 1e9
    assert all(x[5] == pytest.approx(want) for x in res)
    # every rank learns that one rank failed (no rank proceeds alone into a collective)
    assert all(x[6] == (True, False) for x in res)


def test_single_process_is_a_no_op():
    assert bench.max_over_ranks(3.5, None) == 3.5
    assert bench.all_ranks_ok(True, None) and not bench.all_ranks_ok(False, None)
    assert bench.virtual_rank(9, 8) == 1


def _dying_worker(rank, world, port, out):
    import datetime
    os.environ.update(MASTER_ADDR="127.0.0.1", MASTER_PORT=str(port))
    dist.init_process_group("gloo", rank=rank, world_size=world, timeout=datetime.timedelta(seconds=5))
    if rank == 1:
        os._exit(0)  # this rank leaves between steps, before the timing exchange
    try:
        bench.max_over_ranks(10.0, dist)
        out.put((rank, "no error"))
    except Exception as e:  # the survivor must see the failure on the host, not hang
        out.put((rank, "error: %s" % type(e).__name__))


def test_a_rank_that_leaves_is_detected_by_the_other():
    ctx = mp.get_context("spawn")
    q = ctx.Queue()
    port = _free_port()
    procs = [ctx.Process(target=_dying_worker, args=(r, 2, port, q)) for r in range(2)]
    for p in procs:
        p.start()
    rank, status = q.get(timeout=120)
    for p in procs:
        p.join(timeout=60)
    assert rank == 0 and status.startswith("error"), status
