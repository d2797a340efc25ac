"""Host logic of bench.py's multi-process path on CPU (gloo, world size 2).

Under torchrun each rank runs an independent replica of the workload; the
timed region is bracketed by barriers, the time is the maximum over ranks
and the throughput counts the tokens of all ranks.  These tests run that
logic in two spawned CPU processes: no GPU and no collective on a data path.
"""
import os
import socket

import pytest
import torch.multiprocessing as mp

import bench


def _free_port() -> int:
    with socket.socket() as s:
        s.bind(("127.0.0.1", 0))
        return s.getsockname()[1]


def _worker(rank, world, port, out):
    import torch.distributed as dist
    os.environ.update(MASTER_ADDR="127.0.0.1", MASTER_PORT=str(port), RANK=str(rank),
                      WORLD_SIZE=str(world), LOCAL_RANK=str(rank))
    dist.init_process_group("gloo", rank=rank, world_size=world)
    try:
        r, w, local = bench.dist_env()
        assert (r, w, local) == (rank, world, rank)
        bench.dist_barrier()
        # each rank reports its own time; every rank must see the slowest one
        t = bench.dist_max(1.5 + rank)
        out.put((rank, t, bench.throughput(32768, 10, w, t)))
        bench.dist_barrier()
    finally:
        dist.destroy_process_group()


def test_max_over_ranks_and_whole_job_throughput():
    ctx = mp.get_context("spawn")
    q = ctx.Queue()
    port = _free_port()
    procs = [ctx.Process(target=_worker, args=(r, 2, port, q)) for r in range(2)]
    for p in procs:
        p.start()
    for p in procs:
        p.join(timeout=120)
    assert all(p.exitcode == 0 for p in procs), [p.exitcode for p in procs]
    res = sorted(q.get(timeout=10) for _ in range(2))
    for rank, t, tput in res:
        assert t == pytest.approx(2.5)              # max over the two ranks
        assert tput == pytest.approx(32768 * 10 * 2 / 2.5)


def test_single_process_helpers_need_no_process_group():
    assert bench.dist_max(3.25) == 3.25
    bench.dist_barrier()
    assert bench.throughput(1000, 4, 1, 2.0) == 2000.0
