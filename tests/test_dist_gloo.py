"""The N > 1 host logic of bench.py on CPU ranks (gloo, world size 2): the
job's time is the slowest rank's, the matrix count is the sum over ranks,
and the reference arm prints only on rank 0."""

import os
import socket

import pytest
import torch
import torch.distributed as dist
import torch.multiprocessing as mp


def _free_port() -> int:
    with socket.socket() as s:
        s.bind(("127.0.0.1", 0))
        return s.getsockname()[1]


def _worker(rank, world, port, q):
    os.environ.update(MASTER_ADDR="127.0.0.1", MASTER_PORT=str(port), RANK=str(rank),
                      WORLD_SIZE=str(world), LOCAL_RANK=str(rank))
    dist.init_process_group("gloo", rank=rank, world_size=world)
    import bench
    ws, r, local = bench.dist_info()
    t = bench.max_over_ranks(100.0 + 50.0 * rank, ws, "cpu")
    n = bench.sum_over_ranks(168.0, ws, "cpu")
    bench.barrier(ws)
    q.put((rank, ws, r, local, t, n))
    dist.destroy_process_group()


def test_two_rank_aggregation():
    ctx = mp.get_context("spawn")
    q = ctx.Queue()
    port = _free_port()
    procs = [ctx.Process(target=_worker, args=(r, 2, port, q)) for r in range(2)]
    for p in procs:
        p.start()
    out = sorted(q.get(timeout=120) for _ in range(2))
    for p in procs:
        p.join(timeout=60)
        assert p.exitcode == 0
    for rank, ws, r, local, t, n in out:
        assert ws == 2 and r == rank and local == rank
        assert t == 150.0          # slowest rank
        assert n == 336.0          # matrices of both ranks


def _ref_worker(rank, world, port, q):
    import contextlib
    import io
    os.environ.update(MASTER_ADDR="127.0.0.1", MASTER_PORT=str(port), RANK=str(rank),
                      WORLD_SIZE=str(world), LOCAL_RANK=str(rank))
    import bench
    buf = io.StringIO()
    with contextlib.redirect_stdout(buf):
        args = type("A", (), {"steps": 0, "warmup": 0, "gpus": world})()
        if rank != 0:
            bench.run_reference(args)
    q.put((rank, buf.getvalue()))


def test_reference_arm_silent_on_other_ranks():
    ctx = mp.get_context("spawn")
    q = ctx.Queue()
    p = ctx.Process(target=_ref_worker, args=(1, 2, _free_port(), q))
    p.start()
    rank, text = q.get(timeout=120)
    p.join(timeout=60)
    assert p.exitcode == 0 and rank == 1 and text == ""
