"""The multi-replica bench path on CPU: two gloo ranks, each with its own
time, agree on the largest (the job's time); the reference arm does its work
on rank 0 only."""

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


def _rank_main(rank, world, port, times, out):
    import torch.distributed as dist

    sys.path.insert(0, ROOT)
    import bench

    os.environ.update(MASTER_ADDR="127.0.0.1", MASTER_PORT=str(port), RANK=str(rank), LOCAL_RANK=str(rank),
                      WORLD_SIZE=str(world))
    dist.init_process_group("gloo", rank=rank, world_size=world)
    try:
        r, lr, w = bench.dist_env()
        got = bench.max_over_ranks(times[rank], dist, "cpu")
        out.put((rank, r, lr, w, got))
    finally:
        dist.destroy_process_group()


def test_max_over_ranks_two_gloo_ranks():
    ctx = mp.get_context("spawn")
    q = ctx.Queue()
    port = _free_port()
    times = [5.25, 7.5]
    procs = [ctx.Process(target=_rank_main, args=(r, 2, port, times, q)) for r in range(2)]
    for p in procs:
        p.start()
    res = sorted(q.get(timeout=120) for _ in procs)
    for p in procs:
        p.join(timeout=60)
        assert p.exitcode == 0
    assert [(r, lr, w) for _, r, lr, w, _ in res] == [(0, 0, 2), (1, 1, 2)]
    assert all(got == max(times) for *_, got in res)


def test_max_over_ranks_single_process_is_identity():
    sys.path.insert(0, ROOT)
    import bench

    assert bench.max_over_ranks(3.5, None, "cpu") == 3.5


def test_reference_arm_other_ranks_do_no_work(capsys):
    sys.path.insert(0, ROOT)
    import bench

    class Args:
        workload, seed, warmup, steps, gpus = "n32_c1_int8", 0, 1, 1, 2

    bench.run_reference(Args, 1, 2)  # rank 1 of 2: returns at once, prints nothing
    assert capsys.readouterr().out == ""
