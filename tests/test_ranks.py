"""The bench's multi-rank logic on CPU, as two gloo ranks: every rank gets the
slowest rank's time, and the reference arm runs on rank 0 alone."""
import os
import socket
import sys

import pytest

ROOT = os.path.dirname(os.path.dirname(os.path.abspath(__file__)))


def _free_port():
    with socket.socket() as s:
        s.bind(("127.0.0.1", 0))
        return s.getsockname()[1]


def _rank_main(rank, port, values, queue):
    sys.path.insert(0, ROOT)
    os.environ.update(MASTER_ADDR="127.0.0.1", MASTER_PORT=str(port))
    import torch.distributed as dist

    dist.init_process_group("gloo", rank=rank, world_size=2)
    try:
        import bench

        queue.put((rank, bench.max_over_ranks(values[rank], 2, "cpu")))
        dist.barrier()
    finally:
        dist.destroy_process_group()


def test_max_over_ranks_with_two_gloo_ranks():
    import torch.multiprocessing as mp

    ctx = mp.get_context("spawn")
    queue = ctx.Queue()
    port = _free_port()
    values = [0.125, 0.5]
    procs = [ctx.Process(target=_rank_main, args=(r, port, values, queue)) for r in range(2)]
    for p in procs:
        p.start()
    got = dict(queue.get(timeout=120) for _ in range(2))
    for p in procs:
        p.join(timeout=60)
        assert p.exitcode == 0
    assert got == {0: 0.5, 1: 0.5}


def test_max_over_ranks_single_rank_is_the_value():
    sys.path.insert(0, ROOT)
    import bench

    assert bench.max_over_ranks(0.25, 1, "cpu") == 0.25


def test_reference_arm_prints_only_on_rank_0(capsys):
    sys.path.insert(0, ROOT)
    import bench

    class Args:
        config = "tiny"
        steps = 1
        warmup = 0

    assert bench.run_reference(Args(), 1, 2) is None
    assert capsys.readouterr().out == ""
