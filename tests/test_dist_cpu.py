"""The multi-process path of bench.py on CPU: two gloo ranks (127.0.0.1) reduce their times and bytes
the way the bench does (the slowest rank's time, the sum of the bytes every replica streamed), and the
reference arm leaves all work to rank 0."""
import os
import socket
import sys

import pytest
import torch
import torch.distributed as dist
import torch.multiprocessing as mp

ROOT = os.path.dirname(os.path.dirname(os.path.abspath(__file__)))
sys.path.insert(0, ROOT)


def free_port():
    with socket.socket() as s:
        s.bind(("127.0.0.1", 0))
        return s.getsockname()[1]


def _rank_main(rank, world, port, q):
    os.environ.update(MASTER_ADDR="127.0.0.1", MASTER_PORT=str(port), RANK=str(rank), WORLD_SIZE=str(world),
                      LOCAL_RANK=str(rank))
    dist.init_process_group("gloo", rank=rank, world_size=world)
    try:
        import bench
        w, r, local = bench.dist_env()
        secs = 1.0 + 0.5 * rank         # rank 1 is the slower one
        nbytes = 1000 * (rank + 1)      # each replica streams its own bytes
        q.put((r, w, local, bench.over_ranks(secs, nbytes, w, device="cpu")))
    finally:
        dist.destroy_process_group()


def test_over_ranks_two_gloo_ranks():
    world = 2
    ctx = mp.get_context("spawn")
    q = ctx.Queue()
    port = free_port()
    procs = [ctx.Process(target=_rank_main, args=(r, world, port, q)) for r in range(world)]
    for p in procs:
        p.start()
    got = sorted(q.get(timeout=120) for _ in range(world))  # drain before joining
    for p in procs:
        p.join(timeout=60)
    assert all(p.exitcode == 0 for p in procs)
    for r, (rank, w, local, (secs, total)) in enumerate(got):
        assert (rank, w, local) == (r, world, r)
        assert secs == 1.5          # the slowest rank's time
        assert total == 3000.0      # every replica's bytes


def test_over_ranks_single_process_is_identity():
    import bench
    assert bench.over_ranks(2.5, 1234, 1) == (2.5, 1234.0)


def test_reference_arm_runs_on_rank_zero_only(monkeypatch):
    import bench
    monkeypatch.setenv("RANK", "1")
    monkeypatch.setenv("WORLD_SIZE", "2")

    class Args:  # any attribute access would mean rank 1 did work
        def __getattr__(self, name):
            raise AssertionError(f"rank 1 read args.{name}")

    assert bench.run_reference(Args()) is None
