"""The multi-rank benchmark logic on CPU with gloo (world size 2).

Each rank runs its own replica on its own sequences (weak scaling, no
collective on the data path); ranks only meet in a barrier and in the
max-over-ranks reduction of the step time.
"""
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


def _worker(rank, world, port, q):
    sys.path.insert(0, ROOT)
    os.environ.update(MASTER_ADDR="127.0.0.1", MASTER_PORT=str(port), RANK=str(rank),
                      WORLD_SIZE=str(world))
    import torch.distributed as dist
    import bench
    dist.init_process_group("gloo", rank=rank, world_size=world)
    t = bench.reduce_max(10.0 + rank * 5.0, dist, "cpu")
    dist.barrier()
    tags = bench.rank_tags(rank, 16)
    q.put((rank, t, tags))
    dist.destroy_process_group()


def test_two_ranks_partition_and_max_time():
    ctx = mp.get_context("spawn")
    q = ctx.Queue()
    port = _free_port()
    procs = [ctx.Process(target=_worker, args=(r, 2, port, q)) for r in range(2)]
    for p in procs:
        p.start()
    out = [q.get(timeout=120) for _ in procs]
    for p in procs:
        p.join(timeout=60)
        assert p.exitcode == 0
    out.sort()
    assert [o[1] for o in out] == [15.0, 15.0]          # both ranks see the max
    t0, t1 = set(out[0][2]), set(out[1][2])
    assert len(t0) == len(t1) == 16 and not (t0 & t1)   # disjoint sequences


def test_reference_arm_is_rank0_only(monkeypatch, capsys):
    sys.path.insert(0, ROOT)
    import bench
    monkeypatch.setenv("RANK", "1")

    class A:
        steps, warmup = 1, 1
    bench.reference_arm(A())          # returns at once on a non-zero rank
    assert capsys.readouterr().out == ""
