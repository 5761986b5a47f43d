"""World-size-2 gloo checks (CPU) of the bench's multi-rank host logic: the
path shards as independent replicas, so the only cross-rank steps are the
barrier and the max-over-ranks of the timed region; the reference arm runs
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


def _worker(rank, world, port, out):
    sys.path.insert(0, ROOT)
    os.environ.update(MASTER_ADDR="127.0.0.1", MASTER_PORT=str(port), RANK=str(rank),
                      WORLD_SIZE=str(world), LOCAL_RANK=str(rank),
                      OSATTN_DIST_BACKEND="gloo")
    import bench

    r, local, w = bench.dist_setup(world)
    assert (r, local, w) == (rank, rank, world)
    bench.barrier(w)
    got = bench.reduce_max(10.0 + 5.0 * rank, w)
    out[rank] = got
    import torch.distributed as dist

    dist.destroy_process_group()


def test_reduce_max_over_two_gloo_ranks():
    port = _free_port()
    ctx = mp.get_context("spawn")
    out = ctx.Manager().dict()
    procs = [ctx.Process(target=_worker, args=(r, 2, port, out)) for r in range(2)]
    for p in procs:
        p.start()
    for p in procs:
        p.join(120)
        assert p.exitcode == 0
    assert out[0] == 15.0 and out[1] == 15.0


def test_reference_arm_exits_on_non_zero_rank(monkeypatch, capsys):
    sys.path.insert(0, ROOT)
    import bench

    monkeypatch.setenv("RANK", "1")
    monkeypatch.setenv("WORLD_SIZE", "2")
    assert bench.main(["--impl", "reference", "--steps", "1", "--warmup", "0"]) == 0
    assert capsys.readouterr().out == ""
