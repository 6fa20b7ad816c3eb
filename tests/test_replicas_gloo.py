"""The N > 1 path of bench.py (independent replicas, one per GPU) on the CPU
with the gloo backend and two ranks: the barrier and the max-over-ranks
timing reduction that turn per-rank times into the reported step time."""
import os
import socket
import sys

import pytest
import torch
import torch.distributed as dist
import torch.multiprocessing as mp

ROOT = os.path.dirname(os.path.dirname(os.path.abspath(__file__)))


def _free_port():
    with socket.socket() as s:
        s.bind(("127.0.0.1", 0))
        return s.getsockname()[1]


def _worker(rank, world, port, out):
    sys.path.insert(0, ROOT)
    os.environ.update(MASTER_ADDR="127.0.0.1", MASTER_PORT=str(port), RANK=str(rank),
                      WORLD_SIZE=str(world), LOCAL_RANK=str(rank))
    import bench
    ws, r, local = bench.dist_env()
    assert (ws, r, local) == (world, rank, rank)
    bench.init_dist(ws, "gloo")
    bench.barrier(ws)
    got = bench.max_over_ranks(1.5 + rank, ws, torch.device("cpu"))
    out[rank] = got
    dist.destroy_process_group()


def test_two_replicas_max_over_ranks():
    world = 2
    port = _free_port()
    ctx = mp.get_context("spawn")
    out = ctx.Manager().dict()
    procs = [ctx.Process(target=_worker, args=(r, world, port, out)) for r in range(world)]
    for p in procs:
        p.start()
    for p in procs:
        p.join(timeout=120)
        assert p.exitcode == 0
    assert dict(out) == {0: 2.5, 1: 2.5}


def test_reference_arm_other_ranks_do_nothing(capsys, monkeypatch):
    sys.path.insert(0, ROOT)
    import bench
    args = type("A", (), dict(gpus=2, steps=1, warmup=3, workload="gpt2-small"))()
    assert bench.run_reference(args, 2, 1) == 0
    assert capsys.readouterr().out == ""


def _worker_one_dies(rank, world, port, out):
    sys.path.insert(0, ROOT)
    os.environ.update(MASTER_ADDR="127.0.0.1", MASTER_PORT=str(port), RANK=str(rank),
                      WORLD_SIZE=str(world), LOCAL_RANK=str(rank), BENCH_DIST_TIMEOUT_S="5")
    import bench
    ws, r, local = bench.dist_env()
    bench.init_dist(ws, "gloo")
    bench.barrier(ws)                      # both ranks reach the first barrier
    if rank == 1:
        os._exit(3)                        # leaves between steps, nothing in flight
    try:
        bench.barrier(ws)                  # the survivor's next collective
        out[rank] = "no error"
    except Exception as e:                 # noqa: BLE001 -- any error is the point
        out[rank] = type(e).__name__


def test_dead_replica_is_reported_not_hung():
    """A rank that exits between steps: the other rank's next barrier ends
    with an error within the process-group timeout instead of waiting."""
    world = 2
    port = _free_port()
    ctx = mp.get_context("spawn")
    out = ctx.Manager().dict()
    procs = [ctx.Process(target=_worker_one_dies, args=(r, world, port, out))
             for r in range(world)]
    for p in procs:
        p.start()
    procs[0].join(timeout=120)
    procs[1].join(timeout=120)
    assert procs[1].exitcode == 3
    assert procs[0].exitcode == 0
    assert out.get(0) not in (None, "no error")
