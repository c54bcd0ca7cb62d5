"""The benchmark's multi-rank path on CPU: two gloo ranks, each timing its own batch
(weak scaling, no collective on the data path); rank results combine as the max of the
times and the sum of the bytes."""
import os
import socket

import pytest
import torch.distributed as dist
import torch.multiprocessing as mp

import bench


def _free_port():
    s = socket.socket()
    s.bind(("127.0.0.1", 0))
    port = s.getsockname()[1]
    s.close()
    return port


def _worker(rank, world, port, q):
    os.environ.update(MASTER_ADDR="127.0.0.1", MASTER_PORT=str(port), RANK=str(rank),
                      WORLD_SIZE=str(world), LOCAL_RANK=str(rank))
    dist.init_process_group("gloo", rank=rank, world_size=world)
    try:
        r, w, local = bench.dist_setup(world)
        assert (r, w, local) == (rank, world, rank)
        t = bench.aggregate_max(1.0 + rank, w)          # per-rank step time
        b = bench.aggregate_sum(100.0 * (rank + 1), w)  # per-rank bytes
        q.put((rank, t, b))
    finally:
        dist.destroy_process_group()


def test_two_gloo_ranks_aggregate_max_time_and_total_bytes():
    world = 2
    ctx = mp.get_context("spawn")
    q = ctx.Queue()
    port = _free_port()
    procs = [ctx.Process(target=_worker, args=(r, world, port, q)) for r in range(world)]
    for p in procs:
        p.start()
    for p in procs:
        p.join(120)
        assert p.exitcode == 0
    got = sorted(q.get(timeout=10) for _ in range(world))
    for rank, t, b in got:
        assert t == 2.0            # slowest rank sets the time
        assert b == 300.0          # bytes of all ranks
    # whole-job throughput = all ranks' bytes / the slowest rank's time
    assert got[0][2] / got[0][1] == 150.0


def test_single_rank_is_identity():
    assert bench.aggregate_max(3.5, 1) == 3.5
    assert bench.aggregate_sum(7.0, 1) == 7.0


def test_reference_arm_exits_quietly_on_other_ranks(monkeypatch, capsys):
    monkeypatch.setenv("RANK", "1")
    monkeypatch.setenv("WORLD_SIZE", "2")

    class A:
        gpus, steps, warmup, workload, seed = 2, 1, 1, 2, None
    bench.run_reference(A())
    assert capsys.readouterr().out == ""
