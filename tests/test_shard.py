"""Shard plans for a decode batch over several ranks (no collective on the data path).

The planner is checked on its own (cover, order, balance), and then with two gloo
ranks on CPU: each rank takes its shard of one batch -- by requests, or by KV heads
with their query heads -- computes the oracle's attention for that shard alone, and the
gathered shards equal the whole batch's oracle output bit for bit (every output row
depends only on its own unit's inputs)."""
import os
import socket

import numpy as np
import pytest
import torch.distributed as dist
import torch.multiprocessing as mp

import oracle
from paged_kv_cache_289_gb300 import shard
from paged_kv_cache_289_gb300 import workloads as W


def test_plan_requests_covers_in_order_and_balances_tokens():
    rng = np.random.default_rng(3)
    for world in (1, 2, 3, 4, 8):
        for _ in range(20):
            n = int(rng.integers(0, 40))
            lens = rng.integers(0, 5000, size=n)
            plan = shard.plan_requests(lens, world)
            assert len(plan) == world
            assert plan[0][0] == 0 and plan[-1][1] == n
            for (a, b), (c, d) in zip(plan, plan[1:]):
                assert a <= b == c <= d
            if n and lens.sum():
                # no rank exceeds its even share by more than one request's tokens
                share = lens.sum() / world
                for a, b in plan:
                    assert lens[a:b].sum() <= share + lens.max() + 1e-9
    # equal lengths split evenly; fewer requests than ranks leaves ranks empty
    assert shard.plan_requests([10] * 8, 4) == [(0, 2), (2, 4), (4, 6), (6, 8)]
    assert [b - a for a, b in shard.plan_requests([5, 5], 4)].count(0) == 2
    assert shard.plan_requests([0, 0, 0, 0], 2) == [(0, 2), (2, 4)]
    with pytest.raises(ValueError):
        shard.plan_requests([1, 2], 0)


def test_plan_kv_heads_is_contiguous_and_even():
    assert shard.plan_kv_heads(8, 2) == [(0, 4), (4, 8)]
    assert shard.plan_kv_heads(8, 3) == [(0, 3), (3, 6), (6, 8)]
    assert shard.plan_kv_heads(2, 4) == [(0, 1), (1, 2), (2, 2), (2, 2)]
    for H in range(1, 17):
        for world in range(1, 9):
            p = shard.plan_kv_heads(H, world)
            assert p[0][0] == 0 and p[-1][1] == H
            sizes = [b - a for a, b in p]
            assert max(sizes) - min(sizes) <= 1


def _case():
    wl = W.make(2, small=True)
    return wl, W.host_data(wl)


def _shard_output(rank, world, how):
    """The oracle's output for this rank's shard of the batch, computed from the
    shard's own inputs only."""
    wl, d = _case()
    if how == "requests":
        a, b = shard.plan_requests(wl.seq_lens, world)[rank]
        return oracle.decode_attn(d["q"][a:b], d["k_cache"], d["v_cache"], wl.block_table[a:b],
                                  wl.seq_lens[a:b], wl.scale)
    h0, h1 = shard.plan_kv_heads(wl.Hkv, world)[rank]
    G = wl.G
    kc = np.ascontiguousarray(d["k_cache"][:, h0:h1])
    vc = np.ascontiguousarray(d["v_cache"][:, h0:h1])
    q = np.ascontiguousarray(d["q"][:, h0 * G:h1 * G])
    return oracle.decode_attn(q, kc, vc, wl.block_table, wl.seq_lens, wl.scale)


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
        res = {}
        for how in ("requests", "kv_heads"):
            mine = _shard_output(rank, world, how)
            parts = [None] * world
            dist.all_gather_object(parts, mine)
            res[how] = parts
        if rank == 0:
            q.put(res)
    finally:
        dist.destroy_process_group()


def test_two_gloo_ranks_shards_gather_to_the_whole_batch():
    world = 2
    ctx = mp.get_context("spawn")
    qu = ctx.Queue()
    port = _free_port()
    procs = [ctx.Process(target=_worker, args=(r, world, port, qu)) for r in range(world)]
    for p in procs:
        p.start()
    res = qu.get(timeout=300)
    for p in procs:
        p.join(120)
        assert p.exitcode == 0
    wl, d = _case()
    whole = oracle.decode_attn(d["q"], d["k_cache"], d["v_cache"], wl.block_table, wl.seq_lens,
                               wl.scale)
    by_req = np.concatenate(res["requests"], axis=0)
    by_head = np.concatenate(res["kv_heads"], axis=1)
    assert np.array_equal(by_req, whole)
    assert np.array_equal(by_head, whole)
    # both ranks did work
    assert all(p.shape[0] > 0 for p in res["requests"])
    assert all(p.shape[1] == wl.Hq // world for p in res["kv_heads"])
