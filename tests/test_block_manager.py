"""Host block manager: the reference model pinned to the pages' properties, then the
library's native manager compared with the model call by call (no GPU needed).

Properties, by page title and section:
  "深入LLM推理：从KV Cache到PD分离的Serving全景解析", PagedAttention与Cache管理 -- blocks on
      demand (a sequence of n tokens holds ceil(n / BS) blocks), sharing, copy-on-write.
  "ai-infra-7", 优化一：Prefix Cache -- full blocks found again by their chained hash.
  "GPU推理深度拆解：KV Cache视角", 缓存命中与复用 -- hits are a block-granular prefix;
      least-recently-used eviction; blocks in use are never evicted.
"""
import random

import numpy as np
import pytest

import __graft_entry__
import paged_kv_cache_289_gb300 as pkv
from oracle.block_manager import INVALID, NO_BLOCKS, BlockManagerModel, copy_blocks


# ----------------------------------------------------------------------------------
# the model against a hand-worked sequence of calls (values derived by hand from the
# stated policy: smallest free id first, LRU eviction, release last block first)
# ----------------------------------------------------------------------------------
def test_model_hand_worked_sequence():
    m = BlockManagerModel(num_blocks=6, block_size=4)
    # A: 10 tokens -> 3 blocks, two full blocks hashed
    assert m.add_sequence("A", 10, [101, 102]) == ([0, 1, 2], 0)
    # B shares A's first block only (its second hash differs)
    assert m.add_sequence("B", 9, [101, 202]) == ([0, 3, 4], 1)
    assert m.refcount[:6] == [2, 1, 1, 1, 1, 0]
    assert m.available() == 1
    # A leaves: block 2 (unhashed) -> free, block 1 (hash 102) -> cached, block 0 still used
    assert m.free_sequence("A") is None
    assert sorted(m.free) == [2, 5] and m.lru == [1]
    # C repeats A's prefix: both hashed blocks hit (block 1 comes back from the cache)
    assert m.add_sequence("C", 12, [101, 102, 303]) == ([0, 1, 2], 2)
    assert m.lru == [] and sorted(m.free) == [5]
    # D needs 2 blocks, only 1 available -> refused, nothing changes
    before = (list(m.refcount), sorted(m.free), list(m.lru), dict(m.block_of))
    assert m.add_sequence("D", 5, [404]) == NO_BLOCKS
    assert before == (list(m.refcount), sorted(m.free), list(m.lru), dict(m.block_of))
    # C leaves: blocks released 2 (hash 303), 1 (hash 102), 0 (still used by B)
    m.free_sequence("C")
    assert m.lru == [2, 1]
    # E needs 3 blocks: block 5 is free, then the oldest cached blocks 2 and 1 are evicted
    assert m.add_sequence("E", 12, []) == ([5, 2, 1], 0)
    assert 303 not in m.block_of and 102 not in m.block_of and m.block_of[101] == 0
    # B still holds block 0 (hash 101) and was never disturbed
    assert m.block_table("B") == [0, 3, 4]


def test_model_fork_and_copy_on_write():
    m = BlockManagerModel(num_blocks=8, block_size=4)
    assert m.add_sequence("P", 6, [11]) == ([0, 1], 0)
    m.fork("P", "Q")
    assert m.refcount[0] == 2 and m.refcount[1] == 2
    # Q writes into its last (shared, partial) block -> gets block 2, copy 1 -> 2
    assert m.prepare_write("Q", 1) == (1, 2)
    assert m.block_table("Q") == [0, 2] and m.block_table("P") == [0, 1]
    assert m.refcount[1] == 1 and m.refcount[2] == 1
    # P's block 1 is now private and unhashed: written in place
    assert m.prepare_write("P", 1) == (-1, -1)
    # block 0 is registered under hash 11: even a private writer would copy it
    m.free_sequence("Q")
    assert m.refcount[0] == 1
    assert m.prepare_write("P", 0) == (0, 2)
    assert m.lru == [0]          # the hashed original stays cached for later hits
    assert m.add_sequence("R", 4, [11]) == ([0], 1)


def test_model_grow_and_commit():
    m = BlockManagerModel(num_blocks=4, block_size=4)
    assert m.add_sequence(7, 3, []) == ([0], 0)
    assert m.grow(7, 4) == -1                # still one block
    assert m.grow(7, 5) == 1
    assert m.commit_block_hash(7, 1, 99) == INVALID     # block 1 is not full
    assert m.commit_block_hash(7, 0, 99) is None
    assert m.add_sequence(8, 4, [99]) == ([0], 1)
    assert m.grow(7, 3) == INVALID          # shrinking is not a call
    assert m.grow(7, 100) == NO_BLOCKS


# ----------------------------------------------------------------------------------
# the model under random call sequences: invariants the pages fix
# ----------------------------------------------------------------------------------
def _random_hashes(rng, n_full):
    fam = rng.randrange(3)
    share = rng.randrange(n_full + 1)
    return [fam * 1000 + i for i in range(share)] + \
        [rng.getrandbits(63) | (1 << 62) for _ in range(n_full - share)]


def _ops(rng, n_ops, bs):
    live = []
    next_id = 0
    for _ in range(n_ops):
        r = rng.random()
        if r < 0.35 or not live:
            n = rng.randrange(0, 6 * bs)
            nh = rng.randrange(0, n // bs + 1)
            yield ("add", next_id, n, _random_hashes(rng, nh))
            live.append(next_id)
            next_id += 1
        elif r < 0.5:
            yield ("grow", rng.choice(live), rng.randrange(0, 8 * bs))
        elif r < 0.6:
            yield ("fork", rng.choice(live), next_id)
            live.append(next_id)
            next_id += 1
        elif r < 0.75:
            yield ("write", rng.choice(live), rng.randrange(0, 6))
        elif r < 0.85:
            yield ("commit", rng.choice(live), rng.randrange(0, 6), rng.getrandbits(62))
        else:
            s = rng.choice(live)
            yield ("free", s)
            live.remove(s)


def _apply_model(m, op):
    kind = op[0]
    if kind == "add":
        return m.add_sequence(op[1], op[2], op[3])
    if kind == "grow":
        return m.grow(op[1], op[2])
    if kind == "fork":
        return m.fork(op[1], op[2])
    if kind == "write":
        return m.prepare_write(op[1], op[2])
    if kind == "commit":
        return m.commit_block_hash(op[1], op[2], op[3])
    return m.free_sequence(op[1])


@pytest.mark.parametrize("seed", [0, 1, 2, 3])
def test_model_invariants_random(seed):
    rng = random.Random(seed)
    NB, BS = 24, 4
    m = BlockManagerModel(NB, BS)
    release_time = {}     # cached block -> (op index, order within the op)
    evictions = 0
    for t, op in enumerate(_ops(rng, 600, BS)):
        tables_before = {s: list(b) for s, b in m.tables.items()}
        used_before = {b for tb in tables_before.values() for b in tb}
        registered_before = dict(m.block_of)
        cached_before = dict(release_time)
        res = _apply_model(m, op)
        if op[0] == "add" and res not in (INVALID, NO_BLOCKS):
            table, hits = res
            # hits: the longest prefix of hashes registered before the call
            exp = 0
            while exp < len(op[3]) and op[3][exp] in registered_before:
                exp += 1
            assert hits == exp
            assert table[:hits] == [registered_before[h] for h in op[3][:hits]]
        # fresh blocks never come from a table in use
        after_used = {b for tb in m.tables.values() for b in tb}
        for s, tb in m.tables.items():
            old = tables_before.get(s)
            for i, b in enumerate(tb):
                if old is not None and i < len(old) and old[i] == b:
                    continue
                if op[0] in ("fork",) and s == op[2]:
                    continue
                if op[0] == "add" and s == op[1] and i < res[1]:
                    continue          # cache hits
                assert b not in used_before, (t, op, b)
        # an evicted block is the oldest cached one
        if res not in (INVALID, NO_BLOCKS):
            taken = [b for b in after_used - used_before if b in cached_before]
            hit_blocks = set(res[0][:res[1]]) if op[0] == "add" else set()
            evicted = [b for b in taken if b not in hit_blocks]
            if evicted:
                evictions += len(evicted)
                order = sorted(cached_before, key=cached_before.get)
                remaining = [b for b in order if b not in hit_blocks]
                assert sorted(evicted, key=cached_before.get) == remaining[:len(evicted)]
        # bookkeeping of release times for the cached set
        for b in list(release_time):
            if b not in m.lru:
                del release_time[b]
        if op[0] == "free" and res is None:
            for k, b in enumerate(reversed(tables_before[op[1]])):
                if b in m.lru and b not in release_time:
                    release_time[b] = (t, k)
        if op[0] == "write" and res not in (INVALID, NO_BLOCKS) and res[0] >= 0:
            if res[0] in m.lru and res[0] not in release_time:
                release_time[res[0]] = (t, 0)
        # refcount == occurrences in the tables; free / cached / used partition the pool
        occ = [0] * NB
        for tb in m.tables.values():
            for b in tb:
                occ[b] += 1
        assert occ == m.refcount
        free, lru = set(m.free), set(m.lru)
        used = {b for b in range(NB) if occ[b] > 0}
        assert not (free & lru) and not (free & used) and not (lru & used)
        assert len(free) + len(lru) + len(used) == NB
        assert all(b in m.hash_of for b in lru) and not any(b in m.hash_of for b in free)
        # waste under one block per sequence
        for s, tb in m.tables.items():
            assert len(tb) == -(-m.tokens[s] // BS)
    assert evictions > 0


# ----------------------------------------------------------------------------------
# the library's native manager == the model, call by call
# ----------------------------------------------------------------------------------
@pytest.fixture(scope="module")
def built():
    __graft_entry__.build()
    return pkv.lib()


def _apply_native(bm, op):
    try:
        kind = op[0]
        if kind == "add":
            return bm.add_sequence(op[1], op[2], op[3])
        if kind == "grow":
            return bm.grow(op[1], op[2])
        if kind == "fork":
            return bm.fork(op[1], op[2])
        if kind == "write":
            return bm.prepare_write(op[1], op[2])
        if kind == "commit":
            return bm.commit_block_hash(op[1], op[2], op[3])
        return bm.free_sequence(op[1])
    except pkv.PkvError as e:
        return NO_BLOCKS if e.status == pkv.ERR_NO_BLOCKS else INVALID


@pytest.mark.parametrize("seed,NB,BS", [(10, 24, 4), (11, 40, 16), (12, 7, 2), (13, 64, 32)])
def test_native_matches_model(built, seed, NB, BS):
    rng = random.Random(seed)
    m = BlockManagerModel(NB, BS)
    bm = pkv.BlockManager(NB, BS)
    for t, op in enumerate(_ops(rng, 1500, BS)):
        a = _apply_model(m, op)
        b = _apply_native(bm, op)
        assert a == b, (t, op, a, b)
        assert bm.num_available() == m.available()
        if t % 25 == 0:
            for s, tb in m.tables.items():
                assert bm.block_table(s) == tb
            assert [bm.refcount(i) for i in range(NB)] == m.refcount


def test_native_rejects(built):
    bm = pkv.BlockManager(4, 16)
    with pytest.raises(pkv.PkvError):
        bm.add_sequence(1, 16, [1, 2])        # more hashes than full blocks
    bm.add_sequence(1, 16, [5])
    with pytest.raises(pkv.PkvError):
        bm.add_sequence(1, 4)                  # id exists
    for call in (lambda: bm.grow(9, 1), lambda: bm.fork(9, 10), lambda: bm.free_sequence(9),
                 lambda: bm.prepare_write(1, 1), lambda: bm.block_table(9),
                 lambda: bm.refcount(4), lambda: bm.commit_block_hash(1, 1, 3)):
        with pytest.raises(pkv.PkvError) as e:
            call()
        assert e.value.status == -1
    with pytest.raises(pkv.PkvError) as e:
        bm.add_sequence(2, 16 * 4)
    assert e.value.status == pkv.ERR_NO_BLOCKS
    assert bm.num_available() == 3
    L = pkv.lib()
    assert L.pkv_status_string(-5) == b"PKV_ERR_NO_BLOCKS"
    assert L.pkv_bm_create(0, 16, None) == -1


def test_model_copy_blocks_reference():
    """The block-copy reference moves whole blocks (all heads, K and V, scales) and skips
    pairs outside the pool or onto themselves."""
    rng = np.random.default_rng(5)
    k = rng.integers(0, 255, size=(6, 2, 4, 8), dtype=np.uint8)
    v = rng.integers(0, 255, size=(6, 2, 4, 8), dtype=np.uint8)
    ks = rng.random((6, 2)).astype(np.float32)
    vs = rng.random((6, 2)).astype(np.float32)
    k0, v0, ks0, vs0 = k.copy(), v.copy(), ks.copy(), vs.copy()
    copy_blocks(k, v, [[1, 4], [2, 2], [0, 9], [-1, 3], [3, 5]], ks, vs)
    for src, dst in ((1, 4), (3, 5)):
        assert (k[dst] == k0[src]).all() and (v[dst] == v0[src]).all()
        assert (ks[dst] == ks0[src]).all() and (vs[dst] == vs0[src]).all()
    for b in (0, 1, 2, 3):
        assert (k[b] == k0[b]).all() and (v[b] == v0[b]).all() and (ks[b] == ks0[b]).all()
