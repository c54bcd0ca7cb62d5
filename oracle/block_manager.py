"""Plain reference model of the host block manager and of the block copy.

TEST INFRASTRUCTURE ONLY, like the rest of this package: the tests compare the
library's native block manager and its copy kernel with this model.  Plain
Python lists and dicts, every decision spelled out, no attempt at speed.

What it models, by page title and section:
  [P1] "深入LLM推理：从KV Cache到PD分离的Serving全景解析" -- "PagedAttention与Cache管理":
       a sequence's logical blocks map to physical blocks taken on demand, so at most
       one block per sequence is partly empty; physical blocks may be shared between
       sequences, and a shared block is copied before one of its users changes it
       (copy-on-write, beam search).
  [P3] "ai-infra-7" -- "优化一：Prefix Cache": a full block is identified by its chained
       hash, so a new request whose leading blocks hash the same reuses them.
  [P2] "GPU推理深度拆解：KV Cache视角" -- "缓存命中与复用": hits are whole blocks and
       must form a prefix (the chain breaks at the first differing block); unused
       cached blocks are evicted least-recently-used first; a block in use is never
       evicted.

The pages fix the properties but not the tie-breaks.  Readings taken (the native
manager follows the same ones, so the two can be compared call by call):
  - a fresh block is the smallest free id; only when no block is free is the least
    recently released cached block evicted;
  - a released sequence gives its blocks back last block first, so a prefix's tail
    is older in the LRU order than its head and is evicted first (keeps the
    remaining cached blocks a usable prefix);
  - writing into a block that is shared or registered under a hash moves the writer
    to a fresh block after a copy; a private unregistered block is written in place;
  - a hash maps to at most one block, the first one registered under it;
  - a call that cannot get all the blocks it needs changes nothing.

Parity status: pinned by the properties above in tests/test_block_manager.py
(hits = longest registered prefix, refcount conservation, in-use blocks never
reassigned, LRU order on hand-worked sequences, waste < one block per sequence,
copy-on-write isolation).
"""
from __future__ import annotations

import numpy as np

NO_BLOCKS = "no_blocks"
INVALID = "invalid"


class BlockManagerModel:
    """States: free (refcount 0, no hash), used (refcount >= 1), cached (refcount 0,
    still registered under a hash, kept in LRU order)."""

    def __init__(self, num_blocks: int, block_size: int):
        self.num_blocks = num_blocks
        self.block_size = block_size
        self.refcount = [0] * num_blocks
        self.hash_of = {}          # block -> registered hash
        self.block_of = {}         # registered hash -> block
        self.free = list(range(num_blocks))
        self.lru = []              # cached blocks, oldest release first
        self.tables = {}           # seq id -> list of block ids
        self.tokens = {}           # seq id -> token count

    # -- helpers -------------------------------------------------------------------
    def available(self) -> int:
        return len(self.free) + len(self.lru)

    def _blocks_for(self, n_tokens: int) -> int:
        return -(-n_tokens // self.block_size)

    def _fresh(self) -> int:
        if self.free:
            b = min(self.free)
            self.free.remove(b)
        else:
            b = self.lru.pop(0)              # evict the least recently released
            h = self.hash_of.pop(b)
            del self.block_of[h]
        self.refcount[b] = 1
        return b

    def _release(self, b: int) -> None:
        self.refcount[b] -= 1
        if self.refcount[b] == 0:
            if b in self.hash_of:
                self.lru.append(b)
            else:
                self.free.append(b)

    def _register(self, b: int, h: int) -> None:
        if b in self.hash_of or h in self.block_of:
            return
        self.hash_of[b] = h
        self.block_of[h] = b

    # -- operations (same meaning as the library's pkv_bm_* calls) -----------------
    def add_sequence(self, seq_id, n_tokens, hashes):
        hashes = [int(h) for h in hashes]
        if seq_id in self.tables or n_tokens < 0 or len(hashes) > n_tokens // self.block_size:
            return INVALID
        nb = self._blocks_for(n_tokens)
        hits = 0
        while hits < len(hashes) and hashes[hits] in self.block_of:
            hits += 1
        hit_blocks = [self.block_of[h] for h in hashes[:hits]]
        # hit blocks that sit in the LRU list are no longer available once taken
        cached_hits = sum(1 for b in hit_blocks if b in self.lru)
        if nb - hits > self.available() - cached_hits:
            return NO_BLOCKS
        table = []
        for b in hit_blocks:
            if b in self.lru:
                self.lru.remove(b)
            self.refcount[b] += 1
            table.append(b)
        for i in range(hits, nb):
            b = self._fresh()
            if i < len(hashes):
                self._register(b, hashes[i])
            table.append(b)
        self.tables[seq_id] = table
        self.tokens[seq_id] = n_tokens
        return list(table), hits

    def grow(self, seq_id, n_tokens):
        if seq_id not in self.tables or n_tokens < self.tokens[seq_id]:
            return INVALID
        need = self._blocks_for(n_tokens) - len(self.tables[seq_id])
        if need > self.available():
            return NO_BLOCKS
        last = -1
        for _ in range(need):
            last = self._fresh()
            self.tables[seq_id].append(last)
        self.tokens[seq_id] = n_tokens
        return last

    def commit_block_hash(self, seq_id, logical_block, h):
        if seq_id not in self.tables or logical_block < 0 or \
                (logical_block + 1) * self.block_size > self.tokens[seq_id]:
            return INVALID
        self._register(self.tables[seq_id][logical_block], int(h))
        return None

    def fork(self, parent, child):
        if parent not in self.tables or child in self.tables:
            return INVALID
        self.tables[child] = list(self.tables[parent])
        self.tokens[child] = self.tokens[parent]
        for b in self.tables[child]:
            self.refcount[b] += 1
        return None

    def prepare_write(self, seq_id, logical_block):
        if seq_id not in self.tables or not 0 <= logical_block < len(self.tables[seq_id]):
            return INVALID
        b = self.tables[seq_id][logical_block]
        if self.refcount[b] == 1 and b not in self.hash_of:
            return (-1, -1)
        if self.available() < 1:
            return NO_BLOCKS
        nb = self._fresh()
        self._release(b)
        self.tables[seq_id][logical_block] = nb
        return (b, nb)

    def free_sequence(self, seq_id):
        if seq_id not in self.tables:
            return INVALID
        for b in reversed(self.tables[seq_id]):
            self._release(b)
        del self.tables[seq_id]
        del self.tokens[seq_id]
        return None

    def block_table(self, seq_id):
        return list(self.tables[seq_id]) if seq_id in self.tables else INVALID


def copy_blocks(k_cache, v_cache, mapping, k_scale=None, v_scale=None):
    """Apply the (source, destination) block copies in order, in place.

    k_cache, v_cache: numpy [NB, Hkv, BS, D] (any element type); k_scale, v_scale:
    [NB, Hkv] or None.  A pair with an id outside [0, NB) or with source ==
    destination is skipped.
    """
    nb = k_cache.shape[0]
    for src, dst in np.asarray(mapping, dtype=np.int64).reshape(-1, 2):
        if not (0 <= src < nb and 0 <= dst < nb) or src == dst:
            continue
        k_cache[dst] = k_cache[src]
        v_cache[dst] = v_cache[src]
        if k_scale is not None:
            k_scale[dst] = k_scale[src]
            v_scale[dst] = v_scale[src]
