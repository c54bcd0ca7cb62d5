// pkv_block_manager.cpp -- host-side manager of the physical KV blocks.
//
// The block table of each sequence maps its logical blocks to physical blocks of
// BS tokens ("深入LLM推理：从KV Cache到PD分离的Serving全景解析", PagedAttention与Cache
// 管理: blocks are allocated on demand, waste stays within one block, physical
// blocks can be shared between requests -- prefix caching, and copy-on-write for
// beam search).  Full blocks are registered under their chained prefix hash
// ("ai-infra-7", 优化一：Prefix Cache), so a later sequence whose leading blocks
// have the same hashes reuses them ("GPU推理深度拆解：KV Cache视角", 缓存命中与复用:
// block-granular, token-exact hits; LRU eviction; blocks in use are never evicted).
//
// Policy (fixed so that a plain reference model reproduces every decision):
//   - a fresh block is the lowest-numbered block on the free list; when the free
//     list is empty, the least recently released cached block (refcount 0, still
//     registered under its hash) is evicted and reused;
//   - a new sequence reuses cached blocks for its leading full blocks while their
//     hashes are registered, stopping at the first miss (hits are prefixes);
//   - releasing a sequence walks its blocks from last to first, so the tail blocks of
//     a prefix become least recently released and are evicted first;
//   - allocation is all-or-nothing: a call that cannot get every block it needs
//     changes nothing and returns PKV_ERR_NO_BLOCKS.
#include <stdint.h>

#include <list>
#include <mutex>
#include <set>
#include <unordered_map>
#include <vector>

#include "../../include/pagedkv.h"

struct pkv_block_manager {
    int num_blocks = 0;
    int block_size = 0;
    std::mutex mu;
    std::vector<int> refcount;                 // per physical block
    std::vector<uint64_t> hash;                // registered hash (valid if hashed[b])
    std::vector<char> hashed;
    std::set<int> free_list;                   // refcount 0, not registered
    std::list<int> lru;                        // refcount 0, registered; front = oldest
    std::vector<std::list<int>::iterator> lru_pos;
    std::vector<char> in_lru;
    std::unordered_map<uint64_t, int> by_hash;  // registered hash -> block
    struct Seq {
        std::vector<int> blocks;
        int64_t tokens = 0;
    };
    std::unordered_map<int64_t, Seq> seqs;
};

namespace {

int lru_take(pkv_block_manager* m) {   // evict the least recently released cached block
    const int b = m->lru.front();
    m->lru.pop_front();
    m->in_lru[b] = 0;
    m->by_hash.erase(m->hash[b]);
    m->hashed[b] = 0;
    return b;
}

int available(const pkv_block_manager* m) {
    return (int)m->free_list.size() + (int)m->lru.size();
}

// A fresh block (refcount becomes 1); the caller has checked availability.
int fresh_block(pkv_block_manager* m) {
    int b;
    if (!m->free_list.empty()) {
        b = *m->free_list.begin();
        m->free_list.erase(m->free_list.begin());
    } else {
        b = lru_take(m);
    }
    m->refcount[b] = 1;
    return b;
}

void acquire_cached(pkv_block_manager* m, int b) {
    if (m->in_lru[b]) {
        m->lru.erase(m->lru_pos[b]);
        m->in_lru[b] = 0;
    }
    m->refcount[b] += 1;
}

void release(pkv_block_manager* m, int b) {
    if (--m->refcount[b] > 0) return;
    if (m->hashed[b]) {
        m->lru.push_back(b);
        m->lru_pos[b] = std::prev(m->lru.end());
        m->in_lru[b] = 1;
    } else {
        m->free_list.insert(b);
    }
}

void register_hash(pkv_block_manager* m, int b, uint64_t h) {
    if (m->hashed[b] || m->by_hash.count(h)) return;   // first registration of a hash wins
    m->hashed[b] = 1;
    m->hash[b] = h;
    m->by_hash[h] = b;
}

int64_t blocks_for(const pkv_block_manager* m, int64_t tokens) {
    return (tokens + m->block_size - 1) / m->block_size;
}

}  // namespace

extern "C" {

int pkv_bm_create(int num_blocks, int block_size, pkv_block_manager** out) {
    if (!out || num_blocks <= 0 || block_size <= 0) return PKV_ERR_INVALID_ARG;
    pkv_block_manager* m = new (std::nothrow) pkv_block_manager();
    if (!m) return PKV_ERR_NO_BLOCKS;
    m->num_blocks = num_blocks;
    m->block_size = block_size;
    m->refcount.assign(num_blocks, 0);
    m->hash.assign(num_blocks, 0);
    m->hashed.assign(num_blocks, 0);
    m->lru_pos.resize(num_blocks);
    m->in_lru.assign(num_blocks, 0);
    for (int b = 0; b < num_blocks; ++b) m->free_list.insert(b);
    *out = m;
    return PKV_OK;
}

void pkv_bm_destroy(pkv_block_manager* m) { delete m; }

int pkv_bm_num_available(pkv_block_manager* m) {
    if (!m) return PKV_ERR_INVALID_ARG;
    std::lock_guard<std::mutex> lock(m->mu);
    return available(m);
}

int pkv_bm_add_sequence(pkv_block_manager* m, int64_t seq_id, int64_t num_tokens,
                        const uint64_t* block_hashes, int num_hashes, int32_t* block_ids,
                        int* cached_blocks) {
    if (!m || num_tokens < 0 || num_hashes < 0 || (num_hashes > 0 && !block_hashes) ||
        (int64_t)num_hashes > num_tokens / m->block_size)
        return PKV_ERR_INVALID_ARG;
    std::lock_guard<std::mutex> lock(m->mu);
    if (m->seqs.count(seq_id)) return PKV_ERR_INVALID_ARG;
    const int64_t nb = blocks_for(m, num_tokens);
    if (nb > 0 && !block_ids) return PKV_ERR_INVALID_ARG;
    // leading hits: consecutive registered hashes
    int hits = 0;
    while (hits < num_hashes && m->by_hash.count(block_hashes[hits])) ++hits;
    // blocks needed beyond the hits; hit blocks sitting in the LRU list stop being
    // available once acquired
    int hit_in_lru = 0;
    for (int i = 0; i < hits; ++i) hit_in_lru += m->in_lru[m->by_hash[block_hashes[i]]] ? 1 : 0;
    if ((int64_t)(nb - hits) > (int64_t)available(m) - hit_in_lru) return PKV_ERR_NO_BLOCKS;
    pkv_block_manager::Seq s;
    s.tokens = num_tokens;
    for (int i = 0; i < hits; ++i) {
        const int b = m->by_hash[block_hashes[i]];
        acquire_cached(m, b);
        s.blocks.push_back(b);
    }
    for (int64_t i = hits; i < nb; ++i) {
        const int b = fresh_block(m);
        if (i < num_hashes) register_hash(m, b, block_hashes[i]);
        s.blocks.push_back(b);
    }
    for (int64_t i = 0; i < nb; ++i) block_ids[i] = s.blocks[i];
    if (cached_blocks) *cached_blocks = hits;
    m->seqs.emplace(seq_id, std::move(s));
    return PKV_OK;
}

int pkv_bm_grow(pkv_block_manager* m, int64_t seq_id, int64_t num_tokens, int32_t* new_block) {
    if (!m) return PKV_ERR_INVALID_ARG;
    std::lock_guard<std::mutex> lock(m->mu);
    auto it = m->seqs.find(seq_id);
    if (it == m->seqs.end() || num_tokens < it->second.tokens) return PKV_ERR_INVALID_ARG;
    const int64_t need = blocks_for(m, num_tokens) - (int64_t)it->second.blocks.size();
    if (need > available(m)) return PKV_ERR_NO_BLOCKS;
    int32_t last = -1;
    for (int64_t i = 0; i < need; ++i) {
        last = fresh_block(m);
        it->second.blocks.push_back(last);
    }
    it->second.tokens = num_tokens;
    if (new_block) *new_block = last;
    return PKV_OK;
}

int pkv_bm_commit_block_hash(pkv_block_manager* m, int64_t seq_id, int logical_block,
                             uint64_t hash) {
    if (!m) return PKV_ERR_INVALID_ARG;
    std::lock_guard<std::mutex> lock(m->mu);
    auto it = m->seqs.find(seq_id);
    if (it == m->seqs.end() || logical_block < 0 ||
        (int64_t)(logical_block + 1) * m->block_size > it->second.tokens)
        return PKV_ERR_INVALID_ARG;   // only a full block can be registered
    register_hash(m, it->second.blocks[logical_block], hash);
    return PKV_OK;
}

int pkv_bm_fork(pkv_block_manager* m, int64_t parent_id, int64_t child_id) {
    if (!m) return PKV_ERR_INVALID_ARG;
    std::lock_guard<std::mutex> lock(m->mu);
    auto it = m->seqs.find(parent_id);
    if (it == m->seqs.end() || m->seqs.count(child_id)) return PKV_ERR_INVALID_ARG;
    pkv_block_manager::Seq child = it->second;
    for (int b : child.blocks) m->refcount[b] += 1;
    m->seqs.emplace(child_id, std::move(child));
    return PKV_OK;
}

int pkv_bm_prepare_write(pkv_block_manager* m, int64_t seq_id, int logical_block,
                         int32_t* copy_src, int32_t* copy_dst) {
    if (!m || !copy_src || !copy_dst) return PKV_ERR_INVALID_ARG;
    std::lock_guard<std::mutex> lock(m->mu);
    auto it = m->seqs.find(seq_id);
    if (it == m->seqs.end() || logical_block < 0 ||
        logical_block >= (int)it->second.blocks.size())
        return PKV_ERR_INVALID_ARG;
    const int b = it->second.blocks[logical_block];
    *copy_src = -1;
    *copy_dst = -1;
    if (m->refcount[b] == 1 && !m->hashed[b]) return PKV_OK;   // private: write in place
    if (available(m) < 1) return PKV_ERR_NO_BLOCKS;
    const int nbk = fresh_block(m);
    release(m, b);
    it->second.blocks[logical_block] = nbk;
    *copy_src = b;
    *copy_dst = nbk;
    return PKV_OK;
}

int pkv_bm_free_sequence(pkv_block_manager* m, int64_t seq_id) {
    if (!m) return PKV_ERR_INVALID_ARG;
    std::lock_guard<std::mutex> lock(m->mu);
    auto it = m->seqs.find(seq_id);
    if (it == m->seqs.end()) return PKV_ERR_INVALID_ARG;
    const std::vector<int>& bl = it->second.blocks;
    for (auto b = bl.rbegin(); b != bl.rend(); ++b) release(m, *b);
    m->seqs.erase(it);
    return PKV_OK;
}

int pkv_bm_block_table(pkv_block_manager* m, int64_t seq_id, int32_t* block_ids, int capacity) {
    if (!m) return PKV_ERR_INVALID_ARG;
    std::lock_guard<std::mutex> lock(m->mu);
    auto it = m->seqs.find(seq_id);
    if (it == m->seqs.end()) return PKV_ERR_INVALID_ARG;
    const int n = (int)it->second.blocks.size();
    if (!block_ids) return n;   // size query
    if (n > capacity) return PKV_ERR_INVALID_ARG;
    for (int i = 0; i < n; ++i) block_ids[i] = it->second.blocks[i];
    return n;
}

int pkv_bm_refcount(pkv_block_manager* m, int block) {
    if (!m || block < 0 || block >= m->num_blocks) return PKV_ERR_INVALID_ARG;
    std::lock_guard<std::mutex> lock(m->mu);
    return m->refcount[block];
}

}  // extern "C"
