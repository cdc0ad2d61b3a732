// block_manager.cpp -- host-side allocator of the pool's blocks: free list,
// on-demand allocation, reference counts with copy-on-write, and automatic
// prefix caching over a chained block hash with least-recently-used eviction.
#include <cstdint>
#include <cstring>
#include <deque>
#include <list>
#include <mutex>
#include <new>
#include <unordered_map>
#include <vector>

#include "kv_block_manager.h"

namespace {

constexpr uint64_t kNoHash = 0;

// 64-bit mixing (splitmix64 finaliser) for the hash chain.
uint64_t mix64(uint64_t x)
{
    x += 0x9e3779b97f4a7c15ull;
    x = (x ^ (x >> 30)) * 0xbf58476d1ce4e5b9ull;
    x = (x ^ (x >> 27)) * 0x94d049bb133111ebull;
    return x ^ (x >> 31);
}

// Hash of one full block: chains the previous block's hash with the block's
// token ids.  Never returns kNoHash.
uint64_t block_hash(uint64_t prev, const int32_t* tokens, int n)
{
    uint64_t h = mix64(prev ^ 0x5bd1e9955bd1e995ull);
    for (int i = 0; i < n; ++i) h = mix64(h ^ static_cast<uint32_t>(tokens[i]));
    return h == kNoHash ? 1 : h;
}

uint64_t chain_start(uint64_t salt) { return mix64(salt ^ 0x243f6a8885a308d3ull); }

struct Block {
    int ref = 0;
    uint64_t hash = kNoHash;              // registered in the cache when != kNoHash
    std::vector<int32_t> tokens;          // ids of a registered block (exact-match check)
    bool evictable = false;               // in the LRU list
    std::list<int32_t>::iterator lru_it;
};

struct Seq {
    std::vector<int32_t> blocks;
    int64_t len = 0;
    uint64_t salt = 0;
    uint64_t chain = 0;                   // hash of the last full block (or the chain start)
    bool chain_ok = true;                 // every full block so far had its token ids
    std::vector<int32_t> partial;         // ids of the tokens in the last, partial block
};

}  // namespace

struct kv_block_manager {
    int num_blocks = 0;
    int block_size = 0;
    bool lifo = false;
    bool caching = false;
    std::deque<int32_t> free_list;
    std::list<int32_t> lru;               // cached blocks nobody holds; front = evict first
    std::unordered_map<uint64_t, int32_t> cache;
    std::vector<Block> blocks;
    std::unordered_map<int64_t, Seq> seqs;
    mutable std::mutex mu;

    int available() const { return static_cast<int>(free_list.size() + lru.size()); }

    // Takes a block: a free one, else the least recently used cached one.
    int32_t take()
    {
        int32_t b;
        if (!free_list.empty()) {
            if (lifo) {
                b = free_list.back();
                free_list.pop_back();
            } else {
                b = free_list.front();
                free_list.pop_front();
            }
        } else {
            b = lru.front();
            lru.pop_front();
            Block& blk = blocks[b];
            blk.evictable = false;
            cache.erase(blk.hash);
            blk.hash = kNoHash;
            blk.tokens.clear();
        }
        blocks[b].ref = 1;
        return b;
    }

    void hold(int32_t b)
    {
        Block& blk = blocks[b];
        if (blk.ref == 0 && blk.evictable) {
            lru.erase(blk.lru_it);
            blk.evictable = false;
        }
        ++blk.ref;
    }

    // Drops one reference.  A block nobody holds any more goes to the back of
    // the free list and returns false, unless it is registered in the cache: then
    // it is left for the caller to queue for eviction (returns true).
    bool release(int32_t b)
    {
        Block& blk = blocks[b];
        if (--blk.ref > 0) return false;
        if (caching && blk.hash != kNoHash) return true;
        blk.hash = kNoHash;
        blk.tokens.clear();
        free_list.push_back(b);
        return false;
    }

    void make_evictable(int32_t b)
    {
        lru.push_back(b);
        blocks[b].lru_it = std::prev(lru.end());
        blocks[b].evictable = true;
    }

    // A block of `s` just became full with the ids in s.partial: name it.
    void complete_block(Seq& s)
    {
        const int32_t b = s.blocks.back();
        if (!caching || !s.chain_ok || static_cast<int>(s.partial.size()) != block_size) {
            s.chain_ok = false;
            s.partial.clear();
            return;
        }
        const uint64_t h = block_hash(s.chain, s.partial.data(), block_size);
        s.chain = h;
        if (caching && blocks[b].hash == kNoHash && cache.find(h) == cache.end()) {
            blocks[b].hash = h;
            blocks[b].tokens = s.partial;
            cache.emplace(h, b);
        }
        s.partial.clear();
    }
};

extern "C" {

kv_status kv_bm_create(int num_blocks, int block_size, int flags, kv_block_manager** out)
{
    if (out == nullptr) return KV_ERR_INVALID_ARG;
    *out = nullptr;
    if (num_blocks <= 0 || block_size <= 0 || (flags & ~0x3) != 0) return KV_ERR_INVALID_ARG;
    kv_block_manager* bm = new (std::nothrow) kv_block_manager();
    if (bm == nullptr) return KV_ERR_OUT_OF_MEMORY;
    try {
        bm->num_blocks = num_blocks;
        bm->block_size = block_size;
        bm->lifo = (flags & KV_BM_LIFO) != 0;
        bm->caching = (flags & KV_BM_PREFIX_CACHING) != 0;
        bm->blocks.resize(num_blocks);
        for (int i = 0; i < num_blocks; ++i) bm->free_list.push_back(i);
    } catch (...) {
        delete bm;
        return KV_ERR_OUT_OF_MEMORY;
    }
    *out = bm;
    return KV_OK;
}

kv_status kv_bm_destroy(kv_block_manager* bm)
{
    delete bm;
    return KV_OK;
}

kv_status kv_bm_add_sequence(kv_block_manager* bm, int64_t seq, uint64_t salt)
{
    if (bm == nullptr) return KV_ERR_INVALID_ARG;
    std::lock_guard<std::mutex> lock(bm->mu);
    try {
        if (bm->seqs.count(seq)) return KV_ERR_INVALID_ARG;
        Seq s;
        s.salt = salt;
        s.chain = chain_start(salt);
        bm->seqs.emplace(seq, std::move(s));
    } catch (...) {
        return KV_ERR_OUT_OF_MEMORY;
    }
    return KV_OK;
}

kv_status kv_bm_fork(kv_block_manager* bm, int64_t parent, int64_t child)
{
    if (bm == nullptr) return KV_ERR_INVALID_ARG;
    std::lock_guard<std::mutex> lock(bm->mu);
    auto it = bm->seqs.find(parent);
    if (it == bm->seqs.end() || bm->seqs.count(child)) return KV_ERR_INVALID_ARG;
    try {
        Seq copy = it->second;
        for (int32_t b : copy.blocks) bm->hold(b);
        bm->seqs.emplace(child, std::move(copy));
    } catch (...) {
        return KV_ERR_OUT_OF_MEMORY;
    }
    return KV_OK;
}

kv_status kv_bm_append_slots(kv_block_manager* bm, int64_t seq, int n_tokens,
                             const int32_t* token_ids, kv_block_copy* copy, int* n_copies)
{
    if (bm == nullptr || n_tokens < 0 || n_copies == nullptr) return KV_ERR_INVALID_ARG;
    std::lock_guard<std::mutex> lock(bm->mu);
    *n_copies = 0;
    auto it = bm->seqs.find(seq);
    if (it == bm->seqs.end()) return KV_ERR_INVALID_ARG;
    Seq& s = it->second;
    if (n_tokens == 0) return KV_OK;
    const int bs = bm->block_size;
    const int64_t have = static_cast<int64_t>(s.blocks.size()) * bs;
    const int64_t need_tokens = s.len + n_tokens;
    const int64_t new_blocks = need_tokens > have ? (need_tokens - have + bs - 1) / bs : 0;
    const bool partial_last = s.len % bs != 0;
    const bool cow = partial_last && bm->blocks[s.blocks.back()].ref > 1;
    if (cow && copy == nullptr) return KV_ERR_INVALID_ARG;
    if (new_blocks + (cow ? 1 : 0) > bm->available()) return KV_ERR_OUT_OF_BLOCKS;
    try {
        s.blocks.reserve(s.blocks.size() + static_cast<size_t>(new_blocks));
        if (cow) {
            const int32_t old = s.blocks.back();
            const int32_t fresh = bm->take();
            bm->release(old);                               // count > 1: still held
            s.blocks.back() = fresh;
            copy->src = old;
            copy->dst = fresh;
            *n_copies = 1;
        }
        for (int i = 0; i < n_tokens; ++i) {
            if (s.len % bs == 0 && s.len / bs == static_cast<int64_t>(s.blocks.size()))
                s.blocks.push_back(bm->take());
            if (token_ids != nullptr) {
                s.partial.push_back(token_ids[i]);
            } else {
                s.chain_ok = false;
            }
            ++s.len;
            if (s.len % bs == 0) bm->complete_block(s);
        }
    } catch (...) {
        return KV_ERR_OUT_OF_MEMORY;
    }
    return KV_OK;
}

kv_status kv_bm_match_prefix(kv_block_manager* bm, int64_t seq, const int32_t* token_ids,
                             int n_tokens, int* cached_tokens)
{
    if (bm == nullptr || cached_tokens == nullptr || n_tokens < 0 ||
        (token_ids == nullptr && n_tokens > 0))
        return KV_ERR_INVALID_ARG;
    std::lock_guard<std::mutex> lock(bm->mu);
    *cached_tokens = 0;
    auto it = bm->seqs.find(seq);
    if (it == bm->seqs.end() || it->second.len != 0) return KV_ERR_INVALID_ARG;
    if (!bm->caching) return KV_OK;
    Seq& s = it->second;
    const int bs = bm->block_size;
    try {
        for (int start = 0; start + bs <= n_tokens; start += bs) {
            const uint64_t h = block_hash(s.chain, token_ids + start, bs);
            auto hit = bm->cache.find(h);
            if (hit == bm->cache.end()) break;
            const int32_t b = hit->second;
            if (std::memcmp(bm->blocks[b].tokens.data(), token_ids + start,
                            sizeof(int32_t) * bs) != 0)
                break;                                      // same hash, other tokens
            bm->hold(b);
            s.blocks.push_back(b);
            s.len += bs;
            s.chain = h;
            *cached_tokens += bs;
        }
    } catch (...) {
        return KV_ERR_OUT_OF_MEMORY;
    }
    return KV_OK;
}

kv_status kv_bm_free_sequence(kv_block_manager* bm, int64_t seq)
{
    if (bm == nullptr) return KV_ERR_INVALID_ARG;
    std::lock_guard<std::mutex> lock(bm->mu);
    auto it = bm->seqs.find(seq);
    if (it == bm->seqs.end()) return KV_ERR_INVALID_ARG;
    // Unregistered blocks return to the free list in table order; cached ones join
    // the eviction queue tail first, so a sequence's last blocks (the least likely
    // to be shared) are evicted before its first ones.
    std::vector<int32_t> cached;
    try {
        cached.reserve(it->second.blocks.size());
        for (int32_t b : it->second.blocks)
            if (bm->release(b)) cached.push_back(b);
        for (auto b = cached.rbegin(); b != cached.rend(); ++b) bm->make_evictable(*b);
    } catch (...) {
        return KV_ERR_OUT_OF_MEMORY;
    }
    bm->seqs.erase(it);
    return KV_OK;
}

kv_status kv_bm_num_free_blocks(const kv_block_manager* bm, int* n_free, int* n_cached_evictable)
{
    if (bm == nullptr) return KV_ERR_INVALID_ARG;
    std::lock_guard<std::mutex> lock(bm->mu);
    if (n_free) *n_free = static_cast<int>(bm->free_list.size());
    if (n_cached_evictable) *n_cached_evictable = static_cast<int>(bm->lru.size());
    return KV_OK;
}

kv_status kv_bm_sequence_info(const kv_block_manager* bm, int64_t seq, int* n_tokens,
                              int* n_blocks)
{
    if (bm == nullptr) return KV_ERR_INVALID_ARG;
    std::lock_guard<std::mutex> lock(bm->mu);
    auto it = bm->seqs.find(seq);
    if (it == bm->seqs.end()) return KV_ERR_INVALID_ARG;
    if (n_tokens) *n_tokens = static_cast<int>(it->second.len);
    if (n_blocks) *n_blocks = static_cast<int>(it->second.blocks.size());
    return KV_OK;
}

kv_status kv_bm_block_refcount(const kv_block_manager* bm, int32_t block, int* refcount)
{
    if (bm == nullptr || refcount == nullptr || block < 0 || block >= bm->num_blocks)
        return KV_ERR_INVALID_ARG;
    std::lock_guard<std::mutex> lock(bm->mu);
    *refcount = bm->blocks[block].ref;
    return KV_OK;
}

kv_status kv_bm_build_tables(const kv_block_manager* bm, const int64_t* seqs, int batch,
                             int max_blocks, int32_t* block_tables, int32_t* context_lens)
{
    if (bm == nullptr || batch < 0 || max_blocks <= 0 || (batch > 0 && seqs == nullptr) ||
        (batch > 0 && (block_tables == nullptr || context_lens == nullptr)))
        return KV_ERR_INVALID_ARG;
    std::lock_guard<std::mutex> lock(bm->mu);
    for (int i = 0; i < batch; ++i) {
        auto it = bm->seqs.find(seqs[i]);
        if (it == bm->seqs.end() || static_cast<int>(it->second.blocks.size()) > max_blocks)
            return KV_ERR_INVALID_ARG;
    }
    for (int i = 0; i < batch; ++i) {
        const Seq& s = bm->seqs.find(seqs[i])->second;
        int32_t* row = block_tables + static_cast<size_t>(i) * max_blocks;
        const int n = static_cast<int>(s.blocks.size());
        for (int j = 0; j < max_blocks; ++j) row[j] = j < n ? s.blocks[j] : -1;
        context_lens[i] = static_cast<int32_t>(s.len);
    }
    return KV_OK;
}

}  // extern "C"
