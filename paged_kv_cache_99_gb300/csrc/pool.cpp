// Host-side block pool: the allocator of physical cache blocks, with reference
// counts, a null block, copy-on-write and prefix caching.
//
// Problem ("Basics of LLM Inference and vLLM Internals", s.4 "PagedAttention and
// Block Management" and s.5 "Prefix Caching"; "The Memory Trick Behind Fast LLM
// Serving", "The block pool" and "Prefix caching is the second win"):
//  * a pool of fixed-size blocks; free blocks wait in a queue and are popped
//    when a request needs room; block 0 is reserved as the null block;
//  * a physical block may be shared by several block tables (reference count);
//  * a full block is identified by a chain of hashes (its parent block's hash
//    and its own tokens, plus extra keys), so only prefixes hit, in whole
//    blocks, and the block holding a prompt's last token is never a hit;
//  * finished requests return their blocks to the free queue keeping their
//    hashes; reuse takes blocks from the front, returned blocks go to the back
//    with a request's tail blocks ahead of its earlier ones.
// Reading taken where the pages are silent: a freed block that holds no cached
// content (a partial block) goes to the front, since evicting it loses nothing.
// Hits are verified against the stored tokens of the cached block, so a hash
// collision can never share the wrong content.
#include <cstdint>
#include <cstring>
#include <mutex>
#include <new>
#include <unordered_map>
#include <vector>

#include "pa.h"

namespace {

constexpr uint64_t kNoHash = 0;

uint64_t mix64(uint64_t x) {
    // 64-bit finaliser (xor-shift / multiply rounds)
    x ^= x >> 30;
    x *= 0xbf58476d1ce4e5b9ull;
    x ^= x >> 27;
    x *= 0x94d049bb133111ebull;
    x ^= x >> 31;
    return x;
}

struct BlockInfo {
    int ref = 0;
    int prev = -1, next = -1;         // free-queue links (valid while ref == 0 and in_queue)
    bool in_queue = false;
    uint64_t hash = kNoHash;          // registered full-block hash, kNoHash when none
    uint64_t parent = kNoHash;
    std::vector<int32_t> tokens;      // the block's tokens, for exact hit checks
};

}  // namespace

struct pa_block_pool {
    int num_blocks = 0;
    int block_size = 0;
    int head = -1, tail = -1, free_count = 0;
    std::vector<BlockInfo> b;
    std::unordered_map<uint64_t, int> cached;   // hash -> block
    std::mutex mu;

    void push_back(int i) {
        b[i].prev = tail;
        b[i].next = -1;
        if (tail >= 0) b[tail].next = i; else head = i;
        tail = i;
        b[i].in_queue = true;
        ++free_count;
    }
    void push_front(int i) {
        b[i].next = head;
        b[i].prev = -1;
        if (head >= 0) b[head].prev = i; else tail = i;
        head = i;
        b[i].in_queue = true;
        ++free_count;
    }
    void unlink(int i) {
        if (b[i].prev >= 0) b[b[i].prev].next = b[i].next; else head = b[i].next;
        if (b[i].next >= 0) b[b[i].next].prev = b[i].prev; else tail = b[i].prev;
        b[i].prev = b[i].next = -1;
        b[i].in_queue = false;
        --free_count;
    }
    void drop_hash(int i) {
        if (b[i].hash != kNoHash) {
            auto it = cached.find(b[i].hash);
            if (it != cached.end() && it->second == i) cached.erase(it);
            b[i].hash = kNoHash;
            b[i].parent = kNoHash;
            b[i].tokens.clear();
        }
    }
    // the head of the free queue, its cached content evicted, with one reference
    int take() {
        const int i = head;
        unlink(i);
        drop_hash(i);
        b[i].ref = 1;
        return i;
    }
    bool valid(int i) const { return i > 0 && i < num_blocks; }
    void release(const int32_t* ids, int n) {
        // blocks reaching zero: cached ones to the tail, the last given first, others to the front
        for (int k = n - 1; k >= 0; --k) {
            const int i = ids[k];
            if (--b[i].ref > 0) continue;
            if (b[i].hash != kNoHash) push_back(i); else push_front(i);
        }
    }
    uint64_t chain(uint64_t parent, const int32_t* tok) const {
        uint64_t h = mix64(parent ^ 0x9e3779b97f4a7c15ull);
        for (int j = 0; j < block_size; ++j) h = mix64(h ^ (static_cast<uint64_t>(static_cast<uint32_t>(tok[j])) + 0x632be59bd9b4e019ull * (j + 1)));
        return h == kNoHash ? 1 : h;
    }
    int lookup(uint64_t h, uint64_t parent, const int32_t* tok) const {
        auto it = cached.find(h);
        if (it == cached.end()) return -1;
        const BlockInfo& x = b[it->second];
        if (x.parent != parent || std::memcmp(x.tokens.data(), tok, sizeof(int32_t) * block_size) != 0) return -1;
        return it->second;
    }
};

extern "C" {

PA_API pa_block_pool* pa_pool_create(int num_blocks, int block_size) {
    if (num_blocks < 2 || block_size < 1) return nullptr;
    pa_block_pool* p = new (std::nothrow) pa_block_pool;
    if (!p) return nullptr;
    try {
        p->b.resize(static_cast<size_t>(num_blocks));
    } catch (...) {
        delete p;
        return nullptr;
    }
    p->num_blocks = num_blocks;
    p->block_size = block_size;
    for (int i = 1; i < num_blocks; ++i) p->push_back(i);   // block 0 stays out: the null block
    return p;
}

PA_API void pa_pool_destroy(pa_block_pool* pool) { delete pool; }

PA_API int pa_pool_num_free(pa_block_pool* pool) {
    if (!pool) return -1;
    std::lock_guard<std::mutex> lock(pool->mu);
    return pool->free_count;
}

PA_API int pa_pool_num_cached(pa_block_pool* pool) {
    if (!pool) return -1;
    std::lock_guard<std::mutex> lock(pool->mu);
    return static_cast<int>(pool->cached.size());
}

PA_API int pa_pool_ref_count(pa_block_pool* pool, int block) {
    if (!pool || block < 0 || block >= pool->num_blocks) return -1;
    std::lock_guard<std::mutex> lock(pool->mu);
    return pool->b[block].ref;
}

PA_API pa_status pa_pool_allocate(pa_block_pool* pool, int n, int32_t* blocks) {
    if (!pool || n < 0 || (n > 0 && !blocks)) return PA_ERR_INVALID_ARG;
    std::lock_guard<std::mutex> lock(pool->mu);
    if (n > pool->free_count) return PA_ERR_OUT_OF_RANGE;
    for (int k = 0; k < n; ++k) blocks[k] = pool->take();
    return PA_OK;
}

PA_API pa_status pa_pool_share(pa_block_pool* pool, const int32_t* blocks, int n) {
    if (!pool || n < 0 || (n > 0 && !blocks)) return PA_ERR_INVALID_ARG;
    std::lock_guard<std::mutex> lock(pool->mu);
    for (int k = 0; k < n; ++k)
        if (!pool->valid(blocks[k]) || pool->b[blocks[k]].ref <= 0) return PA_ERR_INVALID_ARG;
    for (int k = 0; k < n; ++k) ++pool->b[blocks[k]].ref;
    return PA_OK;
}

PA_API pa_status pa_pool_free(pa_block_pool* pool, const int32_t* blocks, int n) {
    if (!pool || n < 0 || (n > 0 && !blocks)) return PA_ERR_INVALID_ARG;
    std::lock_guard<std::mutex> lock(pool->mu);
    // every block must be in use, counting repeats within the call
    std::unordered_map<int, int> uses;
    for (int k = 0; k < n; ++k) {
        if (!pool->valid(blocks[k])) return PA_ERR_INVALID_ARG;
        if (++uses[blocks[k]] > pool->b[blocks[k]].ref) return PA_ERR_INVALID_ARG;
    }
    pool->release(blocks, n);
    return PA_OK;
}

PA_API pa_status pa_pool_allocate_prompt(pa_block_pool* pool, const int32_t* tokens, int num_tokens,
                                         uint64_t extra_key, int32_t* blocks, int* hit_tokens) {
    if (!pool || num_tokens < 0 || (num_tokens > 0 && (!tokens || !blocks))) return PA_ERR_INVALID_ARG;
    std::lock_guard<std::mutex> lock(pool->mu);
    const int bs = pool->block_size;
    const int nb = (num_tokens + bs - 1) / bs, nfull = num_tokens / bs;
    std::vector<uint64_t> h(static_cast<size_t>(nfull)), parent(static_cast<size_t>(nfull));
    uint64_t prev = mix64(extra_key ^ 0x5851f42d4c957f2dull);   // the chain's root carries the extra keys
    for (int i = 0; i < nfull; ++i) {
        parent[i] = prev;
        h[i] = pool->chain(prev, tokens + static_cast<size_t>(i) * bs);
        prev = h[i];
    }
    // leading cached full blocks, never the one holding the last token
    int hit = 0, hit_free = 0;
    std::vector<int> hb;
    while (hit < nfull && (hit + 1) * bs <= num_tokens - 1) {
        const int i = pool->lookup(h[hit], parent[hit], tokens + static_cast<size_t>(hit) * bs);
        if (i < 0) break;
        hb.push_back(i);
        hit_free += pool->b[i].ref == 0;
        ++hit;
    }
    if (nb - hit > pool->free_count - hit_free) return PA_ERR_OUT_OF_RANGE;
    for (int k = 0; k < hit; ++k) {
        const int i = hb[k];
        if (pool->b[i].ref == 0) pool->unlink(i);
        ++pool->b[i].ref;
        blocks[k] = i;
    }
    for (int k = hit; k < nb; ++k) {
        const int i = pool->take();
        if (k < nfull && pool->cached.find(h[k]) == pool->cached.end()) {
            BlockInfo& x = pool->b[i];
            x.hash = h[k];
            x.parent = parent[k];
            x.tokens.assign(tokens + static_cast<size_t>(k) * bs, tokens + static_cast<size_t>(k + 1) * bs);
            pool->cached[h[k]] = i;
        }
        blocks[k] = i;
    }
    if (hit_tokens) *hit_tokens = hit * bs;
    return PA_OK;
}

PA_API pa_status pa_pool_copy_on_write(pa_block_pool* pool, int32_t* blocks, int n, int32_t* src, int32_t* dst,
                                       int* num_copies) {
    if (!pool || n < 0 || (n > 0 && (!blocks || !src || !dst)) || !num_copies) return PA_ERR_INVALID_ARG;
    std::lock_guard<std::mutex> lock(pool->mu);
    int need = 0;
    for (int k = 0; k < n; ++k) {
        if (!pool->valid(blocks[k]) || pool->b[blocks[k]].ref <= 0) return PA_ERR_INVALID_ARG;
        need += pool->b[blocks[k]].ref > 1;
    }
    if (need > pool->free_count) return PA_ERR_OUT_OF_RANGE;
    int c = 0;
    for (int k = 0; k < n; ++k) {
        const int i = blocks[k];
        if (pool->b[i].ref <= 1) continue;
        const int j = pool->take();      // a private block for the writer
        --pool->b[i].ref;                // the shared one stays with its other owners
        src[c] = i;
        dst[c] = j;
        blocks[k] = j;
        ++c;
    }
    *num_copies = c;
    return PA_OK;
}

}  // extern "C"
