// Prefix cache of full KV blocks and the copy-on-write helper.
//
// "KV cache & continuous batching", section "4. Prefix caching": the KV of a
// shared prefix is computed once and reused (vLLM hashes prefix blocks; a
// radix tree shares any common prefix); "LLM Serving - KV Cache, Batching,
// Speculative Decoding", section "KV memory, paging and prefix identity":
// reuse needs the exact token prefix.  Entry j of a chain stands for the
// tokens [0, (j+1)*bs) of a sequence: it is keyed by its parent entry and its
// own bs tokens, so two sequences share block j exactly when their first
// (j+1)*bs tokens agree.  Only full blocks are cached.  The cache holds one
// reference on every block it lists.
#include <stdint.h>

#include <algorithm>
#include <cstring>
#include <new>
#include <set>
#include <tuple>
#include <unordered_map>
#include <vector>

#include "../../include/pa.h"
#include "pa_host_internal.h"

namespace {

struct Entry {
    int parent;                 // entry id of the previous block of the chain, -1 for the first
    int32_t block;              // physical block
    int depth;                  // 0 for a chain's first block
    int64_t last_use;           // logical clock of the last match / insert that touched it
    std::vector<int32_t> toks;  // the block's bs tokens
    int children;               // live entries whose parent is this one
    bool live;
};

uint64_t mix(uint64_t h, uint64_t v) {
    h ^= v + 0x9e3779b97f4a7c15ull + (h << 6) + (h >> 2);
    return h;
}

}  // namespace

struct pa_prefix_cache {
    pa_allocator* alloc;
    int bs;
    int64_t clock;
    std::vector<Entry> entries;
    std::unordered_multimap<uint64_t, int> index;  // hash(parent, tokens) -> entry id

    uint64_t hash(int parent, const int32_t* toks) const {
        uint64_t h = mix(0x243f6a8885a308d3ull, (uint64_t)(int64_t)parent);
        for (int i = 0; i < bs; ++i) h = mix(h, (uint64_t)(uint32_t)toks[i]);
        return h;
    }

    int find(int parent, const int32_t* toks) const {
        auto range = index.equal_range(hash(parent, toks));
        for (auto it = range.first; it != range.second; ++it) {
            const Entry& e = entries[it->second];
            if (e.live && e.parent == parent && std::memcmp(e.toks.data(), toks, sizeof(int32_t) * bs) == 0)
                return it->second;
        }
        return -1;
    }
};

extern "C" {

pa_prefix_cache* pa_prefix_cache_create(pa_allocator* a) {
    if (!a) return nullptr;
    pa_prefix_cache* c = new (std::nothrow) pa_prefix_cache;
    if (!c) return nullptr;
    c->alloc = a;
    c->bs = pa_allocator_block_size(a);
    c->clock = 0;
    pa::allocator_attach(a);
    return c;
}

void pa_prefix_cache_destroy(pa_prefix_cache* c) {
    if (!c) return;
    for (const Entry& e : c->entries)
        if (e.live) pa_block_free(c->alloc, &e.block, 1);
    pa::allocator_detach(c->alloc);
    delete c;
}

int pa_prefix_cache_size(const pa_prefix_cache* c) {
    if (!c) return -1;
    int n = 0;
    for (const Entry& e : c->entries) n += e.live ? 1 : 0;
    return n;
}

pa_status pa_prefix_match(pa_prefix_cache* c, const int32_t* tokens, int64_t n_tokens, int32_t* out_blocks,
                          int max_out, int* n_blocks) {
    if (!c || n_tokens < 0 || max_out < 0 || !n_blocks || (n_tokens > 0 && !tokens) || (max_out > 0 && !out_blocks))
        return PA_ERR_INVALID;
    const int64_t full = n_tokens / c->bs;
    c->clock++;
    std::vector<int> path;
    int parent = -1;
    for (int64_t j = 0; j < full && (int64_t)path.size() < max_out; ++j) {
        const int id = c->find(parent, tokens + j * c->bs);
        if (id < 0) break;
        path.push_back(id);
        parent = id;
    }
    for (size_t j = 0; j < path.size(); ++j) out_blocks[j] = c->entries[path[j]].block;
    if (!path.empty() && pa_block_share(c->alloc, out_blocks, (int)path.size()) != PA_OK) return PA_ERR_INVALID;
    for (int id : path) c->entries[id].last_use = c->clock;
    *n_blocks = (int)path.size();
    return PA_OK;
}

pa_status pa_prefix_insert(pa_prefix_cache* c, const int32_t* tokens, int64_t n_tokens, const int32_t* blocks,
                           int n_blocks) {
    if (!c || n_tokens < 0 || n_blocks < 0 || (n_tokens > 0 && !tokens) || (n_blocks > 0 && !blocks))
        return PA_ERR_INVALID;
    const int64_t full = std::min<int64_t>(n_tokens / c->bs, n_blocks);
    for (int64_t j = 0; j < full; ++j)
        if (pa_allocator_refcount(c->alloc, blocks[j]) <= 0) return PA_ERR_INVALID;
    c->clock++;
    int parent = -1;
    for (int64_t j = 0; j < full; ++j) {
        const int32_t* toks = tokens + j * c->bs;
        int id = c->find(parent, toks);
        if (id < 0) {
            // a new entry: the cache takes its own reference on the block
            if (pa_block_share(c->alloc, &blocks[j], 1) != PA_OK) return PA_ERR_INVALID;
            Entry e;
            e.parent = parent;
            e.block = blocks[j];
            e.depth = (int)j;
            e.last_use = c->clock;
            e.toks.assign(toks, toks + c->bs);
            e.children = 0;
            e.live = true;
            if (parent >= 0) c->entries[parent].children++;
            id = (int)c->entries.size();
            c->entries.push_back(std::move(e));
            c->index.emplace(c->hash(parent, toks), id);
        } else {
            c->entries[id].last_use = c->clock;
        }
        parent = id;
    }
    return PA_OK;
}

pa_status pa_prefix_evict(pa_prefix_cache* c, int want, int* freed) {
    if (!c || want < 0 || !freed) return PA_ERR_INVALID;
    // candidates: chain ends that only the cache still references; the least
    // recently used first, then the deepest, then the lowest block id.  Freeing
    // an entry can make its parent a candidate.
    using Key = std::tuple<int64_t, int, int32_t, int>;  // (last_use, -depth, block, id)
    auto key = [&](int id) {
        const Entry& e = c->entries[id];
        return Key(e.last_use, -e.depth, e.block, id);
    };
    auto candidate = [&](int id) {
        const Entry& e = c->entries[id];
        return e.live && e.children == 0 && pa_allocator_refcount(c->alloc, e.block) == 1;
    };
    std::set<Key> cand;
    for (int id = 0; id < (int)c->entries.size(); ++id)
        if (candidate(id)) cand.insert(key(id));
    int n = 0;
    while (n < want && !cand.empty()) {
        const int id = std::get<3>(*cand.begin());
        cand.erase(cand.begin());
        Entry& e = c->entries[id];
        pa_block_free(c->alloc, &e.block, 1);
        e.live = false;
        ++n;
        if (e.parent >= 0) {
            c->entries[e.parent].children--;
            if (candidate(e.parent)) cand.insert(key(e.parent));
        }
    }
    *freed = n;
    return PA_OK;
}

pa_status pa_block_cow(pa_allocator* a, int32_t block, int32_t* out_block, int* needs_copy) {
    if (!a || !out_block || !needs_copy) return PA_ERR_INVALID;
    const int rc = pa_allocator_refcount(a, block);
    if (rc <= 0) return PA_ERR_INVALID;
    if (rc == 1) {  // the caller is the only user: write in place
        *out_block = block;
        *needs_copy = 0;
        return PA_OK;
    }
    int32_t fresh;
    const pa_status s = pa_block_alloc(a, 1, &fresh);
    if (s != PA_OK) return s;
    pa_block_free(a, &block, 1);  // the caller's reference moves to the private copy
    *out_block = fresh;
    *needs_copy = 1;
    return PA_OK;
}

namespace {

// n fresh blocks into out; when the pool is short, blocks only the prefix
// cache still holds are evicted first.  All or nothing.
pa_status alloc_evicting(pa_allocator* a, pa_prefix_cache* c, int n, int32_t* out) {
    if (n <= 0) return PA_OK;
    const int shortfall = n - pa_allocator_num_free(a);
    if (shortfall > 0 && c) {
        int freed = 0;
        pa_prefix_evict(c, shortfall, &freed);
    }
    return pa_block_alloc(a, n, out);
}

}  // namespace

pa_status pa_seq_admit(pa_allocator* a, pa_prefix_cache* c, const int32_t* tokens, int64_t n_tokens,
                       int32_t* blocks, int max_blocks, int* n_blocks, int64_t* first_new_pos) {
    if (!a || n_tokens < 0 || max_blocks < 0 || !n_blocks || !first_new_pos || (n_tokens > 0 && !tokens))
        return PA_ERR_INVALID;
    if (c && c->alloc != a) return PA_ERR_INVALID;
    const int bs = pa_allocator_block_size(a);
    const int64_t need = pa_blocks_for_tokens(n_tokens, bs);
    if (need > max_blocks || (need > 0 && !blocks)) return PA_ERR_INVALID;
    int shared = 0;
    if (c && need > 0) {
        const pa_status s = pa_prefix_match(c, tokens, n_tokens, blocks, (int)need, &shared);
        if (s != PA_OK) return s;
    }
    const pa_status s = alloc_evicting(a, c, (int)need - shared, blocks + shared);
    if (s != PA_OK) {
        if (shared) pa_block_free(a, blocks, shared);   // give the matched references back
        *n_blocks = 0;
        *first_new_pos = 0;
        return s;
    }
    *n_blocks = (int)need;
    *first_new_pos = (int64_t)shared * bs;
    return PA_OK;
}

pa_status pa_seq_append_slot(pa_allocator* a, pa_prefix_cache* c, int32_t* blocks, int* n_blocks, int max_blocks,
                             int64_t pos, int64_t* slot, int32_t* copy_src, int32_t* copy_dst) {
    if (!a || !n_blocks || !slot || !copy_src || !copy_dst || pos < 0 || *n_blocks < 0 ||
        (*n_blocks > 0 && !blocks))
        return PA_ERR_INVALID;
    if (c && c->alloc != a) return PA_ERR_INVALID;
    const int bs = pa_allocator_block_size(a);
    const int64_t j = pos / bs;
    if (j > *n_blocks || j >= max_blocks || !blocks) return PA_ERR_INVALID;
    *copy_src = *copy_dst = -1;
    if (j == *n_blocks) {   // the position opens a new block
        const pa_status s = alloc_evicting(a, c, 1, blocks + j);
        if (s != PA_OK) return s;
        *n_blocks += 1;
    } else {                // it lands in a block the sequence holds: write only a private one
        int32_t dst = -1;
        int needs_copy = 0;
        pa_status s = pa_block_cow(a, blocks[j], &dst, &needs_copy);
        if (s == PA_ERR_OOM && c) {
            int freed = 0;
            pa_prefix_evict(c, 1, &freed);
            if (freed > 0) s = pa_block_cow(a, blocks[j], &dst, &needs_copy);
        }
        if (s != PA_OK) return s;
        if (needs_copy) {
            *copy_src = blocks[j];
            *copy_dst = dst;
        }
        blocks[j] = dst;
    }
    *slot = (int64_t)blocks[j] * bs + pos % bs;
    return PA_OK;
}

}  // extern "C"
