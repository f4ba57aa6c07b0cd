// Host-side parts of libpagedattn.so: the paged block allocator, KV
// accounting, slot mapping and the iteration-level scheduler simulators.
// No device access.
#include <stdint.h>
#include <stdlib.h>

#include <algorithm>
#include <deque>
#include <new>
#include <set>
#include <unordered_map>
#include <vector>

#include "../../include/pa.h"
#include "pa_host_internal.h"

// Reference-counted pool of fixed-size KV blocks ("KV cache & continuous
// batching", section "2. PagedAttention"; "LLM Serving - KV Cache, Batching,
// Speculative Decoding", section "KV memory, paging and prefix identity").
// The free set is ordered, so an allocation hands out the lowest free ids.
struct pa_allocator {
    int num_blocks;
    int block_size;
    std::vector<int32_t> refcnt;
    std::set<int32_t> free_ids;
    int attached = 0;       // prefix caches created on this allocator and not yet destroyed
    bool released = false;  // pa_allocator_destroy was called while caches were attached
    int64_t fail_in = 0;    // > 0: the fail_in-th next allocation fails (pa_allocator_fail_nth_alloc)
};

namespace pa {

void allocator_attach(pa_allocator* a) { ++a->attached; }

void allocator_detach(pa_allocator* a) {
    if (--a->attached == 0 && a->released) delete a;
}

}  // namespace pa

extern "C" {

pa_allocator* pa_allocator_create(int num_blocks, int block_size) {
    if (num_blocks < 0 || block_size <= 0) return nullptr;
    pa_allocator* a = new (std::nothrow) pa_allocator;
    if (!a) return nullptr;
    try {
        a->num_blocks = num_blocks;
        a->block_size = block_size;
        a->refcnt.assign((size_t)num_blocks, 0);
        for (int i = 0; i < num_blocks; ++i) a->free_ids.insert(a->free_ids.end(), i);
    } catch (...) {
        delete a;
        return nullptr;
    }
    return a;
}

void pa_allocator_destroy(pa_allocator* a) {
    if (!a) return;
    if (a->attached > 0) {
        a->released = true;   // freed by the last attached cache's destroy
        return;
    }
    delete a;
}

pa_status pa_block_alloc(pa_allocator* a, int n, int32_t* out_ids) {
    if (!a || n < 0 || (n > 0 && !out_ids)) return PA_ERR_INVALID;
    if (n > 0 && a->fail_in > 0 && --a->fail_in == 0) return PA_ERR_OOM;   // injected
    if ((size_t)n > a->free_ids.size()) return PA_ERR_OOM;
    for (int k = 0; k < n; ++k) {
        auto it = a->free_ids.begin();
        out_ids[k] = *it;
        a->refcnt[*it] = 1;
        a->free_ids.erase(it);
    }
    return PA_OK;
}

pa_status pa_block_free(pa_allocator* a, const int32_t* ids, int n) {
    if (!a || n < 0 || (n > 0 && !ids)) return PA_ERR_INVALID;
    std::unordered_map<int32_t, int> drops;
    for (int k = 0; k < n; ++k) {
        if (ids[k] < 0 || ids[k] >= a->num_blocks) return PA_ERR_INVALID;
        drops[ids[k]]++;
    }
    for (const auto& kv : drops)
        if (a->refcnt[kv.first] < kv.second) return PA_ERR_INVALID;
    for (const auto& kv : drops) {
        a->refcnt[kv.first] -= kv.second;
        if (a->refcnt[kv.first] == 0) a->free_ids.insert(kv.first);
    }
    return PA_OK;
}

pa_status pa_block_share(pa_allocator* a, const int32_t* ids, int n) {
    if (!a || n < 0 || (n > 0 && !ids)) return PA_ERR_INVALID;
    for (int k = 0; k < n; ++k)
        if (ids[k] < 0 || ids[k] >= a->num_blocks || a->refcnt[ids[k]] == 0) return PA_ERR_INVALID;
    for (int k = 0; k < n; ++k) a->refcnt[ids[k]]++;
    return PA_OK;
}

pa_status pa_allocator_fail_nth_alloc(pa_allocator* a, int64_t n) {
    if (!a) return PA_ERR_INVALID;
    a->fail_in = n > 0 ? n : 0;
    return PA_OK;
}

int pa_allocator_num_free(const pa_allocator* a) { return a ? (int)a->free_ids.size() : -1; }

int pa_allocator_num_blocks(const pa_allocator* a) { return a ? a->num_blocks : -1; }

int pa_allocator_block_size(const pa_allocator* a) { return a ? a->block_size : -1; }

int pa_allocator_refcount(const pa_allocator* a, int32_t id) {
    if (!a || id < 0 || id >= a->num_blocks) return -1;
    return a->refcnt[id];
}

int64_t pa_blocks_for_tokens(int64_t tokens, int block_size) {
    if (tokens <= 0 || block_size <= 0) return 0;
    return (tokens + block_size - 1) / block_size;
}

uint64_t pa_kv_bytes(int layers, int kv_heads, int head_dim, int dtype_bits, int64_t tokens,
                     int64_t batch) {
    if (layers < 0 || kv_heads < 0 || head_dim < 0 || dtype_bits < 0 || tokens < 0 || batch < 0)
        return 0;
    // K and V, every layer, every KV head, every cached position of every sequence
    const uint64_t elems = 2ull * (uint64_t)layers * (uint64_t)kv_heads * (uint64_t)head_dim *
                           (uint64_t)tokens * (uint64_t)batch;
    return elems * (uint64_t)dtype_bits / 8ull;
}

pa_status pa_slot_mapping(const int32_t* block_tables, int max_blocks_per_seq,
                          const int32_t* seq_ids, const int32_t* positions, int num_tokens,
                          int block_size, int64_t* slots) {
    if (num_tokens < 0 || block_size <= 0 || max_blocks_per_seq < 0) return PA_ERR_INVALID;
    if (num_tokens == 0) return PA_OK;
    if (!block_tables || !seq_ids || !positions || !slots) return PA_ERR_INVALID;
    for (int t = 0; t < num_tokens; ++t) {
        const int p = positions[t];
        if (p < 0 || seq_ids[t] < 0 || p / block_size >= max_blocks_per_seq) return PA_ERR_INVALID;
        const int32_t blk = block_tables[(int64_t)seq_ids[t] * max_blocks_per_seq + p / block_size];
        slots[t] = (int64_t)blk * block_size + p % block_size;
    }
    return PA_OK;
}

pa_status pa_step_slots(const int32_t* block_tables, int max_blocks_per_seq, const int32_t* seq_lens, int batch,
                        int block_size, int64_t* slots) {
    if (batch < 0 || block_size <= 0 || max_blocks_per_seq < 0) return PA_ERR_INVALID;
    if (batch == 0) return PA_OK;
    if (!block_tables || !seq_lens || !slots) return PA_ERR_INVALID;
    for (int b = 0; b < batch; ++b) {
        const int32_t len = seq_lens[b];
        if (len <= 0) {   // no token this step
            slots[b] = -1;
            continue;
        }
        const int p = len - 1;   // the new token is the sequence's last position
        if (p / block_size >= max_blocks_per_seq) return PA_ERR_INVALID;
        const int32_t blk = block_tables[(int64_t)b * max_blocks_per_seq + p / block_size];
        slots[b] = (int64_t)blk * block_size + p % block_size;
    }
    return PA_OK;
}

pa_status pa_share_plan(const int32_t* block_tables, int max_blocks_per_seq, const int32_t* seq_lens, int batch,
                        int block_size, int group_rows, int min_blocks, int32_t* chunk_of, int32_t* chunk_members,
                        int32_t* chunk_blocks, int max_chunks, int* n_chunks, int* max_chunk_blocks) {
    if (batch < 0 || block_size <= 0 || max_blocks_per_seq <= 0 || max_chunks < 0 || !n_chunks ||
        !max_chunk_blocks || group_rows < 0 || group_rows > PA_SHARE_MAX_ROWS)
        return PA_ERR_INVALID;
    *n_chunks = 0;
    *max_chunk_blocks = 0;
    if (batch == 0) return PA_OK;
    if (!block_tables || !seq_lens || !chunk_of || (max_chunks > 0 && (!chunk_members || !chunk_blocks)))
        return PA_ERR_INVALID;
    const int M = max_blocks_per_seq;
    auto row = [&](int b) { return block_tables + (int64_t)b * M; };
    // blocks of b that hold only positions before its newest token (the one
    // a decode step appends): they are complete and the step never writes them
    std::vector<int> cap((size_t)batch);
    for (int b = 0; b < batch; ++b) {
        chunk_of[b] = -1;
        const int64_t len = seq_lens[b];
        cap[b] = len >= 1 ? (int)std::min<int64_t>((len - 1) / block_size, M) : 0;
    }
    if (group_rows < 2) return PA_OK;   // one sequence per chunk shares nothing
    // groups: sequences whose first physical block is the same, in batch order
    std::vector<int> order;
    for (int b = 0; b < batch; ++b)
        if (cap[b] >= std::max(min_blocks, 1)) order.push_back(b);
    std::stable_sort(order.begin(), order.end(), [&](int x, int y) { return row(x)[0] < row(y)[0]; });
    int nc = 0, mx = 0;
    for (size_t i = 0; i < order.size();) {
        size_t e = i + 1;
        while (e < order.size() && row(order[e])[0] == row(order[i])[0]) ++e;
        if (e - i >= 2) {
            // the blocks every member holds at the same positions as the first
            const int first = order[i];
            int L = cap[first];
            for (size_t k = i + 1; k < e; ++k) {
                const int b = order[k];
                int c = 0;
                const int lim = std::min(L, cap[b]);
                while (c < lim && row(b)[c] == row(first)[c]) ++c;
                L = c;
            }
            if (L >= std::max(min_blocks, 1)) {
                for (size_t k = i; k < e && nc < max_chunks; k += group_rows, ++nc) {
                    chunk_blocks[nc] = L;
                    for (int r = 0; r < PA_SHARE_MAX_ROWS; ++r) {
                        const size_t m = k + r;
                        const bool in = r < group_rows && m < e;
                        chunk_members[(int64_t)nc * PA_SHARE_MAX_ROWS + r] = in ? order[m] : -1;
                        if (in) chunk_of[order[m]] = nc * PA_SHARE_MAX_ROWS + r;   // chunk and slot
                    }
                }
                mx = std::max(mx, L);
            }
        }
        i = e;
    }
    *n_chunks = nc;
    *max_chunk_blocks = mx;
    return PA_OK;
}

pa_status pa_sched_simulate(const int64_t* out_lens, int n, int slots, int mode, int64_t* iters) {
    if (n < 0 || slots <= 0 || (mode != 0 && mode != 1) || !iters || (n > 0 && !out_lens))
        return PA_ERR_INVALID;
    for (int i = 0; i < n; ++i)
        if (out_lens[i] <= 0) return PA_ERR_INVALID;
    int64_t total = 0;
    if (mode == 0) {
        for (int i = 0; i < n; i += slots) total += *std::max_element(out_lens + i, out_lens + std::min(n, i + slots));
        *iters = total;
        return PA_OK;
    }
    // Iteration-level: a min-heap of finishing times; a request admitted at
    // tick t with length L occupies its slot for ticks t .. t+L-1.
    std::multiset<int64_t> busy;  // finishing tick of each occupied slot
    int64_t now = 0;
    int next = 0;
    while (next < n) {
        while ((int)busy.size() < slots && next < n) busy.insert(now + out_lens[next++]);
        if (next < n) {  // jump to the next tick at which a slot frees
            now = *busy.begin();
            while (!busy.empty() && *busy.begin() <= now) busy.erase(busy.begin());
        }
    }
    for (int64_t f : busy) total = std::max(total, f);
    *iters = n == 0 ? 0 : total;
    return PA_OK;
}

pa_status pa_sched_continuous_kv(pa_allocator* a, const int64_t* prompt_lens,
                                 const int64_t* out_lens, int n, int max_num_seqs,
                                 int64_t stop_iter, int max_blocks_per_seq, int64_t* iters,
                                 int64_t* admitted_at, int64_t* finished_at, int32_t* tables,
                                 int32_t* lens) {
    if (!a || n < 0 || max_num_seqs <= 0 || max_blocks_per_seq < 0 || (n > 0 && (!prompt_lens || !out_lens)))
        return PA_ERR_INVALID;
    for (int r = 0; r < n; ++r) {
        if (prompt_lens[r] < 0 || out_lens[r] <= 0) return PA_ERR_INVALID;
        const int64_t need = pa_blocks_for_tokens(prompt_lens[r] + out_lens[r], a->block_size);
        if (need > a->num_blocks || (tables && need > max_blocks_per_seq)) return PA_ERR_INVALID;
    }
    struct Req {
        int id;
        int64_t generated;
        std::vector<int32_t> blocks;
    };
    std::vector<Req> active;
    std::deque<int> queue;
    for (int r = 0; r < n; ++r) queue.push_back(r);
    for (int r = 0; r < n; ++r) {
        if (admitted_at) admitted_at[r] = -1;
        if (finished_at) finished_at[r] = -1;
    }
    int64_t it = 0;
    while ((!queue.empty() || !active.empty()) && (stop_iter < 0 || it < stop_iter)) {
        // admission: in arrival order while a sequence slot and the reservation fit;
        // a reservation the pool refuses leaves the request queued, like a full pool
        bool refused = false;
        while (!queue.empty() && (int)active.size() < max_num_seqs) {
            const int r = queue.front();
            const int64_t need = pa_blocks_for_tokens(prompt_lens[r] + out_lens[r], a->block_size);
            if ((int64_t)a->free_ids.size() < need) break;
            Req q{r, 0, std::vector<int32_t>((size_t)need)};
            if (pa_block_alloc(a, (int)need, q.blocks.data()) != PA_OK) {
                refused = true;
                break;
            }
            active.push_back(std::move(q));
            queue.pop_front();
            if (admitted_at) admitted_at[r] = it;
        }
        // nothing can run: the pool refused the head (it holds nothing of this
        // call now), or the head can never fit
        if (active.empty()) return refused ? PA_ERR_OOM : PA_ERR_INVALID;
        // one decode iteration: every active request produces one token
        std::vector<Req> keep;
        keep.reserve(active.size());
        for (auto& q : active) {
            q.generated++;
            if (q.generated >= out_lens[q.id]) {
                pa_block_free(a, q.blocks.data(), (int)q.blocks.size());
                if (finished_at) finished_at[q.id] = it;
            } else {
                keep.push_back(std::move(q));
            }
        }
        active.swap(keep);
        ++it;
    }
    if (iters) *iters = it;
    if (tables || lens) {
        for (int r = 0; r < n; ++r) {
            if (lens) lens[r] = 0;
            if (tables)
                for (int j = 0; j < max_blocks_per_seq; ++j) tables[(int64_t)r * max_blocks_per_seq + j] = -1;
        }
        for (const auto& q : active) {
            if (lens) lens[q.id] = (int32_t)(prompt_lens[q.id] + q.generated);
            if (tables)
                for (size_t j = 0; j < q.blocks.size(); ++j)
                    tables[(int64_t)q.id * max_blocks_per_seq + (int64_t)j] = q.blocks[j];
        }
    }
    return PA_OK;
}

}  // extern "C"
