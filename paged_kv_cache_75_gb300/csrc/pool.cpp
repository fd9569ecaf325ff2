// Host block pool: the block manager of the paged KV cache.
//
// "Как работает paged attention? (детально)" (aivaro.ru answers/837):
//   3.2 BlockManager -- a FIFO list of free physical ids, allocation takes
//       the head and sets the reference count to 1, an empty list is an
//       out-of-memory error, freeing lowers the count and returns the block
//       to the list at 0;
//   3.3 copy-on-write -- sequences that share blocks (parallel sampling, beam
//       search) copy a shared block before writing into it;
//   4.1 allocation -- logical block = pos / block_size, a new physical block
//       when the logical one is not mapped yet, the token goes to offset
//       pos % block_size;
//   4.2 deallocation.
// vLLM paper summary (easyvpn24.com/25506.html) §2-4: per-request mapping of
//   logical to physical blocks, filled left to right; a new block when the
//   last one is full; sharing between samples of one prompt.
//
// Choices where the pages leave room: an append that cannot get all of its
// blocks changes nothing (the page's sketch raises part-way through); the
// copy-on-write block is taken before the blocks for new tokens.
#include <cstdint>
#include <deque>
#include <new>
#include <unordered_map>
#include <vector>

#include "pa_kv.h"

namespace {

struct Sequence {
    std::vector<int32_t> blocks;  // logical index -> physical id
    int64_t length = 0;           // tokens held
};

struct Pool {
    int64_t num_blocks = 0;
    int32_t block_size = 0;
    std::deque<int32_t> free_list;
    std::vector<int32_t> ref;
    std::unordered_map<int64_t, Sequence> seqs;

    int32_t take() {
        int32_t b = free_list.front();
        free_list.pop_front();
        ref[b] = 1;
        return b;
    }
};

Pool* as_pool(void* p) { return static_cast<Pool*>(p); }

}  // namespace

extern "C" {

pa_status pa_pool_create(int64_t num_blocks, int32_t block_size, const int32_t* free_order,
                         void** pool_out) {
    if (pool_out == nullptr || num_blocks <= 0 || num_blocks > INT32_MAX || block_size <= 0)
        return PA_ERR_INVALID_ARG;
    Pool* p = new (std::nothrow) Pool();
    if (p == nullptr) return PA_ERR_OOM;
    p->num_blocks = num_blocks;
    p->block_size = block_size;
    p->ref.assign(static_cast<size_t>(num_blocks), 0);
    if (free_order != nullptr) {
        std::vector<char> seen(static_cast<size_t>(num_blocks), 0);
        for (int64_t i = 0; i < num_blocks; ++i) {
            int32_t b = free_order[i];
            if (b < 0 || b >= num_blocks || seen[b]) {
                delete p;
                return PA_ERR_INVALID_ARG;  // not a permutation
            }
            seen[b] = 1;
            p->free_list.push_back(b);
        }
    } else {
        for (int64_t i = 0; i < num_blocks; ++i) p->free_list.push_back(static_cast<int32_t>(i));
    }
    *pool_out = p;
    return PA_OK;
}

void pa_pool_destroy(void* pool) { delete as_pool(pool); }

pa_status pa_pool_add_seq(void* pool, int64_t seq_id) {
    Pool* p = as_pool(pool);
    if (p == nullptr || p->seqs.count(seq_id)) return PA_ERR_INVALID_ARG;
    p->seqs.emplace(seq_id, Sequence());
    return PA_OK;
}

pa_status pa_pool_append(void* pool, int64_t seq_id, int32_t n_tokens, int64_t* slots_out,
                         int32_t* cow_pairs_out, int32_t* n_cow_out) {
    Pool* p = as_pool(pool);
    if (p == nullptr || n_tokens < 0 || (n_tokens > 0 && slots_out == nullptr))
        return PA_ERR_INVALID_ARG;
    auto it = p->seqs.find(seq_id);
    if (it == p->seqs.end()) return PA_ERR_INVALID_ARG;
    Sequence& s = it->second;
    const int64_t bs = p->block_size;
    if (n_cow_out) *n_cow_out = 0;
    if (n_tokens == 0) return PA_OK;

    // blocks needed: new logical blocks, plus a private copy of a shared,
    // partially filled last block that the first new token writes into
    const int64_t blocks_after = (s.length + n_tokens + bs - 1) / bs;
    const int64_t new_blocks = blocks_after - static_cast<int64_t>(s.blocks.size());
    const bool cow = (s.length % bs) != 0 && p->ref[s.blocks.back()] > 1;
    if (new_blocks + (cow ? 1 : 0) > static_cast<int64_t>(p->free_list.size())) return PA_ERR_OOM;
    if (cow && (cow_pairs_out == nullptr || n_cow_out == nullptr)) return PA_ERR_INVALID_ARG;

    if (cow) {
        int32_t old_b = s.blocks.back();
        int32_t new_b = p->take();
        p->ref[old_b] -= 1;
        s.blocks.back() = new_b;
        cow_pairs_out[0] = old_b;
        cow_pairs_out[1] = new_b;
        *n_cow_out = 1;
    }
    for (int32_t i = 0; i < n_tokens; ++i) {
        const int64_t pos = s.length;
        const int64_t logical = pos / bs;
        if (logical == static_cast<int64_t>(s.blocks.size())) s.blocks.push_back(p->take());
        slots_out[i] = static_cast<int64_t>(s.blocks[logical]) * bs + pos % bs;
        s.length = pos + 1;
    }
    return PA_OK;
}

pa_status pa_pool_fork(void* pool, int64_t parent, int64_t child) {
    Pool* p = as_pool(pool);
    if (p == nullptr || p->seqs.count(child)) return PA_ERR_INVALID_ARG;
    auto it = p->seqs.find(parent);
    if (it == p->seqs.end()) return PA_ERR_INVALID_ARG;
    Sequence copy = it->second;
    for (int32_t b : copy.blocks) p->ref[b] += 1;
    p->seqs.emplace(child, std::move(copy));
    return PA_OK;
}

pa_status pa_pool_free_seq(void* pool, int64_t seq_id) {
    Pool* p = as_pool(pool);
    if (p == nullptr) return PA_ERR_INVALID_ARG;
    auto it = p->seqs.find(seq_id);
    if (it == p->seqs.end()) return PA_ERR_INVALID_ARG;
    for (int32_t b : it->second.blocks) {
        p->ref[b] -= 1;
        if (p->ref[b] == 0) p->free_list.push_back(b);
    }
    p->seqs.erase(it);
    return PA_OK;
}

pa_status pa_pool_block_table(void* pool, const int64_t* seq_ids, int32_t n, int32_t max_blocks,
                              int32_t* table_out, int32_t* lens_out) {
    Pool* p = as_pool(pool);
    if (p == nullptr || n < 0 || max_blocks < 0 || (n > 0 && (seq_ids == nullptr || table_out == nullptr)))
        return PA_ERR_INVALID_ARG;
    for (int32_t r = 0; r < n; ++r) {
        auto it = p->seqs.find(seq_ids[r]);
        if (it == p->seqs.end()) return PA_ERR_INVALID_ARG;
        const Sequence& s = it->second;
        if (static_cast<int64_t>(s.blocks.size()) > max_blocks) return PA_ERR_INVALID_ARG;
        int32_t* row = table_out + static_cast<int64_t>(r) * max_blocks;
        for (int32_t j = 0; j < max_blocks; ++j)
            row[j] = j < static_cast<int32_t>(s.blocks.size()) ? s.blocks[j] : -1;
        if (lens_out) lens_out[r] = static_cast<int32_t>(s.length);
    }
    return PA_OK;
}

int64_t pa_pool_num_free(void* pool) {
    Pool* p = as_pool(pool);
    return p ? static_cast<int64_t>(p->free_list.size()) : -1;
}

int32_t pa_pool_ref_count(void* pool, int64_t block) {
    Pool* p = as_pool(pool);
    if (p == nullptr || block < 0 || block >= p->num_blocks) return -1;
    return p->ref[block];
}

pa_status pa_slot_mapping(const int32_t* block_table, int32_t num_seqs, int32_t max_blocks,
                          int32_t block_size, const int32_t* seq_idx, const int64_t* pos, int64_t n,
                          int64_t* slots_out) {
    if (n < 0 || num_seqs < 0 || max_blocks < 0 || block_size <= 0 ||
        (n > 0 && (block_table == nullptr || seq_idx == nullptr || pos == nullptr || slots_out == nullptr)))
        return PA_ERR_INVALID_ARG;
    for (int64_t i = 0; i < n; ++i) {
        const int32_t b = seq_idx[i];
        if (b < 0 || b >= num_seqs || pos[i] < 0) return PA_ERR_INVALID_ARG;
        const int64_t logical = pos[i] / block_size;
        const int32_t phys = logical < max_blocks
                                 ? block_table[static_cast<int64_t>(b) * max_blocks + logical]
                                 : -1;
        slots_out[i] = phys < 0 ? -1 : static_cast<int64_t>(phys) * block_size + pos[i] % block_size;
    }
    return PA_OK;
}

int32_t pa_pool_seq_len(void* pool, int64_t seq_id) {
    Pool* p = as_pool(pool);
    if (p == nullptr) return -1;
    auto it = p->seqs.find(seq_id);
    return it == p->seqs.end() ? -1 : static_cast<int32_t>(it->second.length);
}

}  // extern "C"
