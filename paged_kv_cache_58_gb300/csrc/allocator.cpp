// Host-side block allocator: on-demand blocks, refcounts, fork and copy-on-write.
//
// Follows the Triptych page ("Paged Attention for Efficient Memory Management",
// body and "Look closer"): a sequence holds a list of physical blocks; a new token
// goes to the next slot of the current block, or to a fresh block when the current
// one is full; a fork references the parent's blocks (refcount + 1) instead of
// copying them; a write into a block that other sequences still reference first
// copies that block (copy-on-write); blocks return to the free list when their
// count reaches zero.  The khotyn.com page ("PagedAttention") adds the bound this
// gives: at most one partially filled block per sequence.
#include <algorithm>
#include <cstdint>
#include <new>
#include <unordered_map>
#include <vector>

#include "../../include/pkv.h"

#include "alloc_internal.h"

namespace {

// splitmix64 step: the seeded shuffle of the initial free list.
uint64_t mix(uint64_t& state) {
    uint64_t z = (state += 0x9E3779B97F4A7C15ull);
    z = (z ^ (z >> 30)) * 0xBF58476D1CE4E5B9ull;
    z = (z ^ (z >> 27)) * 0x94D049BB133111EBull;
    return z ^ (z >> 31);
}

int64_t blocks_for(int64_t tokens, int bs) { return (tokens + bs - 1) / bs; }

}  // namespace

extern "C" {

pkv_alloc* pkv_alloc_create(int64_t num_blocks, int block_size, uint64_t seed) {
    if (num_blocks <= 0 || num_blocks > INT32_MAX || block_size <= 0) return nullptr;
    pkv_alloc* a = new (std::nothrow) pkv_alloc();
    if (!a) return nullptr;
    a->num_blocks = num_blocks;
    a->block_size = block_size;
    a->refcount.assign(static_cast<size_t>(num_blocks), 0);
    a->free_list.resize(static_cast<size_t>(num_blocks));
    // Hand out ascending ids: the stack holds them in descending order.
    for (int64_t i = 0; i < num_blocks; ++i)
        a->free_list[static_cast<size_t>(i)] = static_cast<int32_t>(num_blocks - 1 - i);
    if (seed != 0) {
        uint64_t st = seed;
        for (int64_t i = num_blocks - 1; i > 0; --i) {
            const int64_t j = static_cast<int64_t>(mix(st) % static_cast<uint64_t>(i + 1));
            std::swap(a->free_list[static_cast<size_t>(i)], a->free_list[static_cast<size_t>(j)]);
        }
    }
    return a;
}

void pkv_alloc_destroy(pkv_alloc* a) { delete a; }

pkv_status pkv_alloc_add_seq(pkv_alloc* a, int64_t seq_id, int64_t num_tokens) {
    if (!a || num_tokens < 0) return PKV_ERR_INVALID;
    if (a->seqs.count(seq_id)) return PKV_ERR_NOT_FOUND;
    const int64_t need = blocks_for(num_tokens, a->block_size);
    if (need > static_cast<int64_t>(a->free_list.size())) return PKV_ERR_NOMEM;
    pkv_alloc::Seq s;
    s.num_tokens = num_tokens;
    s.blocks.reserve(static_cast<size_t>(need));
    for (int64_t i = 0; i < need; ++i) s.blocks.push_back(a->take());
    a->seqs.emplace(seq_id, std::move(s));
    return PKV_OK;
}

pkv_status pkv_alloc_add_seq_shared(pkv_alloc* a, int64_t seq_id, const int32_t* shared_blocks,
                                    int num_shared, int64_t num_tokens) {
    if (!a || num_shared < 0 || num_tokens < 0 || (num_shared > 0 && !shared_blocks))
        return PKV_ERR_INVALID;
    if (a->seqs.count(seq_id)) return PKV_ERR_NOT_FOUND;
    const int64_t need = blocks_for(num_tokens, a->block_size);
    if (num_shared > need) return PKV_ERR_INVALID;
    for (int i = 0; i < num_shared; ++i) {
        const int32_t b = shared_blocks[i];
        if (b < 0 || b >= a->num_blocks || a->refcount[b] <= 0) return PKV_ERR_INVALID;
    }
    if (need - num_shared > static_cast<int64_t>(a->free_list.size())) return PKV_ERR_NOMEM;
    pkv_alloc::Seq s;
    s.num_tokens = num_tokens;
    s.blocks.reserve(static_cast<size_t>(need));
    for (int i = 0; i < num_shared; ++i) {
        ++a->refcount[shared_blocks[i]];
        s.blocks.push_back(shared_blocks[i]);
    }
    for (int64_t i = num_shared; i < need; ++i) s.blocks.push_back(a->take());
    a->seqs.emplace(seq_id, std::move(s));
    return PKV_OK;
}

pkv_status pkv_alloc_fork(pkv_alloc* a, int64_t parent, int64_t child) {
    if (!a) return PKV_ERR_INVALID;
    auto it = a->seqs.find(parent);
    if (it == a->seqs.end() || a->seqs.count(child)) return PKV_ERR_NOT_FOUND;
    pkv_alloc::Seq s = it->second;
    for (int32_t b : s.blocks) ++a->refcount[b];
    a->seqs.emplace(child, std::move(s));
    return PKV_OK;
}

pkv_status pkv_alloc_append(pkv_alloc* a, int64_t seq_id, int64_t n, int64_t* slots_out,
                            int32_t* cow_pairs_out, int* num_cow_out) {
    if (!a || n < 0 || (n > 0 && !slots_out) || !num_cow_out) return PKV_ERR_INVALID;
    auto it = a->seqs.find(seq_id);
    if (it == a->seqs.end()) return PKV_ERR_NOT_FOUND;
    pkv_alloc::Seq& s = it->second;
    const int bs = a->block_size;
    *num_cow_out = 0;
    if (n == 0) return PKV_OK;

    const bool partial_last = (s.num_tokens % bs) != 0;
    const bool cow = partial_last && a->refcount[s.blocks.back()] > 1;
    if (cow && !cow_pairs_out) return PKV_ERR_INVALID;
    const int64_t fresh = blocks_for(s.num_tokens + n, bs) - static_cast<int64_t>(s.blocks.size());
    if (fresh + (cow ? 1 : 0) > static_cast<int64_t>(a->free_list.size())) return PKV_ERR_NOMEM;

    if (cow) {
        const int32_t old = s.blocks.back();
        const int32_t mine = a->take();
        a->release(old);
        s.blocks.back() = mine;
        cow_pairs_out[0] = old;
        cow_pairs_out[1] = mine;
        *num_cow_out = 1;
    }
    for (int64_t i = 0; i < fresh; ++i) s.blocks.push_back(a->take());
    for (int64_t i = 0; i < n; ++i) {
        const int64_t pos = s.num_tokens + i;
        slots_out[i] = static_cast<int64_t>(s.blocks[static_cast<size_t>(pos / bs)]) * bs + pos % bs;
    }
    s.num_tokens += n;
    return PKV_OK;
}

pkv_status pkv_alloc_free_seq(pkv_alloc* a, int64_t seq_id) {
    if (!a) return PKV_ERR_INVALID;
    auto it = a->seqs.find(seq_id);
    if (it == a->seqs.end()) return PKV_ERR_NOT_FOUND;
    for (int32_t b : it->second.blocks) a->release(b);
    a->seqs.erase(it);
    return PKV_OK;
}

pkv_status pkv_alloc_block_table(const pkv_alloc* a, const int64_t* seq_ids, int num_seqs,
                                 int32_t* out, int max_blocks) {
    if (!a || num_seqs < 0 || max_blocks <= 0 || (num_seqs > 0 && (!seq_ids || !out)))
        return PKV_ERR_INVALID;
    for (int i = 0; i < num_seqs; ++i) {
        auto it = a->seqs.find(seq_ids[i]);
        if (it == a->seqs.end()) return PKV_ERR_NOT_FOUND;
        if (static_cast<int64_t>(it->second.blocks.size()) > max_blocks) return PKV_ERR_INVALID;
    }
    for (int i = 0; i < num_seqs; ++i) {
        const auto& b = a->seqs.find(seq_ids[i])->second.blocks;
        int32_t* row = out + static_cast<int64_t>(i) * max_blocks;
        std::fill(row, row + max_blocks, -1);
        std::copy(b.begin(), b.end(), row);
    }
    return PKV_OK;
}

int64_t pkv_alloc_num_free(const pkv_alloc* a) {
    return a ? static_cast<int64_t>(a->free_list.size()) : -1;
}

int pkv_alloc_refcount(const pkv_alloc* a, int64_t block) {
    if (!a || block < 0 || block >= a->num_blocks) return -1;
    return a->refcount[static_cast<size_t>(block)];
}

int64_t pkv_alloc_seq_len(const pkv_alloc* a, int64_t seq_id) {
    if (!a) return -1;
    auto it = a->seqs.find(seq_id);
    return it == a->seqs.end() ? -1 : it->second.num_tokens;
}

int64_t pkv_alloc_seq_num_blocks(const pkv_alloc* a, int64_t seq_id) {
    if (!a) return -1;
    auto it = a->seqs.find(seq_id);
    return it == a->seqs.end() ? -1 : static_cast<int64_t>(it->second.blocks.size());
}

}  // extern "C"
