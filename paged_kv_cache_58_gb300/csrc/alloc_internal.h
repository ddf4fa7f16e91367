// Internal layout of the host block allocator, shared by allocator.cpp and the
// prefix-reuse indexes in prefix_cache.cpp.  Not part of the C ABI.
#pragma once

#include <cstdint>
#include <unordered_map>
#include <vector>

struct pkv_alloc {
    struct Seq {
        std::vector<int32_t> blocks;
        int64_t num_tokens = 0;
    };
    int64_t num_blocks = 0;
    int block_size = 16;
    std::vector<int32_t> free_list;  // stack: back() is handed out next
    std::vector<int32_t> refcount;
    std::unordered_map<int64_t, Seq> seqs;

    int32_t take() {
        const int32_t b = free_list.back();
        free_list.pop_back();
        refcount[b] = 1;
        return b;
    }
    void retain(int32_t b) { ++refcount[b]; }
    void release(int32_t b) {
        if (--refcount[b] == 0) free_list.push_back(b);
    }
};
