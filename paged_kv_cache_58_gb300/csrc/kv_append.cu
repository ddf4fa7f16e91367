// kv_append scatter and copy-on-write block copy.
//
// kv_append writes each new token's K/V rows into the next slot of its sequence's
// current block (Triptych "Paged Attention for Efficient Memory Management", body:
// "writes append within the current block"); the slot was chosen on the host by
// the block allocator.  copy_blocks duplicates whole physical blocks when a shared
// block is about to diverge (same page: copy-on-write after a fork).
//
// Both are pure data movement bound by HBM: one thread moves one 16-byte chunk,
// consecutive threads cover consecutive chunks of a row (a pool row of one
// (block, head, slot) is head_dim contiguous elements), so loads and stores are
// 128-bit and fully coalesced within a row.
#include <cuda_runtime.h>

#include <cstdlib>

#include "common.cuh"
#include "kernels.h"

namespace pkv {

namespace {

__global__ void __launch_bounds__(256)
kv_append_kernel(uint8_t* __restrict__ k_pool, uint8_t* __restrict__ v_pool,
                 const int64_t* __restrict__ slots, const uint8_t* __restrict__ k,
                 const uint8_t* __restrict__ v, int64_t num_chunks, int chunks_per_row,
                 int num_kv_heads, int row_bytes, int block_size, int64_t num_slots,
                 int* status) {
    griddep_wait();
    griddep_launch_dependents();
    const int64_t idx = static_cast<int64_t>(blockIdx.x) * blockDim.x + threadIdx.x;
    if (idx >= num_chunks) return;
    const int chunk = static_cast<int>(idx % chunks_per_row);
    const int64_t row = idx / chunks_per_row;            // (token, head)
    const int head = static_cast<int>(row % num_kv_heads);
    const int64_t tok = row / num_kv_heads;
    const int64_t slot = __ldg(slots + tok);
    if (slot < 0) return;                                  // padding row
    if (slot >= num_slots) {
        raise_status(status, PKV_ERR_OOB);
        return;
    }
    const int64_t blk = slot / block_size;
    const int64_t off = slot - blk * block_size;
    const int64_t dst = ((blk * num_kv_heads + head) * block_size + off) * row_bytes + chunk * 16;
    const int64_t src = row * row_bytes + chunk * 16;
    const uint4 kv = __ldg(reinterpret_cast<const uint4*>(k + src));
    const uint4 vv = __ldg(reinterpret_cast<const uint4*>(v + src));
    *reinterpret_cast<uint4*>(k_pool + dst) = kv;
    *reinterpret_cast<uint4*>(v_pool + dst) = vv;
}

// The same scatter with the index arithmetic cut down: chunks per row (8, 16 or 32 for
// the supported head dims and dtypes) is a compile-time constant, the block size a power
// of two, and the chunk index fits 32 bits (the launcher checks), so the decomposition
// is shifts, masks and one 32-bit division instead of five 64-bit divisions.  At about
// 10 us for 8192 rows the general kernel's integer divisions were a visible share.
template <int CPR>
__global__ void __launch_bounds__(256)
kv_append_pow2_kernel(uint8_t* __restrict__ k_pool, uint8_t* __restrict__ v_pool,
                      const int64_t* __restrict__ slots, const uint8_t* __restrict__ k,
                      const uint8_t* __restrict__ v, uint32_t num_chunks, uint32_t num_kv_heads,
                      int block_shift, int64_t num_slots, int* status) {
    griddep_wait();
    griddep_launch_dependents();
    const uint32_t idx = blockIdx.x * 256u + threadIdx.x;
    if (idx >= num_chunks) return;
    const uint32_t chunk = idx % CPR;
    const uint32_t row = idx / CPR;                 // (token, head)
    const uint32_t tok = row / num_kv_heads;
    const uint32_t head = row - tok * num_kv_heads;
    // The row's data do not depend on its slot: their loads go out beside the slot's, so
    // a thread waits for one memory round trip before its stores, not two.
    const int64_t src = (static_cast<int64_t>(row) * CPR + chunk) * 16;
    const uint4 kv = __ldg(reinterpret_cast<const uint4*>(k + src));
    const uint4 vv = __ldg(reinterpret_cast<const uint4*>(v + src));
    const int64_t slot = __ldg(slots + tok);
    if (slot < 0) return;                           // padding row
    if (slot >= num_slots) {
        raise_status(status, PKV_ERR_OOB);
        return;
    }
    const int64_t blk = slot >> block_shift;
    const int64_t off = slot & ((int64_t{1} << block_shift) - 1);
    const int64_t dst =
        ((((blk * num_kv_heads + head) << block_shift) + off) * CPR + chunk) * 16;
    *reinterpret_cast<uint4*>(k_pool + dst) = kv;
    *reinterpret_cast<uint4*>(v_pool + dst) = vv;
}

// grid (pairs, 2): y selects the K or V pool; one CTA copies one whole block.
__global__ void __launch_bounds__(256)
copy_blocks_kernel(uint8_t* __restrict__ k_pool, uint8_t* __restrict__ v_pool,
                   const int32_t* __restrict__ pairs, int64_t block_bytes, int64_t num_blocks,
                   int* status) {
    griddep_wait();
    griddep_launch_dependents();
    const int src = __ldg(pairs + 2 * blockIdx.x);
    const int dst = __ldg(pairs + 2 * blockIdx.x + 1);
    if (src < 0 || src >= num_blocks || dst < 0 || dst >= num_blocks) {
        if (threadIdx.x == 0) raise_status(status, PKV_ERR_OOB);
        return;
    }
    uint8_t* pool = blockIdx.y == 0 ? k_pool : v_pool;
    const uint4* s = reinterpret_cast<const uint4*>(pool + src * block_bytes);
    uint4* d = reinterpret_cast<uint4*>(pool + dst * block_bytes);
    const int64_t n = block_bytes / 16;
    for (int64_t i = threadIdx.x; i < n; i += blockDim.x) d[i] = s[i];
}

}  // namespace

cudaError_t launch_kv_append(void* k_pool, void* v_pool, const int64_t* slot_mapping,
                             const void* k, const void* v, int64_t num_tokens, int num_kv_heads,
                             int row_bytes, int block_size, int64_t num_blocks, int* status,
                             cudaStream_t stream) {
    const int chunks_per_row = row_bytes / 16;
    const int64_t num_chunks = num_tokens * num_kv_heads * chunks_per_row;
    if (num_chunks == 0) return cudaSuccess;
    const int64_t grid = (num_chunks + 255) / 256;
    const int block_shift = block_size == 16 ? 4 : block_size == 32 ? 5 : -1;
    // PKV_TEST_APPEND_GENERIC=1 sends every append to the general kernel (read at each
    // call; tests only: otherwise it runs for 2^31 chunks or more).
    const char* force = std::getenv("PKV_TEST_APPEND_GENERIC");
    const bool generic = force != nullptr && force[0] == '1';
    if (!generic && num_chunks < (int64_t{1} << 31) && block_shift > 0 &&
        (chunks_per_row == 8 || chunks_per_row == 16 || chunks_per_row == 32)) {
        auto kern = chunks_per_row == 8    ? kv_append_pow2_kernel<8>
                    : chunks_per_row == 16 ? kv_append_pow2_kernel<16>
                                           : kv_append_pow2_kernel<32>;
        return launch_pdl(kern, dim3(static_cast<unsigned>(grid)), dim3(256), 0, stream,
                          static_cast<uint8_t*>(k_pool), static_cast<uint8_t*>(v_pool),
                          slot_mapping, static_cast<const uint8_t*>(k),
                          static_cast<const uint8_t*>(v), static_cast<uint32_t>(num_chunks),
                          static_cast<uint32_t>(num_kv_heads), block_shift,
                          num_blocks * block_size, status);
    }
    return launch_pdl(kv_append_kernel, dim3(static_cast<unsigned>(grid)), dim3(256), 0, stream,
                      static_cast<uint8_t*>(k_pool), static_cast<uint8_t*>(v_pool), slot_mapping,
                      static_cast<const uint8_t*>(k), static_cast<const uint8_t*>(v), num_chunks,
                      chunks_per_row, num_kv_heads, row_bytes, block_size,
                      num_blocks * block_size, status);
}

cudaError_t launch_copy_blocks(void* k_pool, void* v_pool, const int32_t* pairs, int num_pairs,
                               int64_t block_bytes, int64_t num_blocks, int* status,
                               cudaStream_t stream) {
    if (num_pairs == 0) return cudaSuccess;
    return launch_pdl(copy_blocks_kernel, dim3(num_pairs, 2), dim3(256), 0, stream,
                      static_cast<uint8_t*>(k_pool), static_cast<uint8_t*>(v_pool), pairs,
                      block_bytes, num_blocks, status);
}

}  // namespace pkv
