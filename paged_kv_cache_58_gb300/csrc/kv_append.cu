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
