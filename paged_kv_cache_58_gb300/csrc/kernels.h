// Host-side launch interface between the C-ABI layer (pkv_api.cu) and the
// kernel translation units.  Internal to libpkv.
#pragma once

#include <cuda.h>
#include <cuda_runtime.h>
#include <stdint.h>

#include <utility>

namespace pkv {

// Launch `kern` with programmatic stream serialisation: its CTAs may be scheduled
// while the previous kernel on the stream drains; every libpkv kernel starts with
// griddep_wait(), so no input is read before the predecessor has completed.
// With pdl false the launch is ordinary: no CTA is placed before the predecessor ends.
template <typename... KArgs, typename... Args>
cudaError_t launch_maybe_pdl(bool pdl, void (*kern)(KArgs...), dim3 grid, dim3 block,
                             size_t smem, cudaStream_t stream, Args&&... args) {
    cudaLaunchConfig_t cfg = {};
    cfg.gridDim = grid;
    cfg.blockDim = block;
    cfg.dynamicSmemBytes = smem;
    cfg.stream = stream;
    cudaLaunchAttribute attr[1];
    attr[0].id = cudaLaunchAttributeProgrammaticStreamSerialization;
    attr[0].val.programmaticStreamSerializationAllowed = 1;
    cfg.attrs = attr;
    cfg.numAttrs = pdl ? 1 : 0;
    return cudaLaunchKernelEx(&cfg, kern, std::forward<Args>(args)...);
}
template <typename... KArgs, typename... Args>
cudaError_t launch_pdl(void (*kern)(KArgs...), dim3 grid, dim3 block, size_t smem,
                       cudaStream_t stream, Args&&... args) {
    return launch_maybe_pdl(true, kern, grid, block, smem, stream, std::forward<Args>(args)...);
}

// Upper bound on split-KV partitions of one sequence (combine kernel's smem).
constexpr int kMaxParts = 1024;

struct DecodeArgs {
    void* out;
    const void* q;
    const void* k_pool;
    const void* v_pool;
    const int32_t* block_tables;
    const int32_t* context_lens;
    float* o_part;   // [S][Hq][max_parts][D]
    float* m_part;   // [S][Hq][max_parts]  (log2 domain)
    float* l_part;   // [S][Hq][max_parts]
    int* status;
    int64_t num_blocks;
    int max_blocks_per_seq;   // block-table row stride, in pool blocks
    int num_seqs;
    int num_q_heads;
    int num_kv_heads;
    // The kernels walk a sequence in 16-token chunks: chunk c is rows
    // 16 (c & (2^chunk_shift - 1)) .. + 15 of the block in table entry c >> chunk_shift
    // (chunk_shift = log2(block_size / 16): 0 for 16-token blocks, 1 for 32).
    int chunk_shift;
    int partition_chunks;   // 16-token chunks per split-KV partition
    int max_parts;          // partitions of the decoded chunk range per sequence
    float scale_log2;       // softmax scale * log2(e)
    // Cascade decode: chunks [0, chunk_offset) of every sequence were handled by a
    // separate shared-prefix pass whose partial sits at partition 0; the split kernel
    // covers chunks [chunk_offset, nchunks) into partitions extra_parts.. and the combine
    // merges extra_parts + max_parts partials per row.
    int chunk_offset;
    int extra_parts;
    int defer_combine;   // nonzero: the launcher leaves the combine to the caller
    // nonzero: the split kernel is launched without programmatic dependent launch, so its
    // CTAs take no SM before the stream's previous kernel has ended (the cascade decode:
    // the prefix pass on the side stream is placed first).
    int no_pdl;
    // Test hook (both decode kernels): nonzero makes warp 0 of CTA (0, 0, 0) arm its first
    // stage for 16 bytes more than the stage's copies deliver, so that wait runs out of
    // time (PKV_ERR_TIMEOUT) while every copy still lands.  Zero in normal use.
    int test_stall;
    // Fused append (decode only): non-null k_new / v_new ([num_seqs][Hkv][D], pool
    // dtype) are the K / V of each sequence's newest token, position context_lens[s] - 1.
    // The CTA whose chunk holds that position stores them into the pool slot the block
    // table gives for it and uses them in place of the row it staged from the pool (which
    // the append has not reached yet).
    const void* k_new;
    const void* v_new;
};

#ifdef __CUDACC__
// Zeros of the G output rows (kv head kvh's query heads) of sequence `seq`, elem_bytes
// per element, stored 16 bytes at a time by the threads of the calling CTA; for a
// sequence the decode kernels reject (context length below 1), so that its rows hold no
// stale memory.
__device__ __forceinline__ void zero_invalid_rows(const DecodeArgs& a, int seq, int kvh, int G,
                                                  int D, int elem_bytes) {
    const size_t row0 = static_cast<size_t>(seq) * a.num_q_heads + static_cast<size_t>(kvh) * G;
    uint4* dst = reinterpret_cast<uint4*>(static_cast<char*>(a.out) + row0 * D * elem_bytes);
    const int n16 = G * D * elem_bytes / 16;
    for (int i = threadIdx.x; i < n16; i += blockDim.x) dst[i] = make_uint4(0, 0, 0, 0);
}
#endif

// CUDA-core decode (fp32 and bf16 pools): split kernel + combine.
cudaError_t launch_paged_decode(const DecodeArgs& a, int dtype, int head_dim, int group,
                                cudaStream_t stream);
// Tensor-core decode for bf16 pools (warp-level MMA): split kernel + combine.
cudaError_t launch_paged_decode_tc(const DecodeArgs& a, int head_dim, int group,
                                   cudaStream_t stream);
// Log-sum-exp merge of the split-KV partials into `out`.
cudaError_t launch_decode_combine(const DecodeArgs& a, int dtype, int head_dim,
                                  cudaStream_t stream);

// Tensor maps (host): a pool viewed as rows [num_blocks * Hkv * 16] x head_dim bf16,
// box 64 columns x 16 rows, 128-byte swizzle.
bool make_pool_map(CUtensorMap* m, const void* pool, int64_t rows, int head_dim);
// The same pool (head_dim 128) as one box per 16-row block: dims {64 columns, 8 rows,
// 2 column halves, rows / 8 row groups}, box {64, 8, 2, 2} = 4 KB, landing in shared
// memory as [row group][half][8 rows][128 B] with the 128-byte swizzle.
bool make_pool_block_map(CUtensorMap* m, const void* pool, int64_t rows);
// cudaFuncSetAttribute(kern, MaxDynamicSharedMemorySize, bytes), made once per kernel and
// device (later calls with no more bytes return at once).
cudaError_t set_smem_once(const void* kern, int bytes);
// q [tokens][Hq][head_dim] bf16 read as boxes of 64 columns x G heads x tok tokens.
bool make_q_group_map(CUtensorMap* m, const void* q, int tokens, int hq, int head_dim, int G,
                      int tok);

cudaError_t launch_kv_append(void* k_pool, void* v_pool, const int64_t* slot_mapping,
                             const void* k, const void* v, int64_t num_tokens, int num_kv_heads,
                             int row_bytes, int block_size, int64_t num_blocks, int* status,
                             cudaStream_t stream);

cudaError_t launch_copy_blocks(void* k_pool, void* v_pool, const int32_t* pairs, int num_pairs,
                               int64_t block_bytes, int64_t num_blocks, int* status,
                               cudaStream_t stream);

struct PrefillArgs {
    int head_dim;     // 64 or 128
    int block_size;   // tokens per pool block: 16 or 32
    void* out;
    const void* q;
    const void* k_pool;
    const void* v_pool;
    const int32_t* block_tables;
    const int32_t* cached_lens;
    const int32_t* new_lens;
    const int32_t* q_offsets;
    int* status;
    int64_t num_blocks;
    int max_blocks_per_seq;
    int num_reqs;
    int total_new;
    int max_new;
    int num_q_heads;
    int num_kv_heads;
    float scale_log2;
    // Cascade mode (shared-prefix decode): one "request" whose cascade_keys keys are the
    // shared prefix and whose cascade_rows query rows are the sequences (one token each);
    // every row attends all prefix keys (no causal mask), the grid's z dimension splits
    // the prefix's tiles (cascade_tiles_per_split each) and split z writes its partial to
    // slot z of the split-KV partials (max_parts_total slots per row) instead of `out`.
    int cascade;
    int cascade_keys;   // cascade: prefix length (keys); rows come from cascade_rows
    int cascade_rows;   // cascade: number of sequences (query rows per head)
    int cascade_tiles_per_split;   // cascade: 128-key tiles per split (grid z = splits)
    int max_parts_total;
    float* o_part;
    float* m_part;
    float* l_part;
    // A CTA whose rows all attend at least this many keys stores P as one bf16 value
    // (round to nearest); otherwise as bf16 hi + lo (see the prefill kernel).
    int p_single_min_keys;
};

cudaError_t launch_paged_prefill(const PrefillArgs& a, int group, cudaStream_t stream);

}  // namespace pkv
