/*
 * pkv.h -- C ABI of libpkv: paged KV-cache attention for one NVIDIA GB300 (sm_103a).
 *
 * The operation (pages: "Paged Attention for Efficient Memory Management",
 * krlt.com Triptych day 152, body and "Look closer"; "PagedAttention and
 * RadixAttention: Let's Talk About KV Cache", aitalk.it, section "PagedAttention:
 * Memory Like an Operating System"): each sequence's keys and values are cut into
 * fixed-size blocks of B tokens held anywhere in one global pool; a per-sequence
 * block table maps logical block j to a physical block id; new tokens are written
 * into the next slot of the current block; attention walks the block table and
 * gathers the blocks, and computes exactly ordinary softmax attention over the
 * logically contiguous sequence.
 *
 * Conventions for every call below
 *  - Pool layout (the pages fix none; this library's contract):
 *      k_pool, v_pool: [num_blocks][num_kv_heads][block_size][head_dim], row-major,
 *      separate tensors, same dtype.  Slot s = block * block_size + offset.
 *  - GQA: query head h reads kv head h / (num_q_heads / num_kv_heads).
 *  - Supported: block_size 16 or 32 (the pages name both), head_dim 64 or 128,
 *    dtype PKV_F32 or PKV_BF16 (cascade decode: PKV_BF16 only),
 *    num_q_heads / num_kv_heads in {1, 2, 4, 8}.
 *    Anything else returns PKV_ERR_UNSUPPORTED before any launch.
 *  - Pointers marked "device" are CUDA device addresses owned by the caller; the
 *    library never frees or retains them after the call returns, and allocates no
 *    device memory on these paths (scratch is passed in as `workspace`).
 *  - `stream` is a cudaStream_t passed as void* (NULL = legacy default stream).
 *    All device work is enqueued asynchronously on it; no call synchronises except
 *    pkv_read_device_status.  The kernel calls may therefore be recorded with stream
 *    capture into a CUDA graph and replayed (make one call outside capture first, so
 *    that the per-device status word and side stream exist); pkv_paged_decode_cascade
 *    forks onto a library-owned stream and joins back within the call.  Kernels are
 *    launched with programmatic dependent launch: a kernel may be placed on the SMs
 *    while the stream's previous kernel finishes, but it reads no input before that
 *    kernel has completed and its writes are visible, so inputs written by the
 *    caller's own kernels on the same stream are safe.
 *  - Argument errors are detected on the host and returned synchronously before any
 *    launch.  A failed launch returns PKV_ERR_CUDA.  Conditions only the device can
 *    see (a slot or block id outside the pool, a pipeline wait that ran out of time)
 *    make the kernel skip the offending access and raise a bit in the library's
 *    device status word; read it with pkv_read_device_status.
 *  - No C++ exception crosses this ABI.
 *  - Each call that enqueues kernels opens an NVTX range named after itself for the
 *    length of the call, so that profilers group and select its kernels (a few
 *    nanoseconds when no tool is attached).
 */
#ifndef PKV_H_
#define PKV_H_

#include <stddef.h>
#include <stdint.h>

#ifdef __cplusplus
extern "C" {
#endif

typedef enum pkv_status {
    PKV_OK = 0,
    PKV_ERR_INVALID = 1,      /* bad argument (null pointer, negative size, inconsistent shape) */
    PKV_ERR_UNSUPPORTED = 2,  /* valid but not implemented (dtype, head_dim, block size, group) */
    PKV_ERR_CUDA = 3,         /* a CUDA runtime call or launch failed */
    PKV_ERR_TIMEOUT = 4,      /* device status: a bounded pipeline wait expired */
    PKV_ERR_OOB = 5,          /* device status: a slot / block id pointed outside the pool */
    PKV_ERR_NOMEM = 6,        /* allocator: not enough free blocks, or workspace too small */
    PKV_ERR_NOT_FOUND = 7     /* allocator: unknown sequence id, or id already present */
} pkv_status;

typedef enum pkv_dtype { PKV_F32 = 0, PKV_BF16 = 1 } pkv_dtype;

/* Description of one K pool and one V pool (same shape and dtype). */
typedef struct pkv_pool_desc {
    int64_t num_blocks;   /* physical blocks in each pool */
    int32_t block_size;   /* tokens per block (B); 16 or 32 */
    int32_t num_kv_heads; /* Hkv */
    int32_t head_dim;     /* D: 64 or 128 */
    int32_t dtype;        /* pkv_dtype */
} pkv_pool_desc;

/* Static string for a status code. */
const char* pkv_status_string(int status);

/* ABI version of this header (major * 100 + minor). */
int pkv_version(void);

/* Bytes of ONE pool (K or V) described by `pool`; 0 for an invalid description.
 * 2 * pkv_pool_bytes(...) / (num_blocks * block_size) is the per-layer KV cost of a
 * token, the figure the aitalk.it page quotes for Llama-3.1-70B (about 0.31 MB per
 * token over all layers in BF16). */
uint64_t pkv_pool_bytes(const pkv_pool_desc* pool);

/* ---------------------------------------------------------------- kv_append
 * Writes new tokens' K/V rows into their pool slots ("writes append within the
 * current block", Triptych page, body; "append on decode", aifetchly SGLang guide,
 * "Dynamic Node Splitting and Branch Insertion").
 *   slot_mapping  device int64 [num_tokens]; token t goes to slot slot_mapping[t];
 *                 a negative slot skips the token (padding).
 *   k, v          device [num_tokens][num_kv_heads][head_dim], pool dtype, contiguous.
 *   k_pool/v_pool device pools (see layout above), written in place.
 * The copy is bit-exact.  A slot >= num_blocks * block_size is not written and raises
 * PKV_ERR_OOB in the device status word.  num_tokens == 0 is a no-op. */
pkv_status pkv_kv_append(const pkv_pool_desc* pool, void* k_pool, void* v_pool,
                         const int64_t* slot_mapping, const void* k, const void* v,
                         int64_t num_tokens, void* stream);

/* ---------------------------------------------------------------- paged_decode
 * One query token per sequence attends to its first context_lens[s] tokens, gathered
 * through block_tables (Triptych page: "the kernel walks the block table and gathers
 * the relevant physical blocks").  Long contexts are split into partitions of
 * `partition_blocks` blocks processed by separate CTAs and merged by a log-sum-exp
 * combine (split-KV decode, aifetchly SGLang guide, "Integrating FlashInfer").
 *   out           device [num_seqs][num_q_heads][head_dim], pool dtype (bf16 rounded
 *                 to nearest even).
 *   q             device [num_seqs][num_q_heads][head_dim], pool dtype.
 *   block_tables  device int32 [num_seqs][max_blocks_per_seq]; entries past
 *                 ceil(context_len / block_size) are never read.
 *   context_lens  device int32 [num_seqs], each in [1, max_blocks_per_seq * block_size]
 *                 (the token being decoded is included: write it with kv_append first).
 *                 A length below 1 raises PKV_ERR_INVALID in the device status word and
 *                 gives that sequence's output rows zeros; a length above the range
 *                 raises PKV_ERR_OOB and is clamped to it.
 *   max_context   host upper bound of context_lens (sizes the grid and workspace).
 *   scale         softmax scale applied to q.k (e.g. 1/sqrt(head_dim)).
 *   partition_blocks  blocks per split-KV partition; 0 lets the library choose.
 *   workspace     device scratch of at least pkv_paged_decode_workspace_bytes(...) bytes,
 *                 16-byte aligned; may be NULL when that size is 0.  Contents need no
 *                 initialisation and are clobbered.
 * Entries past context_len inside the last block may hold anything (NaN included);
 * they never reach the output. */
size_t pkv_paged_decode_workspace_bytes(int num_seqs, int num_q_heads, int head_dim,
                                        int max_context, int block_size, int partition_blocks);
pkv_status pkv_paged_decode(const pkv_pool_desc* pool, void* out, const void* q,
                            const void* k_pool, const void* v_pool,
                            const int32_t* block_tables, int max_blocks_per_seq,
                            const int32_t* context_lens, int max_context, int num_seqs,
                            int num_q_heads, float scale, int partition_blocks,
                            void* workspace, size_t workspace_bytes, void* stream);

/* kv_append and paged_decode of one decode step in one pass.  k_new / v_new hold the K /
 * V of each sequence's newest token, position context_lens[s] - 1; it goes to the slot
 * that position has in the block table, block_tables[s][(L - 1) / block_size] at offset
 * (L - 1) % block_size: the next slot of the sequence, which appending fills (Triptych
 * page, "Paged Attention for Efficient Memory Management").  The decode CTA whose chunk
 * holds that position stores the token into the pool and attends it straight from
 * k_new / v_new, so no append launch precedes the decode.  Pools and output equal those
 * of pkv_kv_append with those slots followed by pkv_paged_decode.
 *   k_new, v_new    device [num_seqs][num_kv_heads][head_dim], pool dtype, 16-byte
 *                   aligned; read only.
 *   k_pool, v_pool  written at the new tokens' slots only.
 * Each sequence's new slot must be its own (not reached through another sequence's table:
 * copy-on-write of a shared last block, pkv_alloc_append, guarantees that).  A table entry
 * outside [0, num_blocks) for the new slot skips its store and raises PKV_ERR_OOB in the
 * device status word.  Other arguments, errors and the workspace as pkv_paged_decode. */
pkv_status pkv_paged_decode_append(const pkv_pool_desc* pool, void* out, const void* q,
                                   void* k_pool, void* v_pool, const void* k_new,
                                   const void* v_new, const int32_t* block_tables,
                                   int max_blocks_per_seq, const int32_t* context_lens,
                                   int max_context, int num_seqs, int num_q_heads, float scale,
                                   int partition_blocks, void* workspace, size_t workspace_bytes,
                                   void* stream);

/* ---------------------------------------------------------------- decode step from host memory
 * The fused decode step with its inputs and output in host memory: the step's inputs sit
 * packed in one host buffer laid out as pkv_decode_step_layout gives (q, k_new, v_new,
 * block_tables, context_lens, each at a 256-byte aligned offset, in the layouts
 * pkv_paged_decode_append takes), so that they move in one host-to-device copy.
 *   layout  out: byte offsets of the five arrays and the buffer's total size.
 * Returns PKV_ERR_INVALID for bad sizes. */
typedef struct pkv_step_layout {
    uint64_t q, k_new, v_new, block_tables, context_lens, bytes;
} pkv_step_layout;
pkv_status pkv_decode_step_layout(const pkv_pool_desc* pool, int num_seqs, int num_q_heads,
                                  int max_blocks_per_seq, pkv_step_layout* layout);

/* Device staging the host step needs: the packed inputs, the output and the split-KV
 * workspace (0 for invalid arguments). */
size_t pkv_paged_decode_append_host_staging_bytes(const pkv_pool_desc* pool, int num_seqs,
                                                  int num_q_heads, int max_blocks_per_seq,
                                                  int max_context, int partition_blocks);

/* One decode step from host memory, queued on `stream`: pkv_paged_decode_append over
 * the inputs packed in host_in (layout.bytes bytes, as pkv_decode_step_layout says),
 * with the output ([num_seqs][num_q_heads][head_dim], pool dtype) going to host_out.
 * Page-locked host buffers that CUDA maps into the device address space (cudaHostAlloc,
 * cudaMallocHost, cudaHostRegister; all of them under unified addressing) are read and
 * written by the kernels in place, over the host link, with no staging copy; other host
 * memory is copied into `staging` first and the output copied back.  host_out is
 * complete once the stream has been synchronised, and host_in must stay unchanged until
 * then.
 *   staging  device, >= pkv_paged_decode_append_host_staging_bytes(...) bytes, 256-byte
 *            aligned; contents need no initialisation and are clobbered (it holds the
 *            split-KV partials in either case).
 * Argument errors as pkv_paged_decode_append; PKV_ERR_NOMEM if staging is too small. */
pkv_status pkv_paged_decode_append_host(const pkv_pool_desc* pool, void* k_pool, void* v_pool,
                                        const void* host_in, void* host_out,
                                        int max_blocks_per_seq, int max_context, int num_seqs,
                                        int num_q_heads, float scale, int partition_blocks,
                                        void* staging, size_t staging_bytes, void* stream);

/* Partition size (in blocks) pkv_paged_decode uses for partition_blocks == 0; it
 * depends only on these arguments (0 for invalid ones). */
int pkv_paged_decode_auto_partition(int num_seqs, int num_q_heads, int max_context,
                                    int block_size);

/* Same decode for callers that cannot allocate device memory: code running where
 * cudaMalloc is not allowed or not wanted (inside a caller-managed memory pool or
 * arena with a fixed budget, a plugin whose host process owns every allocation, a
 * real-time loop that must not touch the allocator).  The pages have no counterpart;
 * this is a library convenience.  Arguments are those of pkv_paged_decode minus the
 * workspace: the split-KV partials go to a scratch array built into the library
 * (64 MiB, reserved on every GPU that loads libpkv's device code and held until the
 * process exits).  The call allocates nothing: no cudaMalloc, no cudaFree, no
 * allocating library routine.
 *  - Its first call on a device looks up that device's copy of the scratch array
 *    (with the device current); make that first call before any stream capture.
 *  - Requests whose partials need more than 64 MiB
 *    (pkv_paged_decode_workspace_bytes(...) > 64 MiB) return PKV_ERR_NOMEM before
 *    any launch.
 *  - Every call shares the one array, which keeps the last call's contents.  The
 *    partials are fully written before they are read, so nothing needs clearing, but
 *    calls whose kernels overlap on the GPU (other streams, other threads) race on
 *    it: serialise them. */
pkv_status pkv_paged_decode_noalloc(const pkv_pool_desc* pool, void* out, const void* q,
                                    const void* k_pool, const void* v_pool,
                                    const int32_t* block_tables, int max_blocks_per_seq,
                                    const int32_t* context_lens, int max_context, int num_seqs,
                                    int num_q_heads, float scale, int partition_blocks,
                                    void* stream);

/* ---------------------------------------------------------------- cascade decode
 * Decode of sequences that all begin with the same prefix_len tokens held in the same physical
 * blocks (a prompt shared through the block tables: Triptych page, "Sharing is a pointer
 * change"; aitalk.it, "RadixAttention").  The result equals pkv_paged_decode's; the work is
 * arranged so that the shared blocks are read once: (1) every sequence's query heads attend
 * the prefix blocks as one tensor-core pass (the prefill kernel with no causal mask), (2) each
 * sequence's private suffix (tokens from prefix_len on) is decoded with split-KV partitions,
 * (3) the log-sum-exp combine merges the prefix partial with the suffix partials.
 *   prefix_blocks  device int32 [prefix_len / block_size]: the shared blocks; every
 *                  sequence's block_tables row must start with them.
 *   prefix_len     > 0, a multiple of block_size; context_lens[s] >= prefix_len.
 *   max_context    host upper bound of context_lens (>= prefix_len).
 *   workspace      >= pkv_paged_decode_cascade_workspace_bytes(...) bytes, 16-byte aligned.
 * Other arguments as pkv_paged_decode.  Requires PKV_BF16.  The prefix pass runs on a
 * library-owned stream forked from `stream`; every return, errors included, first makes
 * `stream` wait for it, so no work of the call outlives its ordering on `stream` and a
 * stream capture always ends with the fork joined. */
size_t pkv_paged_decode_cascade_workspace_bytes(int num_seqs, int num_q_heads, int head_dim,
                                                int prefix_len, int max_context, int block_size,
                                                int partition_blocks);
pkv_status pkv_paged_decode_cascade(const pkv_pool_desc* pool, void* out, const void* q,
                                    const void* k_pool, const void* v_pool,
                                    const int32_t* prefix_blocks, int prefix_len,
                                    const int32_t* block_tables, int max_blocks_per_seq,
                                    const int32_t* context_lens, int max_context, int num_seqs,
                                    int num_q_heads, float scale, int partition_blocks,
                                    void* workspace, size_t workspace_bytes, void* stream);

/* Cascade decode with the step's append fused in, as pkv_paged_decode_append does for
 * pkv_paged_decode: k_new / v_new [num_seqs][num_kv_heads][head_dim] hold each sequence's
 * newest token, position context_lens[s] - 1, which must lie in the private suffix
 * (context_lens[s] > prefix_len).  The suffix decode stores it into the slot the block
 * table gives for that position and attends it from k_new / v_new.  A sequence whose
 * newest token lies inside the shared prefix is not stored and raises PKV_ERR_INVALID in
 * the device status word.  Other arguments, errors and the workspace as
 * pkv_paged_decode_cascade. */
pkv_status pkv_paged_decode_cascade_append(const pkv_pool_desc* pool, void* out, const void* q,
                                           void* k_pool, void* v_pool, const void* k_new,
                                           const void* v_new, const int32_t* prefix_blocks,
                                           int prefix_len, const int32_t* block_tables,
                                           int max_blocks_per_seq, const int32_t* context_lens,
                                           int max_context, int num_seqs, int num_q_heads,
                                           float scale, int partition_blocks, void* workspace,
                                           size_t workspace_bytes, void* stream);

/* ---------------------------------------------------------------- paged_prefill
 * Causal prefill of new tokens over a cached prefix ("computes only the unseen
 * suffix" while reusing the cached prefix's K/V: aitalk.it, "RadixAttention: A Tree
 * That Does Not Forget"; aifetchly guide, "Prefill Bypass").  Request r has
 * cached_lens[r] tokens already in the pool followed by new_lens[r] new tokens whose
 * K/V must already be in the pool (kv_append first).  Query row q_offsets[r] + i
 * (i < new_lens[r]) attends keys 0 .. cached_lens[r] + i.  bf16 pools run on the
 * tcgen05 tensor cores with TMEM accumulators (bf16 in, fp32 accumulate, bf16 out), with
 * one persistent CTA per SM when num_reqs <= 128 (one CTA per 128-row query tile
 * otherwise); fp32 pools run on a tiled CUDA-core kernel (fp32 throughout).  A block id
 * outside [0, num_blocks) inside a request's keys is not read and raises PKV_ERR_OOB in
 * the device status word (that request's output is then not valid).
 *   out, q        device [total_new][num_q_heads][head_dim], the pools' dtype.
 *   block_tables  device int32 [num_reqs][max_blocks_per_seq].
 *   cached_lens, new_lens  device int32 [num_reqs]; cached >= 0, new >= 0,
 *                 cached + new <= max_blocks_per_seq * block_size.
 *   q_offsets     device int32 [num_reqs + 1], exclusive prefix sum of new_lens.
 *   max_new       host upper bound of new_lens (sizes the grid).
 */
pkv_status pkv_paged_prefill(const pkv_pool_desc* pool, void* out, const void* q,
                             const void* k_pool, const void* v_pool,
                             const int32_t* block_tables, int max_blocks_per_seq,
                             const int32_t* cached_lens, const int32_t* new_lens,
                             const int32_t* q_offsets, int num_reqs, int total_new, int max_new,
                             int num_q_heads, float scale, void* stream);

/* ---------------------------------------------------------------- prefill step from host memory
 * The prefill step (kv_append of the new tokens' K/V, then pkv_paged_prefill) with its
 * inputs and output in host memory.  The inputs sit packed in one host buffer laid out
 * as pkv_prefill_step_layout gives, each array at a 256-byte aligned offset and in the
 * layout the device calls take: first the part copied to the device (q, which the
 * tensor-core prefill loads by TMA, and the block tables, cached_lens, new_lens and
 * q_offsets: `copied_bytes` bytes), then the new rows k_new, v_new ([total_new]
 * [num_kv_heads][head_dim]) and slot_mapping (int64 [total_new]).  (All of it is copied
 * to the device; `copied_bytes` marks where the per-request arrays end.)
 *   layout  out: byte offsets of the eight arrays, copied_bytes and the total size.
 * Returns PKV_ERR_INVALID for bad sizes. */
typedef struct pkv_prefill_layout {
    uint64_t q, block_tables, cached_lens, new_lens, q_offsets, copied_bytes;
    uint64_t k_new, v_new, slot_mapping, bytes;
} pkv_prefill_layout;
pkv_status pkv_prefill_step_layout(const pkv_pool_desc* pool, int num_reqs, int total_new,
                                   int num_q_heads, int max_blocks_per_seq,
                                   pkv_prefill_layout* layout);

/* Device staging the host prefill step needs: the packed inputs and the output (0 for
 * invalid arguments). */
size_t pkv_paged_prefill_append_host_staging_bytes(const pkv_pool_desc* pool, int num_reqs,
                                                   int total_new, int num_q_heads,
                                                   int max_blocks_per_seq);

/* One prefill step from host memory, queued on `stream`: host_in goes to `staging`,
 * pkv_kv_append stores the new rows, pkv_paged_prefill writes the output
 * ([total_new][num_q_heads][head_dim], pool dtype) into staging, which is copied back
 * to host_out.  Host buffers should be page-locked for the copies to run
 * asynchronously.  The call reads q_offsets from host_in (it must be the exclusive
 * prefix sum of new_lens, ending at total_new: PKV_ERR_INVALID otherwise) and splits the
 * requests into up to 4 chunks of about equal new rows: a chunk's q, new rows and slots
 * are copied in on a library-owned stream while the previous chunk's append and prefill
 * run on `stream` and the one before's output is copied back on a second library-owned
 * stream; every return, errors included, first makes `stream` wait for both.  host_out
 * is complete once `stream` has been synchronised, and host_in must stay unchanged until
 * then.
 *   staging  device, >= pkv_paged_prefill_append_host_staging_bytes(...) bytes, 256-byte
 *            aligned; contents need no initialisation and are clobbered.
 * Argument errors as pkv_kv_append and pkv_paged_prefill; PKV_ERR_NOMEM if staging is
 * too small. */
pkv_status pkv_paged_prefill_append_host(const pkv_pool_desc* pool, void* k_pool, void* v_pool,
                                         const void* host_in, void* host_out, int num_reqs,
                                         int total_new, int max_new, int num_q_heads,
                                         int max_blocks_per_seq, float scale, void* staging,
                                         size_t staging_bytes, void* stream);

/* ---------------------------------------------------------------- copy_blocks
 * Copy-on-write support (Triptych page: "Mutation after a fork uses copy-on-write so
 * other references stay valid"): pool[dst] = pool[src] for both pools, every kv head
 * and slot of the block.
 *   pairs  device int32 [num_pairs][2] = (src, dst); dst blocks must be distinct and
 *          no dst may be another pair's src.
 * An id outside [0, num_blocks) skips that pair and raises PKV_ERR_OOB in the device
 * status word. */
pkv_status pkv_copy_blocks(const pkv_pool_desc* pool, void* k_pool, void* v_pool,
                           const int32_t* pairs, int num_pairs, void* stream);

/* ---------------------------------------------------------------- device status
 * Synchronises `stream`, returns in *status_out the first error any kernel of this
 * library raised on the current device since the last read (PKV_OK if none), and
 * clears it. */
pkv_status pkv_read_device_status(int* status_out, void* stream);

/* ---------------------------------------------------------------- host block allocator
 * Host-side (pure CPU) block manager that produces slots, block tables and
 * copy-on-write pairs (Triptych page, body: on-demand blocks, refcounts on fork,
 * copy-on-write on divergence, blocks return to the pool at refcount zero; khotyn.com
 * page, "PagedAttention": a new block only when the last one is full, so at most one
 * partially filled block per sequence).  Not thread-safe: one handle per thread.
 * Sequence ids are caller-chosen int64 values. */
typedef struct pkv_alloc pkv_alloc;

/* New allocator over blocks [0, num_blocks).  seed == 0 hands out free blocks in
 * ascending order; any other seed starts from a seeded shuffle of the free list (the
 * scattered placement of a long-running server).  NULL on bad arguments. */
pkv_alloc* pkv_alloc_create(int64_t num_blocks, int block_size, uint64_t seed);
void pkv_alloc_destroy(pkv_alloc* a);

/* Registers seq_id holding num_tokens (>= 0) tokens: ceil(num_tokens / B) new blocks.
 * PKV_ERR_NOMEM leaves the allocator unchanged; PKV_ERR_NOT_FOUND if seq_id exists. */
pkv_status pkv_alloc_add_seq(pkv_alloc* a, int64_t seq_id, int64_t num_tokens);

/* child shares every block of parent (refcount + 1 each) and its token count. */
pkv_status pkv_alloc_fork(pkv_alloc* a, int64_t parent, int64_t child);

/* Reserves slots for n (>= 0) new tokens of seq_id, written to slots_out[n].  A new
 * block is taken only when the last block is full.  If the last, partially filled
 * block is shared (refcount > 1) it is first replaced by a private copy: the pair
 * (old, new) is written to cow_pairs_out[0..1] and *num_cow_out = 1 (else 0); the
 * caller must run pkv_copy_blocks on it before writing the slots.  On PKV_ERR_NOMEM
 * nothing changes. */
pkv_status pkv_alloc_append(pkv_alloc* a, int64_t seq_id, int64_t n, int64_t* slots_out,
                            int32_t* cow_pairs_out, int* num_cow_out);

/* Drops seq_id: refcount - 1 on each of its blocks; a block reaching 0 is free again. */
pkv_status pkv_alloc_free_seq(pkv_alloc* a, int64_t seq_id);

/* Host int32 [S][max_blocks] table of the given sequences, -1 padded.  PKV_ERR_INVALID
 * if a sequence holds more than max_blocks blocks. */
pkv_status pkv_alloc_block_table(const pkv_alloc* a, const int64_t* seq_ids, int num_seqs,
                                 int32_t* out, int max_blocks);

/* Registers seq_id holding num_tokens tokens whose first num_shared blocks are the given
 * existing blocks (refcount + 1 each), e.g. a prefix found by pkv_pcache_match or
 * pkv_radix_match; the remaining ceil(num_tokens / B) - num_shared blocks are new.  The
 * last shared block may be partially filled (num_tokens < num_shared * B): the next
 * pkv_alloc_append then copies it first (copy-on-write).  PKV_ERR_INVALID if a block is
 * not allocated or num_shared exceeds the blocks num_tokens needs. */
pkv_status pkv_alloc_add_seq_shared(pkv_alloc* a, int64_t seq_id, const int32_t* shared_blocks,
                                    int num_shared, int64_t num_tokens);

int64_t pkv_alloc_num_free(const pkv_alloc* a);
int pkv_alloc_refcount(const pkv_alloc* a, int64_t block);            /* -1 if out of range */
int64_t pkv_alloc_seq_len(const pkv_alloc* a, int64_t seq_id);        /* -1 if unknown */
int64_t pkv_alloc_seq_num_blocks(const pkv_alloc* a, int64_t seq_id); /* -1 if unknown */

/* ---------------------------------------------------------------- prefix reuse: block hashes
 * Chained block hashes (aitalk.it, "Two Layers, Not Two Rivals": each completed block is
 * hashed from its parent block's hash, its tokens and extra metadata, so equal prefixes give
 * equal chains; "Beyond the Two Techniques": a tenant salt mixed into the hash keeps tenants'
 * caches apart).  The cache points at allocator blocks and holds one reference per block it
 * registers.  Host only; not thread-safe. */
typedef struct pkv_pcache pkv_pcache;

/* The hash of one block: parent_hash (0 for the first block), salt, n tokens, extra. */
uint64_t pkv_block_hash(uint64_t parent_hash, uint64_t salt, const int32_t* tokens, int n,
                        uint64_t extra);
pkv_pcache* pkv_pcache_create(pkv_alloc* a);
void pkv_pcache_destroy(pkv_pcache* pc); /* drops the cache's references */
/* Longest chain of cached full blocks that spells the first tokens of `tokens` under `salt`;
 * writes their ids to blocks_out (at most max_blocks) and returns how many (matched tokens =
 * count * B), -1 on bad arguments.  Entries compare their tokens, so a hash collision never
 * matches.  Marks the matched entries most recently used. */
int pkv_pcache_match(pkv_pcache* pc, const int32_t* tokens, int64_t n, uint64_t salt,
                     int32_t* blocks_out, int max_blocks);
/* Registers the full blocks of seq_id's first n tokens (`tokens` are those tokens) under
 * `salt`; returns the number of newly cached blocks, -1 on bad arguments / unknown seq. */
int pkv_pcache_insert(pkv_pcache* pc, int64_t seq_id, const int32_t* tokens, int64_t n,
                      uint64_t salt);
/* Drops least recently used entries whose block only the cache still holds until the
 * allocator has at least min_free free blocks (or nothing is left to drop); returns the
 * number dropped. */
int64_t pkv_pcache_evict(pkv_pcache* pc, int64_t min_free);
int64_t pkv_pcache_size(const pkv_pcache* pc);

/* ---------------------------------------------------------------- prefix reuse: radix tree
 * Radix tree (compressed trie) of token sequences over the allocator's blocks (aitalk.it,
 * "RadixAttention: A Tree That Does Not Forget"; khotyn.com, "RadixAttention"; aifetchly
 * SGLang guide, "Radix Tree Topology", "Dynamic Node Splitting and Branch Insertion", "LRU
 * Leaf Eviction").  Edges carry token runs, nodes the blocks holding those positions (one
 * reference each).  Host only; not thread-safe. */
typedef struct pkv_radix pkv_radix;

pkv_radix* pkv_radix_create(pkv_alloc* a);
void pkv_radix_destroy(pkv_radix* t); /* drops the tree's references */
/* Longest common prefix of `tokens` with the tree, in tokens (token granularity); writes the
 * blocks of positions [0, m) to blocks_out[0 .. ceil(m / B)) (entries at index >= max_blocks are
 * skipped).  Pass them to pkv_alloc_add_seq_shared; a partial last block is copied on the
 * sequence's first append.  Marks the path most recently used.  -1 on bad arguments. */
int64_t pkv_radix_match(pkv_radix* t, const int32_t* tokens, int64_t n, int32_t* blocks_out,
                        int max_blocks);
/* Inserts seq_id's first n tokens (`tokens`), splitting an edge where they diverge from the
 * tree; new positions reference seq_id's blocks.  PKV_ERR_NOT_FOUND for an unknown seq or one
 * holding fewer than n tokens. */
pkv_status pkv_radix_insert(pkv_radix* t, int64_t seq_id, const int32_t* tokens, int64_t n);
/* delta = +1 / -1 on the lock count of every node on the path of an inserted token sequence
 * (an active request uses it); locked nodes are never evicted.  PKV_ERR_NOT_FOUND if the path
 * does not end on a node boundary (insert the sequence first). */
pkv_status pkv_radix_lock(pkv_radix* t, const int32_t* tokens, int64_t n, int delta);
/* Evicts least recently used unlocked leaves until the allocator has at least min_free free
 * blocks (e.g. 10 % of the pool) or no unlocked leaf is left; a parent left with one child is
 * merged with it.  Returns the number of leaves evicted. */
int64_t pkv_radix_evict(pkv_radix* t, int64_t min_free);
int64_t pkv_radix_num_nodes(const pkv_radix* t);
int64_t pkv_radix_cached_tokens(const pkv_radix* t);

#ifdef __cplusplus
}
#endif

#endif /* PKV_H_ */
