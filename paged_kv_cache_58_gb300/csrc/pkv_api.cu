// C-ABI entry points of libpkv: argument validation, workspace carving and
// kernel launches.  Declarations and contracts are in include/pkv.h.
#include <cuda_runtime.h>

#include <cstdint>
#include <cstdlib>
#include <algorithm>
#include <climits>
#include <cstring>
#include <mutex>

#include <nvtx3/nvToolsExt.h>

#include "../../include/pkv.h"
#include "kernels.h"
#include "prefill_f32.h"

namespace {

constexpr int kChunk = 16;   // the kernels walk sequences in 16-token chunks
constexpr int kMaxDevices = 64;
constexpr double kLog2e = 1.4426950408889634;

// log2(block_size / 16) for the supported block sizes 16 and 32, else -1.
int chunk_shift(int block_size) { return block_size == 16 ? 0 : block_size == 32 ? 1 : -1; }

// Library device status word: first error code raised by a kernel (0 = none).
__device__ int g_pkv_status = 0;

std::mutex g_status_mu;
int* g_status_addr[kMaxDevices] = {nullptr};

// Device address of g_pkv_status on the current device, looked up once per device
// (a __device__ symbol's host-side name is not a device address).
int* status_word() {
    int dev = 0;
    if (cudaGetDevice(&dev) != cudaSuccess || dev < 0 || dev >= kMaxDevices) return nullptr;
    std::lock_guard<std::mutex> lk(g_status_mu);
    if (!g_status_addr[dev]) {
        void* p = nullptr;
        if (cudaGetSymbolAddress(&p, g_pkv_status) != cudaSuccess) return nullptr;
        g_status_addr[dev] = static_cast<int*>(p);
    }
    return g_status_addr[dev];
}

std::mutex g_side_mu;
cudaStream_t g_side_stream[kMaxDevices] = {nullptr};

// A library-owned non-blocking stream per device, for work that runs beside the
// caller's stream inside one call (joined back before the call's last launch).  It has
// the greatest priority, so that its CTAs -- which need a whole SM's shared memory --
// are placed before the caller stream's kernel fills every SM.
cudaStream_t side_stream() {
    int dev = 0;
    if (cudaGetDevice(&dev) != cudaSuccess || dev < 0 || dev >= kMaxDevices) return nullptr;
    std::lock_guard<std::mutex> lk(g_side_mu);
    int least = 0, greatest = 0;
    if (!g_side_stream[dev] &&
        (cudaDeviceGetStreamPriorityRange(&least, &greatest) != cudaSuccess ||
         cudaStreamCreateWithPriority(&g_side_stream[dev], cudaStreamNonBlocking, greatest) !=
             cudaSuccess))
        g_side_stream[dev] = nullptr;
    return g_side_stream[dev];
}

cudaStream_t g_copy_stream[kMaxDevices][2] = {{nullptr, nullptr}};

// Two more library-owned non-blocking streams per device, for the copies of a host-buffer
// step that overlap its kernels on the caller's stream: 0 carries host-to-device copies,
// 1 device-to-host copies, so that both copy directions and the kernels run at once.
cudaStream_t copy_stream(int which) {
    int dev = 0;
    if (cudaGetDevice(&dev) != cudaSuccess || dev < 0 || dev >= kMaxDevices) return nullptr;
    std::lock_guard<std::mutex> lk(g_side_mu);
    cudaStream_t& s = g_copy_stream[dev][which];
    if (!s && cudaStreamCreateWithFlags(&s, cudaStreamNonBlocking) != cudaSuccess) s = nullptr;
    return s;
}

bool aligned16(const void* p) { return (reinterpret_cast<uintptr_t>(p) & 15u) == 0; }

// An NVTX range around each call that enqueues GPU work, named after the call, so that
// a profiler's timeline groups the call's kernels under it and ncu can select them
// (--nvtx --nvtx-include "pkv_paged_decode/").  With no tool attached a push and a pop
// cost a few nanoseconds.
struct CallRange {
    explicit CallRange(const char* name) { nvtxRangePushA(name); }
    ~CallRange() { nvtxRangePop(); }
    CallRange(const CallRange&) = delete;
    CallRange& operator=(const CallRange&) = delete;
};

int elem_bytes(int dtype) { return dtype == PKV_BF16 ? 2 : 4; }

pkv_status check_pool(const pkv_pool_desc* pool) {
    if (!pool) return PKV_ERR_INVALID;
    if (pool->num_blocks <= 0 || pool->num_kv_heads <= 0 || pool->head_dim <= 0 ||
        pool->block_size <= 0)
        return PKV_ERR_INVALID;
    if (pool->dtype != PKV_F32 && pool->dtype != PKV_BF16) return PKV_ERR_UNSUPPORTED;
    if (chunk_shift(pool->block_size) < 0) return PKV_ERR_UNSUPPORTED;
    if (pool->head_dim != 64 && pool->head_dim != 128) return PKV_ERR_UNSUPPORTED;
    if (pool->num_kv_heads > 65535) return PKV_ERR_UNSUPPORTED;
    if (pool->num_blocks > INT32_MAX) return PKV_ERR_UNSUPPORTED;
    return PKV_OK;
}

pkv_status from_cuda(cudaError_t e) { return e == cudaSuccess ? PKV_OK : PKV_ERR_CUDA; }

int ceil_div(int64_t a, int64_t b) { return static_cast<int>((a + b - 1) / b); }

// Partition policy for split-KV decode, in 16-token chunks: at least 64 chunks (1024
// tokens) per partition -- each CTA pays a fixed start-up (block ids, first copies
// in flight, merge), and on the Llama-3-8B-shaped batch 64 chunks measured best (16:
// 81 %, 32: 89 %, 64: 90 % of the copy bandwidth) -- and at most 64 partitions per
// sequence to bound the workspace; shrink partitions (down to 8 chunks) while fewer
// than 2 x 152 CTAs would be busy.  The result is a multiple of 4 chunks (one per warp
// per step) and so of 2 (a whole number of 32-token blocks): each halving rounds up to
// a multiple of 4.
// The CTA estimate counts ceil(Hq / 8) kv heads per sequence (a lower bound: a
// GQA group is at most 8 query heads) so that the choice, and with it the
// workspace size, depends only on (num_seqs, num_q_heads, max_context).
int auto_partition_chunks(int num_seqs, int num_q_heads, int max_context) {
    const int max_chunks = ceil_div(max_context, kChunk);
    const int64_t kv_heads_min = ceil_div(num_q_heads, 8);
    int pc = ceil_div(max_chunks, 64);
    if (pc < 64) pc = 64;
    pc = (pc + 3) / 4 * 4;
    while (pc > 8 && static_cast<int64_t>(num_seqs) * kv_heads_min * ceil_div(max_chunks, pc) <
                         304)
        pc = (pc / 2 + 3) / 4 * 4;
    return pc;
}

// The same in pool blocks.
int auto_partition(int num_seqs, int num_q_heads, int max_context, int block_size) {
    return auto_partition_chunks(num_seqs, num_q_heads, max_context) >> chunk_shift(block_size);
}

// bf16 decode runs on the tensor-core kernel; PKV_DECODE_KERNEL=simt selects the
// CUDA-core kernel instead (read at each call; used to test and compare the two).
bool decode_use_simt() {
    const char* v = std::getenv("PKV_DECODE_KERNEL");
    return v != nullptr && std::strcmp(v, "simt") == 0;
}

// Prefill probabilities: one bf16 value per weight for query tiles whose rows all
// attend at least kPSingleMinKeys keys, the exact hi + lo split below that;
// PKV_PREFILL_P=split forces the split everywhere (read at each call; used to test and
// compare the two).
constexpr int kPSingleMinKeys = 1024;
int prefill_p_single_min_keys() {
    const char* v = std::getenv("PKV_PREFILL_P");
    return (v != nullptr && std::strcmp(v, "split") == 0) ? INT_MAX : kPSingleMinKeys;
}

// PKV_TEST_DECODE_STALL=1 arms the decode kernels' timeout test hook (one wait of one
// warp runs out of time; read at each call; tests only).
int decode_test_stall() {
    const char* v = std::getenv("PKV_TEST_DECODE_STALL");
    return v != nullptr && std::strcmp(v, "1") == 0;
}

// PKV_TEST_CASCADE_SUFFIX_FAIL=1 makes the cascade decode report a failed suffix launch
// (without launching it) after its prefix pass was forked onto the side stream, so that
// tests reach that error path (read at each call; tests only).
bool cascade_test_fail_suffix() {
    const char* v = std::getenv("PKV_TEST_CASCADE_SUFFIX_FAIL");
    return v != nullptr && std::strcmp(v, "1") == 0;
}

size_t decode_workspace(int num_seqs, int num_q_heads, int head_dim, int max_parts) {
    if (max_parts <= 1) return 0;
    const size_t rows = static_cast<size_t>(num_seqs) * num_q_heads * max_parts;
    const size_t o = rows * head_dim * sizeof(float);
    const size_t ml = (rows * sizeof(float) + 15) / 16 * 16;
    return o + 2 * ml;
}

// Built-in decode scratch for pkv_paged_decode_noalloc: callers that cannot
// allocate device memory get the split-KV partials here.  The array is reserved on
// every GPU that loads this library's device code and held until the process exits.
constexpr size_t kNoAllocScratchBytes = 64u << 20;  // 64 MiB
static __device__ __align__(256) unsigned char g_noalloc_scratch[kNoAllocScratchBytes];

std::mutex g_scratch_mu;
void* g_scratch_addr[kMaxDevices] = {nullptr};

// Device address of g_noalloc_scratch on the current device.  The host-side name
// of a __device__ array is only a stand-in, so the address is looked up once per
// device, with that device current, and cached; nullptr if the lookup fails.
void* noalloc_scratch() {
    int dev = 0;
    if (cudaGetDevice(&dev) != cudaSuccess || dev < 0 || dev >= kMaxDevices) return nullptr;
    std::lock_guard<std::mutex> lk(g_scratch_mu);
    if (!g_scratch_addr[dev]) {
        void* p = nullptr;
        if (cudaGetSymbolAddress(&p, g_noalloc_scratch) != cudaSuccess) return nullptr;
        g_scratch_addr[dev] = p;
    }
    return g_scratch_addr[dev];
}

}  // namespace

extern "C" {

const char* pkv_status_string(int status) {
    switch (status) {
        case PKV_OK: return "ok";
        case PKV_ERR_INVALID: return "invalid argument";
        case PKV_ERR_UNSUPPORTED: return "unsupported configuration";
        case PKV_ERR_CUDA: return "CUDA error";
        case PKV_ERR_TIMEOUT: return "device pipeline wait timed out";
        case PKV_ERR_OOB: return "slot or block id outside the pool";
        case PKV_ERR_NOMEM: return "out of blocks or workspace too small";
        case PKV_ERR_NOT_FOUND: return "unknown or duplicate sequence id";
        default: return "unknown status";
    }
}

int pkv_version(void) { return 100; }

uint64_t pkv_pool_bytes(const pkv_pool_desc* pool) {
    if (!pool || pool->num_blocks <= 0 || pool->block_size <= 0 || pool->num_kv_heads <= 0 ||
        pool->head_dim <= 0 || (pool->dtype != PKV_F32 && pool->dtype != PKV_BF16))
        return 0;
    return static_cast<uint64_t>(pool->num_blocks) * pool->num_kv_heads * pool->block_size *
           pool->head_dim * elem_bytes(pool->dtype);
}

pkv_status pkv_kv_append(const pkv_pool_desc* pool, void* k_pool, void* v_pool,
                         const int64_t* slot_mapping, const void* k, const void* v,
                         int64_t num_tokens, void* stream) {
    CallRange range("pkv_kv_append");
    pkv_status st = check_pool(pool);
    if (st != PKV_OK) return st;
    if (num_tokens < 0) return PKV_ERR_INVALID;
    if (num_tokens == 0) return PKV_OK;
    if (!k_pool || !v_pool || !slot_mapping || !k || !v) return PKV_ERR_INVALID;
    if (!aligned16(k_pool) || !aligned16(v_pool) || !aligned16(k) || !aligned16(v))
        return PKV_ERR_INVALID;
    int* status = status_word();
    if (!status) return PKV_ERR_CUDA;
    const int row_bytes = pool->head_dim * elem_bytes(pool->dtype);
    return from_cuda(pkv::launch_kv_append(k_pool, v_pool, slot_mapping, k, v, num_tokens,
                                           pool->num_kv_heads, row_bytes, pool->block_size,
                                           pool->num_blocks, status,
                                           static_cast<cudaStream_t>(stream)));
}

int pkv_paged_decode_auto_partition(int num_seqs, int num_q_heads, int max_context,
                                    int block_size) {
    if (num_seqs <= 0 || num_q_heads <= 0 || max_context <= 0 || chunk_shift(block_size) < 0)
        return 0;
    return auto_partition(num_seqs, num_q_heads, max_context, block_size);
}

size_t pkv_paged_decode_workspace_bytes(int num_seqs, int num_q_heads, int head_dim,
                                        int max_context, int block_size, int partition_blocks) {
    if (num_seqs <= 0 || num_q_heads <= 0 || head_dim <= 0 || max_context <= 0 ||
        chunk_shift(block_size) < 0 || partition_blocks < 0)
        return 0;
    const int pb = partition_blocks ? partition_blocks
                                    : auto_partition(num_seqs, num_q_heads, max_context, block_size);
    const int max_parts = ceil_div(ceil_div(max_context, block_size), pb);
    return decode_workspace(num_seqs, num_q_heads, head_dim, max_parts);
}

namespace {

// pkv_paged_decode, and with k_new / v_new set pkv_paged_decode_append.
pkv_status decode_impl(const pkv_pool_desc* pool, void* out, const void* q, const void* k_pool,
                       const void* v_pool, const int32_t* block_tables, int max_blocks_per_seq,
                       const int32_t* context_lens, int max_context, int num_seqs,
                       int num_q_heads, float scale, int partition_blocks, void* workspace,
                       size_t workspace_bytes, const void* k_new, const void* v_new,
                       void* stream) {
    pkv_status st = check_pool(pool);
    if (st != PKV_OK) return st;
    if (num_seqs < 0 || num_q_heads <= 0 || partition_blocks < 0) return PKV_ERR_INVALID;
    if (num_seqs == 0) return PKV_OK;
    if (!out || !q || !k_pool || !v_pool || !block_tables || !context_lens)
        return PKV_ERR_INVALID;
    const int B = pool->block_size;
    if (max_blocks_per_seq <= 0 || max_context <= 0 ||
        static_cast<int64_t>(max_context) > static_cast<int64_t>(max_blocks_per_seq) * B)
        return PKV_ERR_INVALID;
    if (num_q_heads % pool->num_kv_heads != 0) return PKV_ERR_INVALID;
    const int group = num_q_heads / pool->num_kv_heads;
    if (group != 1 && group != 2 && group != 4 && group != 8) return PKV_ERR_UNSUPPORTED;
    if (num_seqs > 65535) return PKV_ERR_UNSUPPORTED;
    if (!aligned16(out) || !aligned16(q) || !aligned16(k_pool) || !aligned16(v_pool))
        return PKV_ERR_INVALID;

    const int pb = partition_blocks ? partition_blocks
                                    : auto_partition(num_seqs, num_q_heads, max_context, B);
    const int max_parts = ceil_div(ceil_div(max_context, B), pb);
    if (max_parts > pkv::kMaxParts) return PKV_ERR_UNSUPPORTED;
    const size_t need = decode_workspace(num_seqs, num_q_heads, pool->head_dim, max_parts);
    if (need > 0 && (!workspace || workspace_bytes < need || !aligned16(workspace)))
        return PKV_ERR_NOMEM;
    int* status = status_word();
    if (!status) return PKV_ERR_CUDA;

    pkv::DecodeArgs a{};
    a.out = out;
    a.q = q;
    a.k_pool = k_pool;
    a.v_pool = v_pool;
    a.block_tables = block_tables;
    a.context_lens = context_lens;
    a.status = status;
    a.num_blocks = pool->num_blocks;
    a.max_blocks_per_seq = max_blocks_per_seq;
    a.num_seqs = num_seqs;
    a.num_q_heads = num_q_heads;
    a.num_kv_heads = pool->num_kv_heads;
    a.chunk_shift = chunk_shift(B);
    a.partition_chunks = pb << a.chunk_shift;
    a.max_parts = max_parts;
    a.scale_log2 = static_cast<float>(static_cast<double>(scale) * kLog2e);
    a.k_new = k_new;
    a.v_new = v_new;
    if (need > 0) {
        const size_t rows = static_cast<size_t>(num_seqs) * num_q_heads * max_parts;
        const size_t ml = (rows * sizeof(float) + 15) / 16 * 16;
        char* w = static_cast<char*>(workspace);
        a.o_part = reinterpret_cast<float*>(w);
        a.m_part = reinterpret_cast<float*>(w + rows * pool->head_dim * sizeof(float));
        a.l_part = reinterpret_cast<float*>(w + rows * pool->head_dim * sizeof(float) + ml);
    }
    const cudaStream_t st_ = static_cast<cudaStream_t>(stream);
    a.test_stall = decode_test_stall();
    if (pool->dtype == PKV_BF16 && !decode_use_simt())
        return from_cuda(pkv::launch_paged_decode_tc(a, pool->head_dim, group, st_));
    return from_cuda(pkv::launch_paged_decode(a, pool->dtype, pool->head_dim, group, st_));
}

}  // namespace

pkv_status pkv_paged_decode(const pkv_pool_desc* pool, void* out, const void* q,
                            const void* k_pool, const void* v_pool,
                            const int32_t* block_tables, int max_blocks_per_seq,
                            const int32_t* context_lens, int max_context, int num_seqs,
                            int num_q_heads, float scale, int partition_blocks,
                            void* workspace, size_t workspace_bytes, void* stream) {
    CallRange range("pkv_paged_decode");
    return decode_impl(pool, out, q, k_pool, v_pool, block_tables, max_blocks_per_seq,
                       context_lens, max_context, num_seqs, num_q_heads, scale,
                       partition_blocks, workspace, workspace_bytes, nullptr, nullptr, stream);
}

pkv_status pkv_paged_decode_append(const pkv_pool_desc* pool, void* out, const void* q,
                                   void* k_pool, void* v_pool, const void* k_new,
                                   const void* v_new, const int32_t* block_tables,
                                   int max_blocks_per_seq, const int32_t* context_lens,
                                   int max_context, int num_seqs, int num_q_heads, float scale,
                                   int partition_blocks, void* workspace, size_t workspace_bytes,
                                   void* stream) {
    CallRange range("pkv_paged_decode_append");
    if (num_seqs > 0 && (!k_new || !v_new || !aligned16(k_new) || !aligned16(v_new)))
        return PKV_ERR_INVALID;
    return decode_impl(pool, out, q, k_pool, v_pool, block_tables, max_blocks_per_seq,
                       context_lens, max_context, num_seqs, num_q_heads, scale,
                       partition_blocks, workspace, workspace_bytes, k_new, v_new, stream);
}

namespace {

uint64_t round256(uint64_t x) { return (x + 255) / 256 * 256; }

// The address through which kernels reach host memory `p` in place, or nullptr.
// Page-locked memory from cudaHostAlloc / cudaMallocHost / cudaHostRegister is mapped
// into the device address space under unified addressing (on a Grace-Blackwell node
// the GPU then reads and writes it over NVLink-C2C); pageable memory is not.
void* mapped_host_ptr(const void* p) {
    cudaPointerAttributes a{};
    if (cudaPointerGetAttributes(&a, p) != cudaSuccess) {
        cudaGetLastError();   // a failed query is left as the last error: clear it
        return nullptr;
    }
    return a.type == cudaMemoryTypeHost ? a.devicePointer : nullptr;
}

}  // namespace

pkv_status pkv_decode_step_layout(const pkv_pool_desc* pool, int num_seqs, int num_q_heads,
                                  int max_blocks_per_seq, pkv_step_layout* layout) {
    pkv_status st = check_pool(pool);
    if (st != PKV_OK) return st;
    if (!layout || num_seqs < 0 || num_q_heads <= 0 || max_blocks_per_seq <= 0)
        return PKV_ERR_INVALID;
    const uint64_t row = static_cast<uint64_t>(pool->head_dim) * elem_bytes(pool->dtype);
    const uint64_t S = static_cast<uint64_t>(num_seqs);
    uint64_t off = 0;
    layout->q = off;
    off = round256(off + S * num_q_heads * row);
    layout->k_new = off;
    off = round256(off + S * pool->num_kv_heads * row);
    layout->v_new = off;
    off = round256(off + S * pool->num_kv_heads * row);
    layout->block_tables = off;
    off = round256(off + S * max_blocks_per_seq * sizeof(int32_t));
    layout->context_lens = off;
    off = round256(off + S * sizeof(int32_t));
    layout->bytes = off;
    return PKV_OK;
}

size_t pkv_paged_decode_append_host_staging_bytes(const pkv_pool_desc* pool, int num_seqs,
                                                  int num_q_heads, int max_blocks_per_seq,
                                                  int max_context, int partition_blocks) {
    pkv_step_layout l;
    if (pkv_decode_step_layout(pool, num_seqs, num_q_heads, max_blocks_per_seq, &l) != PKV_OK ||
        num_seqs <= 0 || max_context <= 0 || partition_blocks < 0)
        return 0;
    const uint64_t out = round256(static_cast<uint64_t>(num_seqs) * num_q_heads *
                                  pool->head_dim * elem_bytes(pool->dtype));
    return l.bytes + out +
           pkv_paged_decode_workspace_bytes(num_seqs, num_q_heads, pool->head_dim, max_context,
                                            pool->block_size, partition_blocks);
}

pkv_status pkv_paged_decode_append_host(const pkv_pool_desc* pool, void* k_pool, void* v_pool,
                                        const void* host_in, void* host_out,
                                        int max_blocks_per_seq, int max_context, int num_seqs,
                                        int num_q_heads, float scale, int partition_blocks,
                                        void* staging, size_t staging_bytes, void* stream) {
    CallRange range("pkv_paged_decode_append_host");
    pkv_step_layout l;
    pkv_status st = pkv_decode_step_layout(pool, num_seqs, num_q_heads, max_blocks_per_seq, &l);
    if (st != PKV_OK) return st;
    if (num_seqs == 0) return PKV_OK;
    if (!host_in || !host_out || !staging || (reinterpret_cast<uintptr_t>(staging) & 255u))
        return PKV_ERR_INVALID;
    if (max_context <= 0 || partition_blocks < 0) return PKV_ERR_INVALID;
    const size_t need = pkv_paged_decode_append_host_staging_bytes(
        pool, num_seqs, num_q_heads, max_blocks_per_seq, max_context, partition_blocks);
    if (need == 0) return PKV_ERR_INVALID;
    if (staging_bytes < need) return PKV_ERR_NOMEM;
    const uint64_t out_bytes = static_cast<uint64_t>(num_seqs) * num_q_heads * pool->head_dim *
                               elem_bytes(pool->dtype);
    char* dev = static_cast<char*>(staging);
    char* out = dev + l.bytes;
    char* ws = out + round256(out_bytes);
    const cudaStream_t st_ = static_cast<cudaStream_t>(stream);
    // Mapped (page-locked) host buffers are read and written by the kernels in place;
    // any other host memory, or a buffer not 16-byte aligned (the kernels' vector
    // accesses need that), goes through the staging buffer with one copy each way.
    const char* in = static_cast<const char*>(mapped_host_ptr(host_in));
    char* out_map = static_cast<char*>(mapped_host_ptr(host_out));
    if (!aligned16(in)) in = nullptr;
    if (!aligned16(out_map)) out_map = nullptr;
    if (!in) {
        if (cudaMemcpyAsync(dev, host_in, l.bytes, cudaMemcpyHostToDevice, st_) != cudaSuccess)
            return PKV_ERR_CUDA;
        in = dev;
    }
    st = pkv_paged_decode_append(pool, out_map ? out_map : out, in + l.q, k_pool, v_pool,
                                 in + l.k_new, in + l.v_new,
                                 reinterpret_cast<const int32_t*>(in + l.block_tables),
                                 max_blocks_per_seq,
                                 reinterpret_cast<const int32_t*>(in + l.context_lens),
                                 max_context, num_seqs, num_q_heads, scale, partition_blocks, ws,
                                 need - (ws - dev), stream);
    if (st != PKV_OK || out_map) return st;
    return from_cuda(cudaMemcpyAsync(host_out, out, out_bytes, cudaMemcpyDeviceToHost, st_));
}

pkv_status pkv_paged_decode_noalloc(const pkv_pool_desc* pool, void* out, const void* q,
                                    const void* k_pool, const void* v_pool,
                                    const int32_t* block_tables, int max_blocks_per_seq,
                                    const int32_t* context_lens, int max_context, int num_seqs,
                                    int num_q_heads, float scale, int partition_blocks,
                                    void* stream) {
    CallRange range("pkv_paged_decode_noalloc");
    pkv_status st = check_pool(pool);
    if (st != PKV_OK) return st;
    if (num_seqs < 0 || num_q_heads <= 0 || partition_blocks < 0 || max_context <= 0)
        return PKV_ERR_INVALID;
    if (num_seqs == 0) return PKV_OK;
    const size_t need = pkv_paged_decode_workspace_bytes(
        num_seqs, num_q_heads, pool->head_dim, max_context, pool->block_size, partition_blocks);
    if (need > kNoAllocScratchBytes) return PKV_ERR_NOMEM;
    void* scratch = nullptr;
    if (need > 0) {
        scratch = noalloc_scratch();
        if (!scratch) return PKV_ERR_CUDA;
    }
    return pkv_paged_decode(pool, out, q, k_pool, v_pool, block_tables, max_blocks_per_seq,
                            context_lens, max_context, num_seqs, num_q_heads, scale,
                            partition_blocks, scratch, need, stream);
}

namespace {

// Splits of the cascade decode's prefix pass over its 128-key tiles.  The pass has about
// ceil(S * Hq / 128) CTAs (query tiles times kv heads), each needing a whole SM, and runs
// beside the suffix decode, which is HBM-bound and wants the other SMs: its tiles are
// divided among as many CTAs per query tile (up to 8, none empty) as keep the pass within
// half the SMs (76).  On the shared-prefix batch (64 query tiles) 1, 2, 3 and 4 splits
// measured 113, 121, 125 and 128 us.  Depends only on (num_seqs, num_q_heads, prefix_len).
int cascade_splits(int num_seqs, int num_q_heads, int prefix_len, int* tiles_per_split) {
    const int tiles = ceil_div(prefix_len, 128);
    const int ctas = ceil_div(static_cast<int64_t>(num_seqs) * num_q_heads, 128);
    int ns = 76 / ctas;
    ns = std::max(1, std::min(ns, std::min(8, tiles)));
    const int tps = ceil_div(tiles, ns);
    *tiles_per_split = tps;
    return ceil_div(tiles, tps);
}

}  // namespace

size_t pkv_paged_decode_cascade_workspace_bytes(int num_seqs, int num_q_heads, int head_dim,
                                                int prefix_len, int max_context, int block_size,
                                                int partition_blocks) {
    if (num_seqs <= 0 || num_q_heads <= 0 || head_dim <= 0 || prefix_len <= 0 ||
        max_context < prefix_len || chunk_shift(block_size) < 0 || partition_blocks < 0)
        return 0;
    const int suffix = max_context - prefix_len;
    const int pb = partition_blocks
                       ? partition_blocks
                       : (suffix > 0 ? auto_partition(num_seqs, num_q_heads, suffix, block_size) : 1);
    const int parts = suffix > 0 ? ceil_div(ceil_div(suffix, block_size), pb) : 0;
    int tps = 0;
    const int ns = cascade_splits(num_seqs, num_q_heads, prefix_len, &tps);
    const size_t rows = static_cast<size_t>(num_seqs) * num_q_heads * (parts + ns);
    const size_t ml = (rows * sizeof(float) + 15) / 16 * 16;
    return rows * head_dim * sizeof(float) + 2 * ml;
}

namespace {

// pkv_paged_decode_cascade, and with k_new / v_new set pkv_paged_decode_cascade_append
// (the suffix decode stores and attends each sequence's newest token).
pkv_status cascade_impl(const pkv_pool_desc* pool, void* out, const void* q, const void* k_pool,
                        const void* v_pool, const int32_t* prefix_blocks, int prefix_len,
                        const int32_t* block_tables, int max_blocks_per_seq,
                        const int32_t* context_lens, int max_context, int num_seqs,
                        int num_q_heads, float scale, int partition_blocks, void* workspace,
                        size_t workspace_bytes, const void* k_new, const void* v_new,
                        void* stream) {
    pkv_status st = check_pool(pool);
    if (st != PKV_OK) return st;
    if (num_seqs < 0 || num_q_heads <= 0 || partition_blocks < 0 || !(scale > 0.f))
        return PKV_ERR_INVALID;
    if (num_seqs == 0) return PKV_OK;
    if (!out || !q || !k_pool || !v_pool || !prefix_blocks || !block_tables || !context_lens)
        return PKV_ERR_INVALID;
    const int B = pool->block_size;
    if (prefix_len <= 0 || prefix_len % B != 0 || max_context < prefix_len ||
        max_blocks_per_seq <= 0 ||
        static_cast<int64_t>(max_context) > static_cast<int64_t>(max_blocks_per_seq) * B)
        return PKV_ERR_INVALID;
    if (num_q_heads % pool->num_kv_heads != 0) return PKV_ERR_INVALID;
    const int group = num_q_heads / pool->num_kv_heads;
    if (pool->dtype != PKV_BF16) return PKV_ERR_UNSUPPORTED;
    if (group != 1 && group != 2 && group != 4 && group != 8) return PKV_ERR_UNSUPPORTED;
    if (num_seqs > 65535) return PKV_ERR_UNSUPPORTED;
    if (!aligned16(out) || !aligned16(q) || !aligned16(k_pool) || !aligned16(v_pool))
        return PKV_ERR_INVALID;
    const int suffix = max_context - prefix_len;
    const int pb = partition_blocks
                       ? partition_blocks
                       : (suffix > 0 ? auto_partition(num_seqs, num_q_heads, suffix, B) : 1);
    const int parts = suffix > 0 ? ceil_div(ceil_div(suffix, B), pb) : 0;
    int tps = 0;
    const int ns = cascade_splits(num_seqs, num_q_heads, prefix_len, &tps);
    if (parts + ns > pkv::kMaxParts) return PKV_ERR_UNSUPPORTED;
    const size_t need = pkv_paged_decode_cascade_workspace_bytes(
        num_seqs, num_q_heads, pool->head_dim, prefix_len, max_context, B, partition_blocks);
    if (!workspace || workspace_bytes < need || !aligned16(workspace)) return PKV_ERR_NOMEM;
    int* status = status_word();
    if (!status) return PKV_ERR_CUDA;
    const size_t rows = static_cast<size_t>(num_seqs) * num_q_heads * (parts + ns);
    const size_t ml = (rows * sizeof(float) + 15) / 16 * 16;
    char* w = static_cast<char*>(workspace);
    float* o_part = reinterpret_cast<float*>(w);
    float* m_part = reinterpret_cast<float*>(w + rows * pool->head_dim * sizeof(float));
    float* l_part = reinterpret_cast<float*>(w + rows * pool->head_dim * sizeof(float) + ml);
    const float sl2 = static_cast<float>(static_cast<double>(scale) * kLog2e);
    const cudaStream_t st_ = static_cast<cudaStream_t>(stream);

    // 1. every sequence's query heads against the shared prefix, on the tensor cores
    pkv::PrefillArgs pa{};
    pa.head_dim = pool->head_dim;
    pa.block_size = B;
    pa.q = q;
    pa.k_pool = k_pool;
    pa.v_pool = v_pool;
    pa.block_tables = prefix_blocks;
    pa.status = status;
    pa.num_blocks = pool->num_blocks;
    pa.max_blocks_per_seq = prefix_len / B;
    pa.num_reqs = ns;   // grid z: one per split of the prefix's tiles
    pa.total_new = num_seqs;
    pa.max_new = num_seqs;
    pa.num_q_heads = num_q_heads;
    pa.num_kv_heads = pool->num_kv_heads;
    pa.scale_log2 = sl2;
    pa.cascade = 1;
    pa.cascade_keys = prefix_len;
    pa.cascade_rows = num_seqs;
    pa.cascade_tiles_per_split = tps;
    pa.max_parts_total = parts + ns;
    pa.p_single_min_keys = prefill_p_single_min_keys();
    pa.o_part = o_part;
    pa.m_part = m_part;
    pa.l_part = l_part;
    // The prefix pass (tensor-bound, its K/V L2-resident) runs on a side stream beside
    // the suffix decode (HBM-bound); the combine waits for both.
    cudaStream_t side = side_stream();
    if (!side) return PKV_ERR_CUDA;
    cudaEvent_t fork = nullptr, join = nullptr;
    if (cudaEventCreateWithFlags(&fork, cudaEventDisableTiming) != cudaSuccess)
        return PKV_ERR_CUDA;
    if (cudaEventCreateWithFlags(&join, cudaEventDisableTiming) != cudaSuccess) {
        cudaEventDestroy(fork);
        return PKV_ERR_CUDA;
    }
    struct Events {   // released once their work completes
        cudaEvent_t a, b;
        ~Events() { cudaEventDestroy(a); cudaEventDestroy(b); }
    } ev{fork, join};
    if (cudaEventRecord(fork, st_) != cudaSuccess || cudaStreamWaitEvent(side, fork, 0) != cudaSuccess)
        return PKV_ERR_CUDA;
    // From here on the side stream carries this call's work: every exit, the error
    // returns included, makes the caller's stream wait for it, so that no work of the call
    // runs on past its return unordered with the caller's stream, and a stream capture
    // ends with the side stream joined back.
    struct Rejoin {
        cudaStream_t side, st;
        cudaEvent_t ev;
        bool recorded = false, waited = false;
        cudaError_t record() {
            recorded = true;
            return cudaEventRecord(ev, side);
        }
        cudaError_t wait() {
            cudaError_t e = recorded ? cudaSuccess : record();
            waited = true;
            const cudaError_t w = cudaStreamWaitEvent(st, ev, 0);
            return e != cudaSuccess ? e : w;
        }
        ~Rejoin() {
            if (!waited) wait();
        }
    } rejoin{side, st_, join};
    cudaError_t e = pkv::launch_paged_prefill(pa, group, side);
    if (e != cudaSuccess) return e == cudaErrorNotSupported ? PKV_ERR_UNSUPPORTED : PKV_ERR_CUDA;
    if (rejoin.record() != cudaSuccess) return PKV_ERR_CUDA;

    // 2. private suffixes (blocks from prefix_len / B on) + 3. log-sum-exp merge
    pkv::DecodeArgs a{};
    a.out = out;
    a.q = q;
    a.k_pool = k_pool;
    a.v_pool = v_pool;
    a.block_tables = block_tables;
    a.context_lens = context_lens;
    a.status = status;
    a.num_blocks = pool->num_blocks;
    a.max_blocks_per_seq = max_blocks_per_seq;
    a.num_seqs = num_seqs;
    a.num_q_heads = num_q_heads;
    a.num_kv_heads = pool->num_kv_heads;
    a.chunk_shift = chunk_shift(B);
    a.partition_chunks = pb << a.chunk_shift;
    a.max_parts = parts;
    a.scale_log2 = sl2;
    a.o_part = o_part;
    a.m_part = m_part;
    a.l_part = l_part;
    a.chunk_offset = prefix_len / kChunk;
    a.extra_parts = ns;
    a.defer_combine = 1;
    a.no_pdl = 1;
    a.k_new = k_new;
    a.v_new = v_new;
    if (cascade_test_fail_suffix()) return PKV_ERR_CUDA;   // test hook: the rejoin still runs
    e = decode_use_simt() ? pkv::launch_paged_decode(a, pool->dtype, pool->head_dim, group, st_)
                          : pkv::launch_paged_decode_tc(a, pool->head_dim, group, st_);
    if (e != cudaSuccess) return e == cudaErrorNotSupported ? PKV_ERR_UNSUPPORTED : PKV_ERR_CUDA;
    if (rejoin.wait() != cudaSuccess) return PKV_ERR_CUDA;
    return from_cuda(pkv::launch_decode_combine(a, pool->dtype, pool->head_dim, st_));
}

}  // namespace

pkv_status pkv_paged_decode_cascade(const pkv_pool_desc* pool, void* out, const void* q,
                                    const void* k_pool, const void* v_pool,
                                    const int32_t* prefix_blocks, int prefix_len,
                                    const int32_t* block_tables, int max_blocks_per_seq,
                                    const int32_t* context_lens, int max_context, int num_seqs,
                                    int num_q_heads, float scale, int partition_blocks,
                                    void* workspace, size_t workspace_bytes, void* stream) {
    CallRange range("pkv_paged_decode_cascade");
    return cascade_impl(pool, out, q, k_pool, v_pool, prefix_blocks, prefix_len, block_tables,
                        max_blocks_per_seq, context_lens, max_context, num_seqs, num_q_heads,
                        scale, partition_blocks, workspace, workspace_bytes, nullptr, nullptr,
                        stream);
}

pkv_status pkv_paged_decode_cascade_append(const pkv_pool_desc* pool, void* out, const void* q,
                                           void* k_pool, void* v_pool, const void* k_new,
                                           const void* v_new, const int32_t* prefix_blocks,
                                           int prefix_len, const int32_t* block_tables,
                                           int max_blocks_per_seq, const int32_t* context_lens,
                                           int max_context, int num_seqs, int num_q_heads,
                                           float scale, int partition_blocks, void* workspace,
                                           size_t workspace_bytes, void* stream) {
    CallRange range("pkv_paged_decode_cascade_append");
    if (num_seqs > 0 && (!k_new || !v_new || !aligned16(k_new) || !aligned16(v_new)))
        return PKV_ERR_INVALID;
    return cascade_impl(pool, out, q, k_pool, v_pool, prefix_blocks, prefix_len, block_tables,
                        max_blocks_per_seq, context_lens, max_context, num_seqs, num_q_heads,
                        scale, partition_blocks, workspace, workspace_bytes, k_new, v_new,
                        stream);
}

pkv_status pkv_paged_prefill(const pkv_pool_desc* pool, void* out, const void* q,
                             const void* k_pool, const void* v_pool,
                             const int32_t* block_tables, int max_blocks_per_seq,
                             const int32_t* cached_lens, const int32_t* new_lens,
                             const int32_t* q_offsets, int num_reqs, int total_new, int max_new,
                             int num_q_heads, float scale, void* stream) {
    CallRange range("pkv_paged_prefill");
    pkv_status st = check_pool(pool);
    if (st != PKV_OK) return st;
    if (num_reqs < 0 || total_new < 0 || max_new < 0 || num_q_heads <= 0 || !(scale > 0.f))
        return PKV_ERR_INVALID;
    if (num_reqs == 0 || total_new == 0 || max_new == 0) return PKV_OK;
    if (!out || !q || !k_pool || !v_pool || !block_tables || !cached_lens || !new_lens ||
        !q_offsets || max_blocks_per_seq <= 0)
        return PKV_ERR_INVALID;
    if (num_q_heads % pool->num_kv_heads != 0) return PKV_ERR_INVALID;
    const int group = num_q_heads / pool->num_kv_heads;
    if (group != 1 && group != 2 && group != 4 && group != 8) return PKV_ERR_UNSUPPORTED;
    if (num_reqs > 65535) return PKV_ERR_UNSUPPORTED;
    if (!aligned16(out) || !aligned16(q) || !aligned16(k_pool) || !aligned16(v_pool))
        return PKV_ERR_INVALID;
    int* status = status_word();
    if (!status) return PKV_ERR_CUDA;
    pkv::PrefillArgs a{};
    a.head_dim = pool->head_dim;
    a.block_size = pool->block_size;
    a.out = out;
    a.q = q;
    a.k_pool = k_pool;
    a.v_pool = v_pool;
    a.block_tables = block_tables;
    a.cached_lens = cached_lens;
    a.new_lens = new_lens;
    a.q_offsets = q_offsets;
    a.status = status;
    a.num_blocks = pool->num_blocks;
    a.max_blocks_per_seq = max_blocks_per_seq;
    a.num_reqs = num_reqs;
    a.total_new = total_new;
    a.max_new = max_new;
    a.num_q_heads = num_q_heads;
    a.num_kv_heads = pool->num_kv_heads;
    a.scale_log2 = static_cast<float>(static_cast<double>(scale) * kLog2e);
    a.p_single_min_keys = prefill_p_single_min_keys();
    // fp32 pools run on the CUDA cores: the tensor cores would round fp32 operands to tf32.
    const cudaError_t e =
        pool->dtype == PKV_F32
            ? pkv::launch_paged_prefill_f32(a, group, static_cast<cudaStream_t>(stream))
            : pkv::launch_paged_prefill(a, group, static_cast<cudaStream_t>(stream));
    if (e == cudaErrorNotSupported) return PKV_ERR_UNSUPPORTED;
    return from_cuda(e);
}

pkv_status pkv_prefill_step_layout(const pkv_pool_desc* pool, int num_reqs, int total_new,
                                   int num_q_heads, int max_blocks_per_seq,
                                   pkv_prefill_layout* layout) {
    pkv_status st = check_pool(pool);
    if (st != PKV_OK) return st;
    if (!layout || num_reqs < 0 || total_new < 0 || num_q_heads <= 0 || max_blocks_per_seq <= 0)
        return PKV_ERR_INVALID;
    const uint64_t row = static_cast<uint64_t>(pool->head_dim) * elem_bytes(pool->dtype);
    const uint64_t R = static_cast<uint64_t>(num_reqs);
    const uint64_t T = static_cast<uint64_t>(total_new);
    uint64_t off = 0;
    layout->q = off;
    off = round256(off + T * num_q_heads * row);
    layout->block_tables = off;
    off = round256(off + R * max_blocks_per_seq * sizeof(int32_t));
    layout->cached_lens = off;
    off = round256(off + R * sizeof(int32_t));
    layout->new_lens = off;
    off = round256(off + R * sizeof(int32_t));
    layout->q_offsets = off;
    off = round256(off + (R + 1) * sizeof(int32_t));
    layout->copied_bytes = off;
    layout->k_new = off;
    off = round256(off + T * pool->num_kv_heads * row);
    layout->v_new = off;
    off = round256(off + T * pool->num_kv_heads * row);
    layout->slot_mapping = off;
    off = round256(off + T * sizeof(int64_t));
    layout->bytes = off;
    return PKV_OK;
}

size_t pkv_paged_prefill_append_host_staging_bytes(const pkv_pool_desc* pool, int num_reqs,
                                                   int total_new, int num_q_heads,
                                                   int max_blocks_per_seq) {
    pkv_prefill_layout l;
    if (pkv_prefill_step_layout(pool, num_reqs, total_new, num_q_heads, max_blocks_per_seq,
                                &l) != PKV_OK)
        return 0;
    const uint64_t out = round256(static_cast<uint64_t>(total_new) * num_q_heads *
                                  pool->head_dim * elem_bytes(pool->dtype));
    return l.bytes + out;
}

pkv_status pkv_paged_prefill_append_host(const pkv_pool_desc* pool, void* k_pool, void* v_pool,
                                         const void* host_in, void* host_out, int num_reqs,
                                         int total_new, int max_new, int num_q_heads,
                                         int max_blocks_per_seq, float scale, void* staging,
                                         size_t staging_bytes, void* stream) {
    CallRange range("pkv_paged_prefill_append_host");
    pkv_prefill_layout l;
    pkv_status st =
        pkv_prefill_step_layout(pool, num_reqs, total_new, num_q_heads, max_blocks_per_seq, &l);
    if (st != PKV_OK) return st;
    if (num_reqs == 0 || total_new == 0) return PKV_OK;
    if (!host_in || !host_out || !staging || (reinterpret_cast<uintptr_t>(staging) & 255u))
        return PKV_ERR_INVALID;
    const size_t need = pkv_paged_prefill_append_host_staging_bytes(
        pool, num_reqs, total_new, num_q_heads, max_blocks_per_seq);
    if (need == 0) return PKV_ERR_INVALID;
    if (staging_bytes < need) return PKV_ERR_NOMEM;
    const char* hin = static_cast<const char*>(host_in);
    const int32_t* qoff = reinterpret_cast<const int32_t*>(hin + l.q_offsets);
    if (qoff[0] != 0 || qoff[num_reqs] != total_new) return PKV_ERR_INVALID;
    for (int r = 0; r < num_reqs; ++r)
        if (qoff[r + 1] < qoff[r]) return PKV_ERR_INVALID;
    char* dev = static_cast<char*>(staging);
    char* out = dev + l.bytes;
    const uint64_t esz = elem_bytes(pool->dtype);
    const uint64_t qrow = static_cast<uint64_t>(num_q_heads) * pool->head_dim * esz;
    const uint64_t kvrow = static_cast<uint64_t>(pool->num_kv_heads) * pool->head_dim * esz;
    const cudaStream_t st_ = static_cast<cudaStream_t>(stream);
    // Every input goes to the device by copy (the prefill loads q by TMA) and the output
    // comes back by copy, chunk by chunk, on two library streams beside the kernels.  On
    // the 16 x 512-token batch the link moves about 200 GB/s each way, whether copy
    // engines or SMs drive it; read in place by the append kernel, the new rows cost
    // more on the kernels' stream than their copy does beside it, and stored in place the
    // prefill's output tiles held the kernel up (1.23 -> 1.87 ms a step unchunked).
    // Requests in up to kChunks chunks of about equal new rows: chunk c's query rows are
    // copied in on one copy stream while chunk c - 1's append and prefill run on `stream`
    // and chunk c - 2's output is copied back on the other.
    constexpr int kChunks = 4;
    int bounds[kChunks + 1];
    int nch = 0;
    bounds[0] = 0;
    for (int c = 1; c <= kChunks && bounds[nch] < num_reqs; ++c) {
        const int64_t target = static_cast<int64_t>(total_new) * c / kChunks;
        int r = bounds[nch] + 1;
        while (r < num_reqs && qoff[r] < target) ++r;
        if (c == kChunks) r = num_reqs;
        bounds[++nch] = r;
    }
    cudaStream_t cin = copy_stream(0), cout = copy_stream(1);
    if (!cin || !cout) return PKV_ERR_CUDA;
    struct Events {   // the fork, two per chunk and the two joins
        cudaEvent_t e[2 * kChunks + 3] = {};
        int n = 0;
        cudaEvent_t make() {
            cudaEvent_t ev = nullptr;
            if (n < 2 * kChunks + 3 &&
                cudaEventCreateWithFlags(&ev, cudaEventDisableTiming) == cudaSuccess)
                e[n++] = ev;
            return ev;
        }
        ~Events() {   // released once their work completes
            for (int i = 0; i < n; ++i) cudaEventDestroy(e[i]);
        }
    } ev;
    cudaEvent_t fork = ev.make();
    if (!fork || cudaEventRecord(fork, st_) != cudaSuccess ||
        cudaStreamWaitEvent(cin, fork, 0) != cudaSuccess ||
        cudaStreamWaitEvent(cout, fork, 0) != cudaSuccess)
        return PKV_ERR_CUDA;
    // From here on the copy streams carry this call's work: every exit makes `stream` wait
    // for both, so that nothing of the call runs on past it unordered and a stream capture
    // ends with them joined.
    struct Rejoin {
        cudaStream_t a, b, st;
        Events* ev;
        ~Rejoin() {
            for (cudaStream_t s : {a, b}) {
                cudaEvent_t j = ev->make();
                if (j && cudaEventRecord(j, s) == cudaSuccess) cudaStreamWaitEvent(st, j, 0);
            }
        }
    } rejoin{cin, cout, st_, &ev};
    // the control arrays, then chunk by chunk q, the new rows and their slots
    if (cudaMemcpyAsync(dev + l.block_tables, hin + l.block_tables,
                        l.copied_bytes - l.block_tables, cudaMemcpyHostToDevice, cin) != cudaSuccess)
        return PKV_ERR_CUDA;
    cudaEvent_t in_done[kChunks];
    for (int c = 0; c < nch; ++c) {
        const uint64_t t0 = qoff[bounds[c]], t1 = qoff[bounds[c + 1]];
        const struct { uint64_t off, row; } parts[4] = {
            {l.q, qrow}, {l.k_new, kvrow}, {l.v_new, kvrow}, {l.slot_mapping, sizeof(int64_t)}};
        for (const auto& pt : parts)
            if (t1 > t0 && cudaMemcpyAsync(dev + pt.off + t0 * pt.row, hin + pt.off + t0 * pt.row,
                                           (t1 - t0) * pt.row, cudaMemcpyHostToDevice,
                                           cin) != cudaSuccess)
                return PKV_ERR_CUDA;
        in_done[c] = ev.make();
        if (!in_done[c] || cudaEventRecord(in_done[c], cin) != cudaSuccess) return PKV_ERR_CUDA;
    }
    const int32_t* dbt = reinterpret_cast<const int32_t*>(dev + l.block_tables);
    const int32_t* dcl = reinterpret_cast<const int32_t*>(dev + l.cached_lens);
    const int32_t* dnl = reinterpret_cast<const int32_t*>(dev + l.new_lens);
    const int32_t* dqo = reinterpret_cast<const int32_t*>(dev + l.q_offsets);
    const char* rows = dev;
    const int64_t* slots = reinterpret_cast<const int64_t*>(rows + l.slot_mapping);
    for (int c = 0; c < nch; ++c) {
        const int r0 = bounds[c], r1 = bounds[c + 1];
        const int64_t t0 = qoff[r0], t1 = qoff[r1];
        if (cudaStreamWaitEvent(st_, in_done[c], 0) != cudaSuccess) return PKV_ERR_CUDA;
        st = pkv_kv_append(pool, k_pool, v_pool, slots + t0, rows + l.k_new + t0 * kvrow,
                           rows + l.v_new + t0 * kvrow, t1 - t0, stream);
        if (st != PKV_OK) return st;
        // the chunk's requests; q_offsets stay absolute rows of the whole q and out
        st = pkv_paged_prefill(pool, out, dev + l.q, k_pool, v_pool,
                               dbt + static_cast<size_t>(r0) * max_blocks_per_seq,
                               max_blocks_per_seq, dcl + r0, dnl + r0, dqo + r0, r1 - r0,
                               total_new, max_new, num_q_heads, scale, stream);
        if (st != PKV_OK) return st;
        cudaEvent_t done = ev.make();
        if (!done || cudaEventRecord(done, st_) != cudaSuccess ||
            cudaStreamWaitEvent(cout, done, 0) != cudaSuccess)
            return PKV_ERR_CUDA;
        if (t1 > t0 && cudaMemcpyAsync(static_cast<char*>(host_out) + t0 * qrow, out + t0 * qrow,
                                       (t1 - t0) * qrow, cudaMemcpyDeviceToHost, cout) != cudaSuccess)
            return PKV_ERR_CUDA;
    }
    return PKV_OK;
}

pkv_status pkv_copy_blocks(const pkv_pool_desc* pool, void* k_pool, void* v_pool,
                           const int32_t* pairs, int num_pairs, void* stream) {
    CallRange range("pkv_copy_blocks");
    pkv_status st = check_pool(pool);
    if (st != PKV_OK) return st;
    if (num_pairs < 0) return PKV_ERR_INVALID;
    if (num_pairs == 0) return PKV_OK;
    if (!k_pool || !v_pool || !pairs) return PKV_ERR_INVALID;
    if (!aligned16(k_pool) || !aligned16(v_pool)) return PKV_ERR_INVALID;
    if (num_pairs > 65535 * 1024) return PKV_ERR_UNSUPPORTED;
    int* status = status_word();
    if (!status) return PKV_ERR_CUDA;
    const int64_t block_bytes = static_cast<int64_t>(pool->num_kv_heads) * pool->block_size *
                                pool->head_dim * elem_bytes(pool->dtype);
    return from_cuda(pkv::launch_copy_blocks(k_pool, v_pool, pairs, num_pairs, block_bytes,
                                             pool->num_blocks, status,
                                             static_cast<cudaStream_t>(stream)));
}

pkv_status pkv_read_device_status(int* status_out, void* stream) {
    if (!status_out) return PKV_ERR_INVALID;
    int* status = status_word();
    if (!status) return PKV_ERR_CUDA;
    cudaStream_t s = static_cast<cudaStream_t>(stream);
    int v = 0;
    if (cudaMemcpyAsync(&v, status, sizeof(int), cudaMemcpyDeviceToHost, s) != cudaSuccess)
        return PKV_ERR_CUDA;
    if (cudaMemsetAsync(status, 0, sizeof(int), s) != cudaSuccess) return PKV_ERR_CUDA;
    if (cudaStreamSynchronize(s) != cudaSuccess) return PKV_ERR_CUDA;
    *status_out = v;
    return PKV_OK;
}

}  // extern "C"
