// Host-side TMA tensor-map construction (cuTensorMapEncodeTiled through the
// runtime's driver entry point, so libpkv needs no direct libcuda link).
#include <cuda.h>
#include <cuda_runtime.h>
#include <cudaTypedefs.h>

#include <mutex>
#include <vector>

#include "kernels.h"

namespace pkv {

namespace {

PFN_cuTensorMapEncodeTiled_v12000 encode_fn() {
    static PFN_cuTensorMapEncodeTiled_v12000 fn = nullptr;
    static std::once_flag once;
    std::call_once(once, [] {
        void* p = nullptr;
        cudaDriverEntryPointQueryResult q;
        if (cudaGetDriverEntryPointByVersion("cuTensorMapEncodeTiled", &p, 12000,
                                             cudaEnableDefault, &q) == cudaSuccess &&
            q == cudaDriverEntryPointSuccess)
            fn = reinterpret_cast<PFN_cuTensorMapEncodeTiled_v12000>(p);
    });
    return fn;
}

// Pool maps are rebuilt for the same pools on every call; a small per-thread cache of
// the last few (kind, pool, rows, head_dim) keeps cuTensorMapEncodeTiled off the call
// path.  A map holds only the address, sizes and box, so it does not depend on the
// device, and a reused address with the same sizes encodes to the same map.
struct MapEntry {
    int kind;   // 0: make_pool_map, 1: make_pool_block_map
    const void* ptr;
    int64_t rows;
    int head_dim;
    CUtensorMap map;
};
constexpr int kMapCache = 8;
thread_local MapEntry t_maps[kMapCache];
thread_local int t_maps_used = 0;
thread_local int t_maps_next = 0;

bool cached_map(int kind, const void* ptr, int64_t rows, int head_dim, CUtensorMap* m) {
    for (int i = 0; i < t_maps_used; ++i) {
        const MapEntry& e = t_maps[i];
        if (e.kind == kind && e.ptr == ptr && e.rows == rows && e.head_dim == head_dim) {
            *m = e.map;
            return true;
        }
    }
    return false;
}

void remember_map(int kind, const void* ptr, int64_t rows, int head_dim, const CUtensorMap& m) {
    MapEntry& e = t_maps[t_maps_next];
    e = MapEntry{kind, ptr, rows, head_dim, m};
    t_maps_next = (t_maps_next + 1) % kMapCache;
    if (t_maps_used < kMapCache) ++t_maps_used;
}

bool encode_pool_map(CUtensorMap* m, const void* pool, int64_t rows, int head_dim) {
    auto fn = encode_fn();
    if (!fn) return false;
    cuuint64_t dims[2] = {static_cast<cuuint64_t>(head_dim), static_cast<cuuint64_t>(rows)};
    cuuint64_t strides[1] = {static_cast<cuuint64_t>(head_dim) * 2};
    cuuint32_t box[2] = {64, 16};
    cuuint32_t estr[2] = {1, 1};
    return fn(m, CU_TENSOR_MAP_DATA_TYPE_BFLOAT16, 2, const_cast<void*>(pool), dims, strides, box,
              estr, CU_TENSOR_MAP_INTERLEAVE_NONE, CU_TENSOR_MAP_SWIZZLE_128B,
              CU_TENSOR_MAP_L2_PROMOTION_L2_256B, CU_TENSOR_MAP_FLOAT_OOB_FILL_NONE) ==
           CUDA_SUCCESS;
}

bool encode_pool_block_map(CUtensorMap* m, const void* pool, int64_t rows) {
    auto fn = encode_fn();
    if (!fn || rows % 8 != 0) return false;
    // Row r of the pool starts at r * 256 bytes; its column half h at + h * 128.
    cuuint64_t dims[4] = {64, 8, 2, static_cast<cuuint64_t>(rows / 8)};
    cuuint64_t strides[3] = {256, 128, 8 * 256};
    cuuint32_t box[4] = {64, 8, 2, 2};
    cuuint32_t estr[4] = {1, 1, 1, 1};
    return fn(m, CU_TENSOR_MAP_DATA_TYPE_BFLOAT16, 4, const_cast<void*>(pool), dims, strides, box,
              estr, CU_TENSOR_MAP_INTERLEAVE_NONE, CU_TENSOR_MAP_SWIZZLE_128B,
              CU_TENSOR_MAP_L2_PROMOTION_L2_256B, CU_TENSOR_MAP_FLOAT_OOB_FILL_NONE) ==
           CUDA_SUCCESS;
}

}  // namespace

bool make_pool_map(CUtensorMap* m, const void* pool, int64_t rows, int head_dim) {
    if (cached_map(0, pool, rows, head_dim, m)) return true;
    if (!encode_pool_map(m, pool, rows, head_dim)) return false;
    remember_map(0, pool, rows, head_dim, *m);
    return true;
}

bool make_pool_block_map(CUtensorMap* m, const void* pool, int64_t rows) {
    if (cached_map(1, pool, rows, 128, m)) return true;
    if (!encode_pool_block_map(m, pool, rows)) return false;
    remember_map(1, pool, rows, 128, *m);
    return true;
}

cudaError_t set_smem_once(const void* kern, int bytes) {
    int dev = 0;
    cudaError_t e = cudaGetDevice(&dev);
    if (e != cudaSuccess) return e;
    struct Done {
        const void* kern;
        int dev;
        int bytes;
    };
    static std::mutex mu;
    static std::vector<Done> done;
    {
        std::lock_guard<std::mutex> lk(mu);
        for (const Done& d : done)
            if (d.kern == kern && d.dev == dev && d.bytes >= bytes) return cudaSuccess;
    }
    e = cudaFuncSetAttribute(kern, cudaFuncAttributeMaxDynamicSharedMemorySize, bytes);
    if (e != cudaSuccess) return e;
    std::lock_guard<std::mutex> lk(mu);
    done.push_back(Done{kern, dev, bytes});
    return cudaSuccess;
}

bool make_q_group_map(CUtensorMap* m, const void* q, int tokens, int hq, int head_dim, int G,
                      int tok) {
    auto fn = encode_fn();
    if (!fn) return false;
    cuuint64_t dims[3] = {static_cast<cuuint64_t>(head_dim), static_cast<cuuint64_t>(hq),
                          static_cast<cuuint64_t>(tokens)};
    cuuint64_t strides[2] = {static_cast<cuuint64_t>(head_dim) * 2,
                             static_cast<cuuint64_t>(hq) * head_dim * 2};
    cuuint32_t box[3] = {64, static_cast<cuuint32_t>(G), static_cast<cuuint32_t>(tok)};
    cuuint32_t estr[3] = {1, 1, 1};
    return fn(m, CU_TENSOR_MAP_DATA_TYPE_BFLOAT16, 3, const_cast<void*>(q), dims, strides, box,
              estr, CU_TENSOR_MAP_INTERLEAVE_NONE, CU_TENSOR_MAP_SWIZZLE_128B,
              CU_TENSOR_MAP_L2_PROMOTION_L2_256B, CU_TENSOR_MAP_FLOAT_OOB_FILL_NONE) ==
           CUDA_SUCCESS;
}

}  // namespace pkv
