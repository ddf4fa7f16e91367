// Prefix-chunk causal prefill for fp32 pools, on the CUDA cores.
//
// The same computation as the tcgen05 prefill kernel (new query tokens of a request
// attend to its cached prefix plus the new tokens up to themselves, K/V gathered
// through the block table: Triptych "Paged Attention for Efficient Memory
// Management"; only the unseen suffix is computed: aitalk.it "RadixAttention: A Tree
// That Does Not Forget"), for fp32 K/V, where the tensor cores would round the
// operands to tf32.  FlashAttention-style tiling on the FMA pipe:
//
// One CTA (256 threads) computes one query tile of 16 R rows (R = 8 at head_dim 128,
// 4 at 64): 16 R / G consecutive new tokens x the G query heads of kv head `kvh` (rows
// token-major, heads inner), so each staged K/V tile serves all G heads.  Per 64-key KV
// tile:
//   S = Q K^T     thread (ty, tx) = (threadIdx.x / 16, threadIdx.x % 16) computes rows
//                 R ty + i and keys tx + 16 j (i < R, j < 4) from shared memory, float4
//                 reads (R + 4 reads per 16 R FMAs).  Only K rows are padded by 16
//                 bytes: a K read touches 16 rows at one column, while Q and P reads
//                 are broadcasts and V reads cover 16 consecutive pieces of one row, so
//                 they are conflict-free unpadded (head_dim 128: 161 KB, one CTA per SM
//                 with up to 255 registers a thread; head_dim 64: 66 KB, three)
//   softmax       online, log2 domain; the 16 threads of a half-warp share a row and
//                 meet by shuffles for its max; each keeps its share of the row sum
//   O += P V      P through shared memory; the same thread owns rows R ty + i and
//                 columns 4 tx + 64 c of O in registers (R + 2 D / 64 reads per 8 R D / 64
//                 FMAs per key step)
// K and V are staged by cp.async (16-byte pieces, zero-filled past the last key the
// tile needs); the next tile's K loads while P.V runs and its V while S runs.
#include <cuda_runtime.h>

#include "common.cuh"
#include "kernels.h"

namespace pkv {

namespace {

constexpr int kFKeys = 64;      // keys per KV tile
constexpr int kFThreads = 256;
// Query rows per thread: 8 at head_dim 128 (a 128-row tile, one CTA per SM), 4 at 64.
template <int D>
constexpr int rows_per_thread() { return D == 128 ? 8 : 4; }

template <int D>
struct FGeom {
    static constexpr int kRows = 16 * rows_per_thread<D>();   // query rows per CTA
    static constexpr int kKStride = D + 4;         // floats per staged K row (16-byte pad)
    static constexpr int kPStride = kFKeys;
    static constexpr int kOffQ = 0;
    static constexpr int kOffK = kOffQ + kRows * D * 4;
    static constexpr int kOffV = kOffK + kFKeys * kKStride * 4;
    static constexpr int kOffP = kOffV + kFKeys * D * 4;
    static constexpr int kBytes = kOffP + kRows * kPStride * 4;
    static constexpr int kPieces = D / 4;          // 16-byte pieces per row
};

// 16-byte global -> shared copy; src_bytes 0 writes zeros (no global read).
PKV_DEVINL void cp_async16(void* dst, const void* src, int src_bytes) {
    asm volatile("cp.async.cg.shared.global [%0], [%1], 16, %2;" ::"r"(smem_u32(dst)), "l"(src),
                 "r"(src_bytes)
                 : "memory");
}
PKV_DEVINL void cp_async_commit() { asm volatile("cp.async.commit_group;" ::: "memory"); }
// Wait until at most `n` of this thread's committed groups are still in flight.
template <int N>
PKV_DEVINL void cp_async_wait() {
    asm volatile("cp.async.wait_group %0;" ::"n"(N) : "memory");
}

// Stage keys [kbase, kbase + 64) of kv head kvh: key kbase + k into row k (kStride
// floats apart).  Keys past `last` (the last key any row of the tile sees) and keys of
// out-of-range blocks are zero-filled (an out-of-range block id also raises
// PKV_ERR_OOB).
template <int D, int kStride>
PKV_DEVINL void stage_kv(float* dst, const float* pool, const int32_t* bt, int kbase, int last,
                         int kvh, const PrefillArgs& a) {
    using FG = FGeom<D>;
    const int piece = threadIdx.x % FG::kPieces;
#pragma unroll
    for (int k = threadIdx.x / FG::kPieces; k < kFKeys; k += kFThreads / FG::kPieces) {
        const int pos = kbase + k;
        const float* src = pool;
        int bytes = 0;
        if (pos <= last) {
            const int phys = __ldg(bt + pos / a.block_size);
            if (phys >= 0 && phys < a.num_blocks) {
                src = pool + ((static_cast<size_t>(phys) * a.num_kv_heads + kvh) * a.block_size +
                              pos % a.block_size) * D + piece * 4;
                bytes = 16;
            } else if (piece == 0) {
                raise_status(a.status, PKV_ERR_OOB);
            }
        }
        cp_async16(dst + k * kStride + piece * 4, src, bytes);
    }
}

// At head_dim 128 one CTA per SM with 8 query rows a thread: against 4 rows and two
// CTAs per SM it halves the shared-memory reads per FMA and keeps twice the independent
// accumulators per thread, which outweighs the halved warp count (15.27 -> 14.23 ms on
// the prefix-cached prefill batch).  Three CTAs per SM at head_dim 64 (66 KB), where the
// extra warps hide more shared-memory latency than the registers given up for them
// cost (a few values spill at 80 registers).
template <int D, int G>
__global__ void __launch_bounds__(kFThreads, D == 64 ? 3 : 1)
prefill_f32_kernel(const PrefillArgs a) {
    using FG = FGeom<D>;
    constexpr int kFRows = FG::kRows;
    constexpr int R = rows_per_thread<D>();
    constexpr int kPvUnroll = D == 128 ? 4 : 2;   // P.V steps of 4 keys unrolled
    constexpr int TOK = kFRows / G;
    constexpr int OC = D / 64;   // float4 column groups of O per thread: 4 tx + 64 c
    extern __shared__ __align__(16) uint8_t smem_f[];
    float* Qs = reinterpret_cast<float*>(smem_f + FG::kOffQ);
    float* Ks = reinterpret_cast<float*>(smem_f + FG::kOffK);
    float* Vs = reinterpret_cast<float*>(smem_f + FG::kOffV);
    float* Ps = reinterpret_cast<float*>(smem_f + FG::kOffP);

    griddep_wait();
    griddep_launch_dependents();
    const int qt = blockIdx.x;
    const int kvh = blockIdx.y;
    const int r = blockIdx.z;
    const int n = a.new_lens[r];
    const int c = a.cached_lens[r];
    const int t0 = qt * TOK;
    if (t0 >= n) return;   // uniform over the CTA
    const int L = c + n;
    if (c < 0 || L > a.max_blocks_per_seq * a.block_size) {
        if (threadIdx.x == 0) raise_status(a.status, PKV_ERR_OOB);
        return;
    }
    const int max_lim = c + min(t0 + TOK, n) - 1;   // last key any row of the tile sees
    const int ntiles = max_lim / kFKeys + 1;
    const int qoff = a.q_offsets[r];
    const int32_t* bt = a.block_tables + static_cast<size_t>(r) * a.max_blocks_per_seq;
    const float* kpool = static_cast<const float*>(a.k_pool);
    const float* vpool = static_cast<const float*>(a.v_pool);

    // Q tile: row rho = token t0 + rho / G, head kvh G + rho % G; rows past the last new
    // token are zero.
    {
        const float* q = static_cast<const float*>(a.q);
        const int piece = threadIdx.x % FG::kPieces;
#pragma unroll
        for (int rho = threadIdx.x / FG::kPieces; rho < kFRows; rho += kFThreads / FG::kPieces) {
            const int tok = t0 + rho / G;
            const float* src = q;
            int bytes = 0;
            if (tok < n) {
                src = q + (static_cast<size_t>(qoff + tok) * a.num_q_heads + kvh * G + rho % G) * D +
                      piece * 4;
                bytes = 16;
            }
            cp_async16(Qs + rho * D + piece * 4, src, bytes);
        }
    }
    stage_kv<D, FG::kKStride>(Ks, kpool, bt, 0, max_lim, kvh, a);
    cp_async_commit();   // group: Q, K_0
    stage_kv<D, D>(Vs, vpool, bt, 0, max_lim, kvh, a);
    cp_async_commit();   // group: V_0

    const int tx = threadIdx.x & 15;
    const int ty = threadIdx.x >> 4;
    int lim[R];   // last key row R ty + i sees
#pragma unroll
    for (int i = 0; i < R; ++i) {
        const int tok = t0 + (R * ty + i) / G;
        lim[i] = tok < n ? c + tok : c + n - 1;
    }
    const float sl2 = a.scale_log2;
    float m[R], l[R], o[R][OC][4];
#pragma unroll
    for (int i = 0; i < R; ++i) {
        m[i] = -1.0e30f;   // finite: exp2(m_old - m_new) stays 0 before the first key
        l[i] = 0.f;
#pragma unroll
        for (int cc = 0; cc < OC; ++cc)
#pragma unroll
            for (int e = 0; e < 4; ++e) o[i][cc][e] = 0.f;
    }

    for (int jt = 0; jt < ntiles; ++jt) {
        const int kbase = jt * kFKeys;
        cp_async_wait<1>();   // Q and K_jt landed (V_jt may still be in flight)
        __syncthreads();

        // S = Q K^T for rows 4 ty + i, keys tx + 16 j.
        float s[R][4];
#pragma unroll
        for (int i = 0; i < R; ++i)
#pragma unroll
            for (int j = 0; j < 4; ++j) s[i][j] = 0.f;
#pragma unroll 4
        for (int d = 0; d < D; d += 4) {
            float4 qv[R], kv[4];
#pragma unroll
            for (int i = 0; i < R; ++i)
                qv[i] = *reinterpret_cast<const float4*>(Qs + (R * ty + i) * D + d);
#pragma unroll
            for (int j = 0; j < 4; ++j)
                kv[j] = *reinterpret_cast<const float4*>(Ks + (tx + 16 * j) * FG::kKStride + d);
#pragma unroll
            for (int i = 0; i < R; ++i)
#pragma unroll
                for (int j = 0; j < 4; ++j) {
                    s[i][j] = fmaf(qv[i].x, kv[j].x, s[i][j]);
                    s[i][j] = fmaf(qv[i].y, kv[j].y, s[i][j]);
                    s[i][j] = fmaf(qv[i].z, kv[j].z, s[i][j]);
                    s[i][j] = fmaf(qv[i].w, kv[j].w, s[i][j]);
                }
        }
        // Online softmax in the log2 domain; the row max over the half-warp.
        float alpha[R];
#pragma unroll
        for (int i = 0; i < R; ++i) {
            float mx = -INFINITY;
#pragma unroll
            for (int j = 0; j < 4; ++j) {
                s[i][j] = (kbase + tx + 16 * j <= lim[i]) ? s[i][j] * sl2 : -INFINITY;
                mx = fmaxf(mx, s[i][j]);
            }
#pragma unroll
            for (int off = 1; off < 16; off <<= 1)
                mx = fmaxf(mx, __shfl_xor_sync(0xffffffffu, mx, off));
            const float m_new = fmaxf(m[i], mx);
            alpha[i] = fast_exp2(m[i] - m_new);
            m[i] = m_new;
            float rs = 0.f;
#pragma unroll
            for (int j = 0; j < 4; ++j) {
                const float p = fast_exp2(s[i][j] - m_new);
                rs += p;
                Ps[(R * ty + i) * FG::kPStride + tx + 16 * j] = p;
            }
            l[i] = l[i] * alpha[i] + rs;
        }
        __syncthreads();   // P written; every thread is done with K_jt

        // K of the next tile into the freed buffer while P.V runs.
        if (jt + 1 < ntiles) stage_kv<D, FG::kKStride>(Ks, kpool, bt, kbase + kFKeys, max_lim, kvh, a);
        cp_async_commit();   // (possibly empty) group: K_jt+1
        cp_async_wait<1>();  // V_jt landed
        __syncthreads();

        // O = alpha O + P V for rows 4 ty + i, columns 4 tx + 64 cc.
#pragma unroll
        for (int i = 0; i < R; ++i)
#pragma unroll
            for (int cc = 0; cc < OC; ++cc)
#pragma unroll
                for (int e = 0; e < 4; ++e) o[i][cc][e] *= alpha[i];
#pragma unroll kPvUnroll
        for (int k = 0; k < kFKeys; k += 4) {
            float4 pv[R];
#pragma unroll
            for (int i = 0; i < R; ++i)
                pv[i] = *reinterpret_cast<const float4*>(Ps + (R * ty + i) * FG::kPStride + k);
#pragma unroll
            for (int kk = 0; kk < 4; ++kk) {
                float4 vv[OC];
#pragma unroll
                for (int cc = 0; cc < OC; ++cc)
                    vv[cc] = *reinterpret_cast<const float4*>(Vs + (k + kk) * D + 64 * cc + 4 * tx);
#pragma unroll
                for (int i = 0; i < R; ++i) {
                    const float p = kk == 0 ? pv[i].x : kk == 1 ? pv[i].y : kk == 2 ? pv[i].z : pv[i].w;
#pragma unroll
                    for (int cc = 0; cc < OC; ++cc) {
                        o[i][cc][0] = fmaf(p, vv[cc].x, o[i][cc][0]);
                        o[i][cc][1] = fmaf(p, vv[cc].y, o[i][cc][1]);
                        o[i][cc][2] = fmaf(p, vv[cc].z, o[i][cc][2]);
                        o[i][cc][3] = fmaf(p, vv[cc].w, o[i][cc][3]);
                    }
                }
            }
        }
        __syncthreads();   // every thread is done with V_jt and P

        // V of the next tile while the next S runs.
        if (jt + 1 < ntiles) stage_kv<D, D>(Vs, vpool, bt, kbase + kFKeys, max_lim, kvh, a);
        cp_async_commit();   // (possibly empty) group: V_jt+1
    }
    cp_async_wait<0>();

    // Row sums over the half-warp, then O / l for the rows of real tokens.
    float* out = static_cast<float*>(a.out);
#pragma unroll
    for (int i = 0; i < R; ++i) {
        float li = l[i];
#pragma unroll
        for (int off = 1; off < 16; off <<= 1) li += __shfl_xor_sync(0xffffffffu, li, off);
        const int rho = R * ty + i;
        const int tok = t0 + rho / G;
        if (tok >= n) continue;
        const float inv = 1.f / li;
        float* dst = out + (static_cast<size_t>(qoff + tok) * a.num_q_heads + kvh * G + rho % G) * D;
#pragma unroll
        for (int cc = 0; cc < OC; ++cc)
            *reinterpret_cast<float4*>(dst + 64 * cc + 4 * tx) =
                make_float4(o[i][cc][0] * inv, o[i][cc][1] * inv, o[i][cc][2] * inv,
                            o[i][cc][3] * inv);
    }
}

template <int D, int G>
cudaError_t launch_f32_g(const PrefillArgs& a, cudaStream_t stream) {
    using FG = FGeom<D>;
    auto kern = prefill_f32_kernel<D, G>;
    cudaError_t e = set_smem_once(reinterpret_cast<const void*>(kern), FG::kBytes);
    if (e != cudaSuccess) return e;
    constexpr int TOK = FG::kRows / G;
    dim3 grid((a.max_new + TOK - 1) / TOK, a.num_kv_heads, a.num_reqs);
    return launch_pdl(kern, grid, dim3(kFThreads), FG::kBytes, stream, a);
}

template <int D>
cudaError_t launch_f32_d(const PrefillArgs& a, int group, cudaStream_t stream) {
    switch (group) {
        case 1: return launch_f32_g<D, 1>(a, stream);
        case 2: return launch_f32_g<D, 2>(a, stream);
        case 4: return launch_f32_g<D, 4>(a, stream);
        case 8: return launch_f32_g<D, 8>(a, stream);
        default: return cudaErrorNotSupported;
    }
}

}  // namespace

cudaError_t launch_paged_prefill_f32(const PrefillArgs& a, int group, cudaStream_t stream) {
    if (a.block_size != 16 && a.block_size != 32) return cudaErrorNotSupported;
    if (a.head_dim == 128) return launch_f32_d<128>(a, group, stream);
    if (a.head_dim == 64) return launch_f32_d<64>(a, group, stream);
    return cudaErrorNotSupported;
}

}  // namespace pkv
