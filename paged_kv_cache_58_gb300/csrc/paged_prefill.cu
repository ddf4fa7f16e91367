// Prefix-chunk causal prefill on the tcgen05 tensor cores.
//
// New query tokens of a request attend to the request's cached prefix plus the
// new tokens up to themselves; only the unseen suffix is computed while the
// cached K/V are reused from the pool (aitalk.it "RadixAttention: A Tree That
// Does Not Forget": compute only the unseen suffix; aifetchly SGLang guide,
// "Prefill Bypass").  K/V are gathered through the block table ("the kernel walks
// the block table", Triptych "Paged Attention for Efficient Memory Management").
//
// One CTA computes one 128-row query tile: TOK = 128 / G consecutive new tokens x
// the G query heads that share kv head `kvh` (rows token-major, heads inner), so
// every K/V tile it stages serves all G heads.  Per 128-key KV tile:
//   S = Q K^T     tcgen05.mma kind::f16 (bf16 in, fp32 accumulate) -> TMEM
//   softmax       4 warps, one thread per row: tcgen05.ld S, causal mask, exp2,
//                 row sums in fp32; P is split into bf16 hi + lo parts (P = hi + lo
//                 to ~2^-17 relative) stored to TMEM with tcgen05.st
//   O += P V      two tcgen05.mma passes (A = P hi, then P lo, read from TMEM; B = V
//                 from shared memory) into a TMEM accumulator that lives across tiles
// The split keeps the probabilities at fp32-like precision: a single bf16 P is off by
// up to 2^-9 per weight, which rows attending only a few keys do not average away.
// The running max is updated lazily: O and l are rescaled only when a row's max
// grows by more than 2^8, which keeps P <= 256 and leaves the result exact.
//
// Warp roles (192 threads): warps 0-3 softmax + epilogue (warp w owns TMEM lanes
// 32w..32w+31), warp 4 TMA producer, warp 5 TMEM owner + MMA issuer.  K and V
// tiles are double-buffered; each 16-token block of a tile arrives as two TMA
// boxes (64 columns x 16 rows, 128-byte swizzle) per pool.
//
// TMEM columns: S buffers at [0, 128) and [128, 256), O at [256, 384), P hi at
// [384, 448) and P lo at [448, 512) (two bf16 per column).
#include <cuda.h>
#include <cuda_runtime.h>

#include "common.cuh"
#include "kernels.h"
#include "tcgen05.cuh"

namespace pkv {

namespace {

constexpr int kRows = 128;                 // query rows per tile
constexpr int kKeys = 128;                 // keys per KV tile
constexpr int kHead = 128;                 // head_dim
constexpr int kBlk = 16;                   // tokens per pool block
constexpr int kHalf = kRows * 128;         // one 64-column half of a 128-row tile: 16 KB
constexpr int kTileBytes = 2 * kHalf;      // 32 KB
constexpr int kBoxBytes = kBlk * 128;      // one TMA box: 16 rows x 128 B
constexpr int kStages = 2;
constexpr int kOffQ = 0;
constexpr int kOffK = kOffQ + kTileBytes;
constexpr int kOffV = kOffK + kStages * kTileBytes;
constexpr int kOffBar = kOffV + kStages * kTileBytes;
constexpr int kNumBars = 12;
constexpr int kSmemBytes = kOffBar + kNumBars * 8 + 16 + 1024;  // + 1 KB alignment slack
constexpr int kThreads = 192;
constexpr uint32_t kTmemCols = 512;
constexpr float kLazyRescale = 8.0f;       // log2 units

// barrier indices
constexpr int BQ = 0, BKV_FULL = 1, BKV_EMPTY = 3, BS_FULL = 5, BS_FREE = 7, BP_FULL = 9,
              BPV_DONE = 10;

struct Ctl {
    uint64_t* bars;
    volatile int* abort_flag;
    int* status;
};

// Bounded mbarrier wait shared by all roles: gives up when another role aborted
// or after the time budget (then raises PKV_ERR_TIMEOUT and aborts the CTA).
PKV_DEVINL bool wait_bar(const Ctl& c, int idx, uint32_t parity) {
    uint64_t* bar = &c.bars[idx];
    if (mbar_try_wait(bar, parity)) return true;
    const unsigned long long t0 = globaltimer_ns();
    for (;;) {
        if (mbar_try_wait(bar, parity)) return true;
        if (*c.abort_flag) return false;
        if (globaltimer_ns() - t0 > kWaitBudgetNs) {
            raise_status(c.status, PKV_ERR_TIMEOUT);
            *c.abort_flag = 1;
            return false;
        }
    }
}

// Warp-uniform variant for the softmax warps: lane 0 polls, the result is broadcast,
// and __syncwarp orders the other lanes after lane 0's acquire.
PKV_DEVINL bool wait_bar_warp(const Ctl& c, int idx, uint32_t parity, int lane) {
    int ok = 1;
    if (lane == 0) ok = wait_bar(c, idx, parity) ? 1 : 0;
    ok = __shfl_sync(0xffffffffu, ok, 0);
    __syncwarp();
    return ok != 0;
}

template <int G>
__global__ void __launch_bounds__(kThreads, 1)
prefill_tcgen05_kernel(const __grid_constant__ CUtensorMap tm_q,
                       const __grid_constant__ CUtensorMap tm_k,
                       const __grid_constant__ CUtensorMap tm_v, const PrefillArgs a) {
    constexpr int TOK = kRows / G;
    extern __shared__ uint8_t smem_raw[];
    uint8_t* smem = reinterpret_cast<uint8_t*>(
        (reinterpret_cast<uintptr_t>(smem_raw) + 1023) & ~static_cast<uintptr_t>(1023));

    const int qt = blockIdx.x;
    const int kvh = blockIdx.y;
    const int r = blockIdx.z;
    const int warp = threadIdx.x >> 5;
    const int lane = threadIdx.x & 31;

    const int n = a.new_lens[r];
    const int c = a.cached_lens[r];
    const int t0 = qt * TOK;
    if (t0 >= n) return;  // uniform over the CTA, before any barrier or TMEM use
    const int L = c + n;
    if (c < 0 || L > a.max_blocks_per_seq * kBlk) {
        if (threadIdx.x == 0) raise_status(a.status, PKV_ERR_OOB);
        return;
    }
    const int i_last = min(t0 + TOK, n) - 1;
    const int max_lim = c + i_last;          // last key any row of this tile sees
    const int ntiles = max_lim / kKeys + 1;
    const int qrow0 = a.q_offsets[r] + t0;   // first token row of the tile in q / out

    uint64_t* bars = reinterpret_cast<uint64_t*>(smem + kOffBar);
    uint32_t* tmem_slot = reinterpret_cast<uint32_t*>(smem + kOffBar + kNumBars * 8);
    volatile int* abort_flag = reinterpret_cast<volatile int*>(tmem_slot + 1);
    Ctl ctl{bars, abort_flag, a.status};

    if (warp == 5) {
        if (lane == 0) {
            mbar_init(&bars[BQ], 1);
            for (int s = 0; s < kStages; ++s) {
                mbar_init(&bars[BKV_FULL + s], 1);
                mbar_init(&bars[BKV_EMPTY + s], 1);
                mbar_init(&bars[BS_FULL + s], 1);
                mbar_init(&bars[BS_FREE + s], 4);
            }
            mbar_init(&bars[BP_FULL], 4);
            mbar_init(&bars[BPV_DONE], 1);
            *abort_flag = 0;
            fence_mbar_init();
        }
        __syncwarp();
        tmem_alloc(tmem_slot, kTmemCols);
        tmem_relinquish();
    }
    tc_fence_before();
    __syncthreads();
    tc_fence_after();
    const uint32_t tmem = *tmem_slot;

    const uint32_t sQ = smem_u32(smem + kOffQ);
    const uint32_t sK = smem_u32(smem + kOffK);
    const uint32_t sV = smem_u32(smem + kOffV);

    if (warp == 4) {
        // ------------------------------------------------------------ TMA producer
        if (lane == 0) {
            prefetch_tmap(&tm_q);
            prefetch_tmap(&tm_k);
            prefetch_tmap(&tm_v);
            const int32_t* bt = a.block_tables + static_cast<size_t>(r) * a.max_blocks_per_seq;
            const int nblk_needed = max_lim / kBlk + 1;
            mbar_arrive_expect_tx(&bars[BQ], kTileBytes);
            tma_load_3d(smem + kOffQ, &tm_q, 0, kvh * G, qrow0, &bars[BQ]);
            tma_load_3d(smem + kOffQ + kHalf, &tm_q, 64, kvh * G, qrow0, &bars[BQ]);
            for (int jt = 0; jt < ntiles; ++jt) {
                const int s = jt & 1;
                if (jt >= 2 && !wait_bar(ctl, BKV_EMPTY + s, ((jt >> 1) - 1) & 1)) break;
                const int nb = min(kKeys / kBlk, nblk_needed - jt * (kKeys / kBlk));
                mbar_arrive_expect_tx(&bars[BKV_FULL + s], nb * 4 * kBoxBytes);
                uint8_t* kdst = smem + kOffK + s * kTileBytes;
                uint8_t* vdst = smem + kOffV + s * kTileBytes;
                for (int b = 0; b < nb; ++b) {
                    int phys = __ldg(bt + jt * (kKeys / kBlk) + b);
                    if (phys < 0 || phys >= a.num_blocks) {
                        raise_status(a.status, PKV_ERR_OOB);
                        phys = 0;  // keep the byte count; the output is flagged invalid
                    }
                    const int row = (phys * a.num_kv_heads + kvh) * kBlk;
                    tma_load_2d(kdst + b * kBoxBytes, &tm_k, 0, row, &bars[BKV_FULL + s]);
                    tma_load_2d(kdst + kHalf + b * kBoxBytes, &tm_k, 64, row,
                                &bars[BKV_FULL + s]);
                    tma_load_2d(vdst + b * kBoxBytes, &tm_v, 0, row, &bars[BKV_FULL + s]);
                    tma_load_2d(vdst + kHalf + b * kBoxBytes, &tm_v, 64, row,
                                &bars[BKV_FULL + s]);
                }
            }
        }
    } else if (warp == 5) {
        // ------------------------------------------------------------ MMA issuer
        if (lane == 0) {
            constexpr uint32_t idesc_qk = idesc_bf16_f32(kRows, kKeys, false, false);
            constexpr uint32_t idesc_pv = idesc_bf16_f32(kRows, kHead, false, true);
            const uint32_t tO = tmem + 256;
            bool ok = wait_bar(ctl, BQ, 0);
            for (int jt = 0; ok && jt <= ntiles; ++jt) {
                if (jt < ntiles) {
                    const int s = jt & 1;
                    if (!wait_bar(ctl, BKV_FULL + s, (jt >> 1) & 1)) break;
                    if (jt >= 2 && !wait_bar(ctl, BS_FREE + s, ((jt >> 1) - 1) & 1)) break;
                    tc_fence_after();
                    const uint32_t tS = tmem + s * 128;
#pragma unroll
                    for (int ks = 0; ks < kHead / 16; ++ks) {
                        const uint32_t off = (ks >> 2) * kHalf + (ks & 3) * 32;
                        umma_bf16(tS, smem_desc_sw128(sQ + off, 16, 1024),
                                  smem_desc_sw128(sK + s * kTileBytes + off, 16, 1024), idesc_qk,
                                  ks > 0);
                    }
                    umma_commit(&bars[BS_FULL + s]);
                }
                if (jt >= 1) {
                    const int j = jt - 1;
                    const int sj = j & 1;
                    if (!wait_bar(ctl, BP_FULL, j & 1)) break;
                    tc_fence_after();
#pragma unroll
                    for (int ks = 0; ks < kKeys / 16; ++ks) {
                        const uint64_t bv =
                            smem_desc_sw128(sV + sj * kTileBytes + ks * 2048, kHalf, 1024);
                        umma_bf16_ta(tO, tmem + 384 + ks * 8, bv, idesc_pv, (j > 0) || (ks > 0));
                        umma_bf16_ta(tO, tmem + 448 + ks * 8, bv, idesc_pv, true);
                    }
                    umma_commit(&bars[BPV_DONE]);
                    umma_commit(&bars[BKV_EMPTY + sj]);
                }
            }
        }
    } else {
        // ------------------------------------------------------------ softmax + epilogue
        const int row = threadIdx.x;              // 0..127 == TMEM lane
        const uint32_t lane_addr = static_cast<uint32_t>(warp * 32) << 16;
        const int tok = t0 + row / G;
        const int head = kvh * G + row % G;
        const bool row_valid = tok < n;
        const int lim = row_valid ? c + tok : c + n - 1;   // last key this row sees
        const float sl2 = a.scale_log2;
        float m_used = -INFINITY;
        float l = 0.f;
        bool ok = true;
        for (int jt = 0; jt < ntiles; ++jt) {
            const int s = jt & 1;
            if (!wait_bar_warp(ctl, BS_FULL + s, (jt >> 1) & 1, lane)) { ok = false; break; }
            tc_fence_after();
            float x[kKeys];
#pragma unroll
            for (int q = 0; q < 4; ++q)
                tmem_ld32(tmem + lane_addr + s * 128 + q * 32,
                          *reinterpret_cast<float(*)[32]>(&x[q * 32]));
            tmem_wait_ld();
            tc_fence_before();
            __syncwarp();
            if (lane == 0) mbar_arrive(&bars[BS_FREE + s]);

            const int kbase = jt * kKeys;
            float mx = -INFINITY;
            if (kbase + kKeys - 1 <= lim) {
#pragma unroll
                for (int k = 0; k < kKeys; ++k) mx = fmaxf(mx, x[k]);
            } else {
#pragma unroll
                for (int k = 0; k < kKeys; ++k) {
                    x[k] = (kbase + k <= lim) ? x[k] : -INFINITY;
                    mx = fmaxf(mx, x[k]);
                }
            }
            const float m_tile = mx * sl2;   // scale > 0: max commutes with scaling
            const bool grow = m_tile > m_used + kLazyRescale;
            const float m_cur = grow ? m_tile : m_used;
            const float alpha = fast_exp2(m_used - m_cur);   // 1 unless grow; 0 at start
            float rs = 0.f;
            float phi[kKeys / 2], plo[kKeys / 2];   // packed bf16 pairs, as fp32 bit patterns
#pragma unroll
            for (int k = 0; k < kKeys; k += 2) {
                const float p0 = fast_exp2(fmaf(x[k], sl2, -m_cur));
                const float p1 = fast_exp2(fmaf(x[k + 1], sl2, -m_cur));
                rs += p0 + p1;
                const uint32_t h = pack_bf16x2(p0, p1);
                const float r0 = p0 - bf16lo_to_f32(h);
                const float r1 = p1 - bf16hi_to_f32(h);
                phi[k / 2] = __uint_as_float(h);
                plo[k / 2] = __uint_as_float(pack_bf16x2(r0, r1));
            }
            l = l * alpha + rs;
            m_used = m_cur;

            // P and O may be touched only after the previous tile's P.V finished.
            if (jt >= 1 && !wait_bar_warp(ctl, BPV_DONE, (jt - 1) & 1, lane)) {
                ok = false;
                break;
            }
            tc_fence_after();
            if (jt >= 1 && __any_sync(0xffffffffu, grow)) {
#pragma unroll
                for (int q = 0; q < 4; ++q) {
                    float o[32];
                    const uint32_t ta = tmem + lane_addr + 256 + q * 32;
                    tmem_ld32(ta, o);
                    tmem_wait_ld();
#pragma unroll
                    for (int e = 0; e < 32; ++e) o[e] *= alpha;
                    tmem_st32(ta, o);
                }
                tmem_wait_st();
            }
            // P row -> TMEM (this thread's lane), hi and lo parts.
#pragma unroll
            for (int q = 0; q < 2; ++q) {
                tmem_st32(tmem + lane_addr + 384 + q * 32,
                          *reinterpret_cast<float(*)[32]>(&phi[q * 32]));
                tmem_st32(tmem + lane_addr + 448 + q * 32,
                          *reinterpret_cast<float(*)[32]>(&plo[q * 32]));
            }
            tmem_wait_st();
            // Keys past the last one this tile needs are masked for every row, but their
            // V rows may hold anything (NaN in unused slots, stale data where no block was
            // loaded this tile); zero them so that 0 * V stays 0 in the P.V product.
            if (kbase + row > max_lim) {
                uint8_t* vrow = smem + kOffV + s * kTileBytes + row * 128;
                const uint4 z = make_uint4(0, 0, 0, 0);
#pragma unroll
                for (int j = 0; j < 8; ++j) {
                    *reinterpret_cast<uint4*>(vrow + (j << 4)) = z;
                    *reinterpret_cast<uint4*>(vrow + kHalf + (j << 4)) = z;
                }
            }
            fence_proxy_async_smem();
            tc_fence_before();
            __syncwarp();
            if (lane == 0) mbar_arrive(&bars[BP_FULL]);
        }
        // ------------------------------------------------------------ epilogue
        if (ok && wait_bar_warp(ctl, BPV_DONE, (ntiles - 1) & 1, lane)) {
            tc_fence_after();
            const float inv_l = 1.f / l;
            uint16_t* orow = static_cast<uint16_t*>(a.out) +
                             (static_cast<size_t>(a.q_offsets[r] + tok) * a.num_q_heads + head) *
                                 kHead;
#pragma unroll
            for (int q = 0; q < 4; ++q) {
                float o[32];
                tmem_ld32(tmem + lane_addr + 256 + q * 32, o);
                tmem_wait_ld();
                if (row_valid) {
#pragma unroll
                    for (int e = 0; e < 32; e += 8) {
                        uint4 w;
                        w.x = pack_bf16x2(o[e] * inv_l, o[e + 1] * inv_l);
                        w.y = pack_bf16x2(o[e + 2] * inv_l, o[e + 3] * inv_l);
                        w.z = pack_bf16x2(o[e + 4] * inv_l, o[e + 5] * inv_l);
                        w.w = pack_bf16x2(o[e + 6] * inv_l, o[e + 7] * inv_l);
                        *reinterpret_cast<uint4*>(orow + q * 32 + e) = w;
                    }
                }
            }
        }
    }

    tc_fence_before();
    __syncthreads();
    if (warp == 5) {
        __syncwarp();
        tc_fence_after();
        tmem_dealloc(tmem, kTmemCols);
    }
}

template <int G>
cudaError_t launch_g(const PrefillArgs& a, cudaStream_t stream) {
    CUtensorMap mq, mk, mv;
    const int64_t rows = a.num_blocks * a.num_kv_heads * kBlk;
    if (!make_q_group_map(&mq, a.q, a.total_new, a.num_q_heads, kHead, G, kRows / G) ||
        !make_pool_map(&mk, a.k_pool, rows, kHead) || !make_pool_map(&mv, a.v_pool, rows, kHead))
        return cudaErrorInvalidValue;
    auto kern = prefill_tcgen05_kernel<G>;
    cudaError_t e =
        cudaFuncSetAttribute(kern, cudaFuncAttributeMaxDynamicSharedMemorySize, kSmemBytes);
    if (e != cudaSuccess) return e;
    constexpr int TOK = kRows / G;
    dim3 grid((a.max_new + TOK - 1) / TOK, a.num_kv_heads, a.num_reqs);
    kern<<<grid, kThreads, kSmemBytes, stream>>>(mq, mk, mv, a);
    return cudaGetLastError();
}

}  // namespace

cudaError_t launch_paged_prefill(const PrefillArgs& a, int group, cudaStream_t stream) {
    switch (group) {
        case 1: return launch_g<1>(a, stream);
        case 2: return launch_g<2>(a, stream);
        case 4: return launch_g<4>(a, stream);
        case 8: return launch_g<8>(a, stream);
        default: return cudaErrorNotSupported;
    }
}

}  // namespace pkv
