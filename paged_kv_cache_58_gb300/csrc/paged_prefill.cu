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
// every K/V tile it stages serves all G heads.  Per 128-key KV tile j:
//   S_j = Q K_j^T  tcgen05.mma kind::f16 (bf16 in, fp32 accumulate) into TMEM
//                  buffer j % 3
//   softmax        4 warps, one thread per row: tcgen05.ld S_j, causal mask, exp2,
//                  row sums in fp32; P_j is split into bf16 hi + lo parts (P = hi +
//                  lo to ~2^-17 relative) and stored back over S_j in the same TMEM
//                  buffer (hi in its first 64 columns, lo in the next 64)
//   O += P_j V_j   two tcgen05.mma passes (A = P hi, then P lo, from TMEM; B = V_j
//                  from shared memory) into a TMEM accumulator kept across tiles
// The split keeps the probabilities at fp32-like precision: a single bf16 P is off by
// up to 2^-9 per weight, which rows attending only a few keys do not average away.
// The running max is updated lazily: O and l are rescaled only when a row's max
// grows by more than 2^8, which keeps P <= 256 and leaves the result exact.
//
// Pipelining.  The MMA issuer runs S_{j+1} before P_j V_j; S_{j+3} reuses the
// buffer of P_j once P_j V_j has completed (its own per-buffer barrier: MMAs with
// different accumulators are not ordered against each other), which with three
// buffers is normally long done.  The softmax of tile j+1 overlaps P_j V_j and waits
// for it only when a row's max grew (O rescale).  K stages (3) are released as soon
// as their S has run, V stages (3) after their P.V, so the gathers of the next tiles
// are in flight while the current one is computed.  Each 16-token block of a tile
// arrives as two TMA boxes (64 columns x 16 rows, 128-byte swizzle) per pool.
//
// Measured limit: a 128 x 128 x 16 tcgen05.mma issues in about the time of a
// 128 x 256 x 16 one, so the 24 N = 128 MMAs per tile (8 for S, 16 for the hi + lo
// P.V) set the pace; the softmax finishes inside that time.
//
// Warp roles (192 threads): warps 0-3 softmax + epilogue (warp w owns TMEM lanes
// 32w..32w+31), warp 4 TMA producer, warp 5 TMEM owner + MMA issuer.
// TMEM columns: S/P buffers at [0, 128), [128, 256), [256, 384); O at [384, 512).
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
constexpr int kStagesK = 3;                // K stages: freed right after S = Q K^T
constexpr int kStagesV = 3;                // V stages: freed after P.V
constexpr int kOffQ = 0;
constexpr int kOffK = kOffQ + kTileBytes;
constexpr int kOffV = kOffK + kStagesK * kTileBytes;
constexpr int kOffBar = kOffV + kStagesV * kTileBytes;
constexpr int kNumBars = 24;
constexpr int kSmemBytes = kOffBar + kNumBars * 8 + 16 + 1024;  // + 1 KB alignment slack
constexpr int kSoftmaxWarps = 4;
constexpr int kProducerWarp = 4;
constexpr int kMmaWarp = 5;
constexpr int kThreads = 192;
constexpr uint32_t kTmemCols = 512;
constexpr uint32_t kTmemO = 384;
constexpr int kBufs = 3;                   // S/P buffers in TMEM
constexpr float kLazyRescale = 8.0f;       // log2 units

// barrier indices
constexpr int BQ = 0, BK_FULL = 1, BK_EMPTY = 4, BV_FULL = 7, BV_EMPTY = 10, BS_FULL = 13,
              BP_FULL = 16, BPV_DONE = 19;   // S_FULL / P_FULL / PV_DONE: one per buffer

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

    griddep_wait();
    griddep_launch_dependents();
    const int qt = blockIdx.x;
    const int kvh = blockIdx.y;
    const int r = blockIdx.z;
    const int warp = threadIdx.x >> 5;
    const int lane = threadIdx.x & 31;

    const bool cascade = a.cascade != 0;    // rows = sequences over the c shared keys
    const int n = cascade ? a.cascade_rows : a.new_lens[r];
    const int c = cascade ? a.cascade_keys : a.cached_lens[r];
    const int t0 = qt * TOK;
    if (t0 >= n) return;  // uniform over the CTA, before any barrier or TMEM use
    const int L = cascade ? c : c + n;       // keys in the pool for this request
    if (c < 0 || L <= 0 || L > a.max_blocks_per_seq * kBlk) {
        if (threadIdx.x == 0) raise_status(a.status, PKV_ERR_OOB);
        return;
    }
    const int i_last = min(t0 + TOK, n) - 1;
    const int max_lim = cascade ? c - 1 : c + i_last;   // last key any row of this tile sees
    const int ntiles = max_lim / kKeys + 1;
    const int qoff = cascade ? 0 : a.q_offsets[r];
    const int qrow0 = qoff + t0;             // first token row of the tile in q / out

    uint64_t* bars = reinterpret_cast<uint64_t*>(smem + kOffBar);
    uint32_t* tmem_slot = reinterpret_cast<uint32_t*>(smem + kOffBar + kNumBars * 8);
    volatile int* abort_flag = reinterpret_cast<volatile int*>(tmem_slot + 1);
    Ctl ctl{bars, abort_flag, a.status};

    if (warp == kMmaWarp) {
        if (lane == 0) {
            mbar_init(&bars[BQ], 1);
            for (int s = 0; s < kStagesK; ++s) {
                mbar_init(&bars[BK_FULL + s], 1);
                mbar_init(&bars[BK_EMPTY + s], 1);
            }
            for (int s = 0; s < kStagesV; ++s) {
                mbar_init(&bars[BV_FULL + s], 1);
                mbar_init(&bars[BV_EMPTY + s], 1);
            }
            for (int b = 0; b < kBufs; ++b) {
                mbar_init(&bars[BS_FULL + b], 1);
                mbar_init(&bars[BP_FULL + b], kSoftmaxWarps);
                mbar_init(&bars[BPV_DONE + b], 1);
            }
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

    if (warp == kProducerWarp) {
        // ------------------------------------------------------------ TMA producer
        // The whole warp runs the loop: each lane prefetches one block id (32 ids =
        // 4 KV tiles per refill, independent loads), lane 0 sets the byte counts and
        // lane b < 8 issues the boxes of block b of the tile.
        const int32_t* bt = a.block_tables + static_cast<size_t>(r) * a.max_blocks_per_seq;
        const int nblk_needed = max_lim / kBlk + 1;
        if (lane == 0) {
            prefetch_tmap(&tm_q);
            prefetch_tmap(&tm_k);
            prefetch_tmap(&tm_v);
            mbar_arrive_expect_tx(&bars[BQ], kTileBytes);
            tma_load_3d(smem + kOffQ, &tm_q, 0, kvh * G, qrow0, &bars[BQ]);
            tma_load_3d(smem + kOffQ + kHalf, &tm_q, 64, kvh * G, qrow0, &bars[BQ]);
        }
        int ids = 0;
        for (int jt = 0; jt < ntiles; ++jt) {
            constexpr int kPerTile = kKeys / kBlk;   // 8 blocks per KV tile
            if ((jt & 3) == 0) {
                const int i = jt * kPerTile + lane;
                ids = (i < nblk_needed) ? __ldg(bt + i) : 0;
            }
            const int sk = jt % kStagesK;
            const int sv = jt % kStagesV;
            const int nb = min(kPerTile, nblk_needed - jt * kPerTile);
            int phys = __shfl_sync(0xffffffffu, ids, ((jt & 3) * kPerTile) + (lane & 7));
            if (phys < 0 || phys >= a.num_blocks) {
                if (lane < nb) raise_status(a.status, PKV_ERR_OOB);
                phys = 0;  // keep the byte count; the output is flagged invalid
            }
            const int row = (phys * a.num_kv_heads + kvh) * kBlk;
            // K of tile jt: its stage is free once S of tile jt - kStagesK has run.
            int ok = 1;
            if (lane == 0 && jt >= kStagesK)
                ok = wait_bar(ctl, BK_EMPTY + sk, ((jt / kStagesK) - 1) & 1);
            ok = __shfl_sync(0xffffffffu, ok, 0);
            if (!ok) break;
            if (lane == 0) mbar_arrive_expect_tx(&bars[BK_FULL + sk], nb * 2 * kBoxBytes);
            __syncwarp();
            if (lane < nb) {
                uint8_t* kdst = smem + kOffK + sk * kTileBytes + lane * kBoxBytes;
                tma_load_2d(kdst, &tm_k, 0, row, &bars[BK_FULL + sk]);
                tma_load_2d(kdst + kHalf, &tm_k, 64, row, &bars[BK_FULL + sk]);
            }
            // V of tile jt: its stage is free once P.V of tile jt - kStagesV has run.
            if (lane == 0 && jt >= kStagesV)
                ok = wait_bar(ctl, BV_EMPTY + sv, ((jt / kStagesV) - 1) & 1);
            ok = __shfl_sync(0xffffffffu, ok, 0);
            if (!ok) break;
            if (lane == 0) mbar_arrive_expect_tx(&bars[BV_FULL + sv], nb * 2 * kBoxBytes);
            __syncwarp();
            if (lane < nb) {
                uint8_t* vdst = smem + kOffV + sv * kTileBytes + lane * kBoxBytes;
                tma_load_2d(vdst, &tm_v, 0, row, &bars[BV_FULL + sv]);
                tma_load_2d(vdst + kHalf, &tm_v, 64, row, &bars[BV_FULL + sv]);
            }
            __syncwarp();
        }
    } else if (warp == kMmaWarp) {
        // ------------------------------------------------------------ MMA issuer
        if (lane == 0) {
            constexpr uint32_t idesc_qk = idesc_bf16_f32(kRows, kKeys, false, false);
            constexpr uint32_t idesc_pv = idesc_bf16_f32(kRows, kHead, false, true);
            const uint32_t tO = tmem + kTmemO;
            bool ok = wait_bar(ctl, BQ, 0);
            for (int jt = 0; ok && jt <= ntiles; ++jt) {
                if (jt < ntiles) {
                    // S_jt into buffer jt % 3, once P_{jt-3} in it has been consumed.
                    const int ks_ = jt % kStagesK;
                    const int sb = jt % kBufs;
                    if (!wait_bar(ctl, BK_FULL + ks_, (jt / kStagesK) & 1)) break;
                    if (jt >= kBufs && !wait_bar(ctl, BPV_DONE + sb, ((jt / kBufs) - 1) & 1))
                        break;
                    tc_fence_after();
                    const uint32_t tS = tmem + sb * 128;
#pragma unroll
                    for (int ks = 0; ks < kHead / 16; ++ks) {
                        const uint32_t off = (ks >> 2) * kHalf + (ks & 3) * 32;
                        umma_bf16(tS, smem_desc_sw128(sQ + off, 16, 1024),
                                  smem_desc_sw128(sK + ks_ * kTileBytes + off, 16, 1024),
                                  idesc_qk, ks > 0);
                    }
                    umma_commit(&bars[BS_FULL + sb]);
                    umma_commit(&bars[BK_EMPTY + ks_]);
                }
                if (jt >= 1) {
                    const int j = jt - 1;
                    const int pb = j % kBufs;
                    const int vs = j % kStagesV;
                    if (!wait_bar(ctl, BP_FULL + pb, (j / kBufs) & 1)) break;
                    if (!wait_bar(ctl, BV_FULL + vs, (j / kStagesV) & 1)) break;
                    tc_fence_after();
                    const uint32_t tP = tmem + pb * 128;
#pragma unroll
                    for (int ks = 0; ks < kKeys / 16; ++ks) {
                        const uint64_t bv =
                            smem_desc_sw128(sV + vs * kTileBytes + ks * 2048, kHalf, 1024);
                        umma_bf16_ta(tO, tP + ks * 8, bv, idesc_pv, (j > 0) || (ks > 0));
                        umma_bf16_ta(tO, tP + 64 + ks * 8, bv, idesc_pv, true);
                    }
                    umma_commit(&bars[BPV_DONE + pb]);
                    umma_commit(&bars[BV_EMPTY + vs]);
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
        const int lim = cascade ? c - 1 : (row_valid ? c + tok : c + n - 1);  // last key seen
        const float sl2 = a.scale_log2;
        float m_used = -INFINITY;
        float l = 0.f;
        bool ok = true;
        for (int jt = 0; jt < ntiles; ++jt) {
            const int b = jt % kBufs;
            const uint32_t tS = tmem + lane_addr + b * 128;
            if (!wait_bar_warp(ctl, BS_FULL + b, (jt / kBufs) & 1, lane)) { ok = false; break; }
            tc_fence_after();
            float x[kKeys];
#pragma unroll
            for (int q = 0; q < 4; ++q)
                tmem_ld32(tS + q * 32, *reinterpret_cast<float(*)[32]>(&x[q * 32]));
            tmem_wait_ld();

            const int kbase = jt * kKeys;
            // Row max over 8 independent chains (one softmax warp per scheduler has
            // no other warp to hide long dependency chains behind).
            float m8[8];
#pragma unroll
            for (int u = 0; u < 8; ++u) m8[u] = -INFINITY;
            if (kbase + kKeys - 1 <= lim) {
#pragma unroll
                for (int k = 0; k < kKeys; ++k) m8[k & 7] = fmaxf(m8[k & 7], x[k]);
            } else {
#pragma unroll
                for (int k = 0; k < kKeys; ++k) {
                    x[k] = (kbase + k <= lim) ? x[k] : -INFINITY;
                    m8[k & 7] = fmaxf(m8[k & 7], x[k]);
                }
            }
            const float mx = fmaxf(fmaxf(fmaxf(m8[0], m8[1]), fmaxf(m8[2], m8[3])),
                                   fmaxf(fmaxf(m8[4], m8[5]), fmaxf(m8[6], m8[7])));
            const float m_tile = mx * sl2;   // scale > 0: max commutes with scaling
            const bool grow = m_tile > m_used + kLazyRescale;
            const float m_cur = grow ? m_tile : m_used;
            const float alpha = fast_exp2(m_used - m_cur);   // 1 unless grow; 0 at start
            // O is rescaled only when some row of the warp grew its max; that needs the
            // previous tile's P.V to have finished.  Otherwise P.V of tile jt - 1 keeps
            // running while this tile's P is written to its own buffer.
            if (jt >= 1 && __any_sync(0xffffffffu, grow)) {
                if (!wait_bar_warp(ctl, BPV_DONE + (jt - 1) % kBufs, ((jt - 1) / kBufs) & 1,
                                   lane)) {
                    ok = false;
                    break;
                }
                tc_fence_after();
#pragma unroll
                for (int q = 0; q < 4; ++q) {
                    float o[32];
                    const uint32_t ta = tmem + lane_addr + kTmemO + q * 32;
                    tmem_ld32(ta, o);
                    tmem_wait_ld();
#pragma unroll
                    for (int e = 0; e < 32; ++e) o[e] *= alpha;
                    tmem_st32(ta, o);
                }
            }
            // P_jt over S_jt in the same buffer (S is already in registers): hi in columns
            // [0, 64), lo in [64, 128), written 32 keys at a time so that few packed
            // values are live and the exp chains of a chunk overlap.
            float rs8[8];
#pragma unroll
            for (int u = 0; u < 8; ++u) rs8[u] = 0.f;
#pragma unroll
            for (int q = 0; q < kKeys / 32; ++q) {
                uint32_t phi[16], plo[16];
#pragma unroll
                for (int e = 0; e < 16; ++e) {
                    const int k = q * 32 + 2 * e;
                    const float p0 = fast_exp2(fmaf(x[k], sl2, -m_cur));
                    const float p1 = fast_exp2(fmaf(x[k + 1], sl2, -m_cur));
                    rs8[e & 7] += p0 + p1;
                    const uint32_t h = pack_bf16x2(p0, p1);
                    phi[e] = h;
                    plo[e] = pack_bf16x2(p0 - bf16lo_to_f32(h), p1 - bf16hi_to_f32(h));
                }
                tmem_st16(tS + q * 16, phi);
                tmem_st16(tS + 64 + q * 16, plo);
            }
            const float rs = ((rs8[0] + rs8[1]) + (rs8[2] + rs8[3])) +
                             ((rs8[4] + rs8[5]) + (rs8[6] + rs8[7]));
            l = l * alpha + rs;
            m_used = m_cur;
            tmem_wait_st();
            // Keys past the last one this tile needs are masked for every row, but their
            // V rows may hold anything (NaN in unused slots, stale data where no block was
            // loaded this tile); zero them so that 0 * V stays 0 in the P.V product, once
            // this tile's V has landed.
            if (kbase + kKeys - 1 > max_lim) {
                if (!wait_bar_warp(ctl, BV_FULL + jt % kStagesV, (jt / kStagesV) & 1, lane)) {
                    ok = false;
                    break;
                }
                if (kbase + row > max_lim) {
                    uint8_t* vrow = smem + kOffV + (jt % kStagesV) * kTileBytes + row * 128;
                    const uint4 z = make_uint4(0, 0, 0, 0);
#pragma unroll
                    for (int j = 0; j < 8; ++j) {
                        *reinterpret_cast<uint4*>(vrow + (j << 4)) = z;
                        *reinterpret_cast<uint4*>(vrow + kHalf + (j << 4)) = z;
                    }
                }
                fence_proxy_async_smem();
            }
            tc_fence_before();
            __syncwarp();
            if (lane == 0) mbar_arrive(&bars[BP_FULL + b]);
        }
        // ------------------------------------------------------------ epilogue
        if (ok && wait_bar_warp(ctl, BPV_DONE + (ntiles - 1) % kBufs,
                                ((ntiles - 1) / kBufs) & 1, lane)) {
            tc_fence_after();
            const float inv_l = 1.f / l;
            const size_t orow_idx = static_cast<size_t>(qoff + tok) * a.num_q_heads + head;
            uint16_t* orow = static_cast<uint16_t*>(a.out) + orow_idx * kHead;
            const size_t prow = orow_idx * a.max_parts_total;   // cascade: partition 0
            if (cascade && row_valid) {
                a.m_part[prow] = m_used;   // log2 domain, as the decode partials
                a.l_part[prow] = l;
            }
#pragma unroll
            for (int q = 0; q < 4; ++q) {
                float o[32];
                tmem_ld32(tmem + lane_addr + kTmemO + q * 32, o);
                tmem_wait_ld();
                if (cascade && row_valid) {
                    float* dst = a.o_part + prow * kHead + q * 32;
#pragma unroll
                    for (int e = 0; e < 32; e += 4)
                        *reinterpret_cast<float4*>(dst + e) =
                            make_float4(o[e] * inv_l, o[e + 1] * inv_l, o[e + 2] * inv_l,
                                        o[e + 3] * inv_l);
                } else if (row_valid) {
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
    if (warp == kMmaWarp) {
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
    return launch_pdl(kern, grid, dim3(kThreads), kSmemBytes, stream, mq, mk, mv, a);
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
