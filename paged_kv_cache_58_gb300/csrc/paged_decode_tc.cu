// Paged decode for bf16 pools on the tensor cores (warp-level MMA).
//
// Same work split as the CUDA-core decode: one CTA per (partition, kv head, sequence), 4
// warps per CTA, warp w streams every 4th 16-token chunk of the partition through
// its own ring of shared-memory stages and keeps its own online-softmax state; the
// CTA merges the 4 states; a log-sum-exp combine merges partitions (split-KV
// decode, aifetchly SGLang guide, "Integrating FlashInfer").  The blocks are
// located through the block table (Triptych "Paged Attention for Efficient Memory
// Management": the kernel chases the block table).
//
// Why tensor cores in an HBM-bound kernel: with GQA the G query heads of a kv head
// read the same 16-token block, so per block the work is two small dense products,
//   S^T[16 tok x 8 heads] = K[16 x D] . q^T[D x 8]          (D/16 MMAs m16n8k16)
//   O^T[D x 8 heads]     += V^T[D x 16 tok] . P^T[16 x 8]    (D/16 MMAs, twice)
// which on CUDA cores cost ~50 issue slots per token and kv head and left the
// kernel issue-bound; as MMAs they cost ~5.  Tokens sit on the M side, heads on N
// (heads >= G are zero padding).  P^T comes out of the score accumulators in the
// wrong orientation and is transposed in registers with movmatrix; it is split into
// bf16 hi + lo parts so the probabilities keep ~2^-17 relative precision.
//
// Staging: the kernel walks 16-token chunks (a 16-token block, or half of a 32-token
// one); each chunk's K slab and V slab arrive as one TMA box each (under an L2
// evict-first policy, since no other CTA reads them), with the 128-byte
// swizzle so that ldmatrix reads them without bank conflicts: for head_dim 128 a 4-D
// box (the chunk's 16 rows x 256 B as 2 row groups x 2 column halves x 8 rows x 128 B),
// for head_dim 64 a 16-row x 64-column box.  The warp stays converged throughout: the
// stage waits vote across lanes and the copies are predicated, because reconverging a
// diverged warp costs hundreds of cycles on a busy scheduler.
//
// Fused append: with k_new / v_new set, the warp whose chunk holds a sequence's newest
// token overwrites that token's staged K and V rows with the input rows (the pool does
// not hold it yet) and stores the same bytes into the token's pool slot, so the step
// needs no separate append launch.
#include <cuda.h>
#include <cuda_runtime.h>

#include "common.cuh"
#include "kernels.h"

namespace pkv {

namespace {

constexpr int kWarps = 4;
constexpr int kThreads = kWarps * 32;
constexpr int kStages = 2;
constexpr int kBlk = 16;
constexpr int kAtom = 8 * 128;    // 8 rows x 128 B: one swizzle atom
constexpr float kLazyRescale = 8.0f;

PKV_DEVINL void ldsm_x4(uint32_t addr, uint32_t& r0, uint32_t& r1, uint32_t& r2, uint32_t& r3) {
    asm volatile("ldmatrix.sync.aligned.m8n8.x4.shared.b16 {%0,%1,%2,%3}, [%4];"
                 : "=r"(r0), "=r"(r1), "=r"(r2), "=r"(r3)
                 : "r"(addr));
}
PKV_DEVINL void ldsm_x4_t(uint32_t addr, uint32_t& r0, uint32_t& r1, uint32_t& r2,
                          uint32_t& r3) {
    asm volatile("ldmatrix.sync.aligned.m8n8.x4.trans.shared.b16 {%0,%1,%2,%3}, [%4];"
                 : "=r"(r0), "=r"(r1), "=r"(r2), "=r"(r3)
                 : "r"(addr));
}
PKV_DEVINL uint32_t movm_t(uint32_t x) {
    uint32_t y;
    asm volatile("movmatrix.sync.aligned.m8n8.trans.b16 %0, %1;" : "=r"(y) : "r"(x));
    return y;
}
// D = A (16x16 bf16, row) * B (16x8 bf16, col) + D, fp32 accumulate.
PKV_DEVINL void mma_bf16(float (&d)[4], uint32_t a0, uint32_t a1, uint32_t a2, uint32_t a3,
                         uint32_t b0, uint32_t b1) {
    asm volatile(
        "mma.sync.aligned.m16n8k16.row.col.f32.bf16.bf16.f32 {%0,%1,%2,%3}, {%4,%5,%6,%7}, "
        "{%8,%9}, {%0,%1,%2,%3};"
        : "+f"(d[0]), "+f"(d[1]), "+f"(d[2]), "+f"(d[3])
        : "r"(a0), "r"(a1), "r"(a2), "r"(a3), "r"(b0), "r"(b1));
}

// Address of 16-byte chunk `c` (0 .. D/8-1) of row `t` (0..15) of a slab staged as
// [row group t/8][column half c/8][8 rows][128 B] with the 128-byte swizzle (chunk
// index XOR row % 8).
template <int D>
PKV_DEVINL uint32_t slab_addr(uint32_t base, int t, int c) {
    return base + (t >> 3) * (D / 64) * kAtom + (c >> 3) * kAtom + (t & 7) * 128 +
           (((c & 7) ^ (t & 7)) << 4);
}

template <int D, int G>
struct TcSmem {
    static constexpr int kHalves = D / 64;
    static constexpr int kSlab = kBlk * D * 2;            // K or V slab of one block
    static constexpr int kStageBytes = 2 * kSlab;
    static constexpr int kRing = kWarps * kStages * kStageBytes;
    // merge scratch reuses the ring once every warp is done
    static constexpr int kMerge = kWarps * G * D * 4 + 2 * kWarps * G * 4;
    static_assert(kMerge <= kRing, "merge scratch must fit in the ring");
    static constexpr int kBars = kWarps * kStages * 8;
    static constexpr int kTotal = kRing + kBars + 1024;   // + alignment slack
};

template <int D, int G>
__global__ void __launch_bounds__(kThreads)
decode_tc_kernel(const __grid_constant__ CUtensorMap tm_k, const __grid_constant__ CUtensorMap tm_v,
                 const DecodeArgs a) {
    using SM = TcSmem<D, G>;
    constexpr int KS = D / 16;  // k-steps of the score MMA == m-tiles of the P.V MMA
    extern __shared__ uint8_t smem_raw[];
    uint8_t* smem = reinterpret_cast<uint8_t*>(
        (reinterpret_cast<uintptr_t>(smem_raw) + 1023) & ~static_cast<uintptr_t>(1023));

    griddep_wait();
    griddep_launch_dependents();
    // Grid (kv head, sequence, partition), partition slowest: CTAs are placed in index
    // order, so every sequence's first (mostly full-length) partition starts before any
    // second one and the last wave holds only the short final partitions of the longest
    // sequences: an approximate longest-first order that shortens the tail.
    const int kvh = blockIdx.x;
    const int seq = blockIdx.y;
    const int part = blockIdx.z;
    const int warp = threadIdx.x >> 5;
    const int lane = threadIdx.x & 31;

    const int32_t* bt = a.block_tables + static_cast<size_t>(seq) * a.max_blocks_per_seq;
    const int b0 = a.chunk_offset + part * a.partition_chunks;
    const int my_first = b0 + warp;
    // The partition's start does not depend on the context length, so the block ids of
    // this warp's first 32 chunks are loaded together with it rather than after it (one
    // dependent round trip less before the first copy); ids past the sequence's end are
    // loaded from inside the table row and then ignored.
    int ids0;
    {
        const int e = (my_first + lane * kWarps) >> a.chunk_shift;
        ids0 = e < a.max_blocks_per_seq ? __ldg(bt + e) : -1;
    }
    int L = a.context_lens[seq];
    const int span_end = a.chunk_offset + a.max_parts * a.partition_chunks;  // chunks covered
    const int max_chunks = a.max_blocks_per_seq << a.chunk_shift;
    bool append = a.k_new != nullptr;
    if (L > max_chunks * kBlk || L > span_end * kBlk) {
        if (part == 0 && threadIdx.x == 0) raise_status(a.status, PKV_ERR_OOB);
        L = min(max_chunks, span_end) * kBlk;
        append = false;   // the clamped end is not the new token
    }
    const int nblk = (L + kBlk - 1) / kBlk;
    if (L <= 0 || b0 >= nblk) {   // uniform over the CTA, before any barrier
        // A fused append in a cascade decode needs the newest token in the private
        // suffix; one inside the shared prefix is not stored: report it.
        if (append && part == 0 && threadIdx.x == 0 && L > 0 && nblk <= a.chunk_offset)
            raise_status(a.status, PKV_ERR_INVALID);
        // A context length below 1 is outside the contract (a query sees at least its own
        // key): report it, and give the sequence's rows zeros rather than stale memory.
        if (L <= 0 && part == 0 && threadIdx.x == 0) raise_status(a.status, PKV_ERR_INVALID);
        if (L <= 0 && part == 0 && a.chunk_offset == 0)
            zero_invalid_rows(a, seq, kvh, G, D, 2);   // bf16 output
        return;
    }
    const int b1 = min(nblk, b0 + a.partition_chunks);
    const int my_count = my_first < b1 ? (b1 - my_first + kWarps - 1) / kWarps : 0;

    uint8_t* ring = smem + warp * kStages * SM::kStageBytes;
    uint64_t* bars = reinterpret_cast<uint64_t*>(smem + SM::kRing) + warp * kStages;

    if (lane == 0) {   // once per CTA
        prefetch_tmap(&tm_k);
        prefetch_tmap(&tm_v);
#pragma unroll
        for (int i = 0; i < kStages; ++i) mbar_init(&bars[i], 1);
        fence_mbar_init();
        fence_proxy_async_smem();
    }
    __syncwarp();

    const uint64_t stream_policy = l2_policy_evict_first();   // K/V are read once
    int ids = -1;
    auto fetch_ids = [&](int base) {
        const int i = base + lane;
        ids = (i < my_count) ? __ldg(bt + ((my_first + i * kWarps) >> a.chunk_shift)) : -1;
    };
    ids = lane < my_count ? ids0 : -1;

    // Stage i: lane 0 sets the byte count, lane 0 copies the K slab and lane 1 the V
    // slab; all lanes execute the predicated instructions (no branch).
    auto issue = [&](int i, int phys, bool on) {
        uint8_t* st = ring + (i % kStages) * SM::kStageBytes;
        uint64_t* bar = &bars[i % kStages];
        const bool bad = phys < 0 || phys >= a.num_blocks;
        if (on && bad && lane == 0) raise_status(a.status, PKV_ERR_OOB);
        mbar_arrive_if(on && bad && lane == 0, bar);  // complete the phase without data
        const int ci = my_first + i * kWarps;   // chunk: rows 16 (ci & mask) of its block
        const int row = ((bad ? kvh : phys * a.num_kv_heads + kvh) << a.chunk_shift) * kBlk +
                        (ci & ((1 << a.chunk_shift) - 1)) * kBlk;
        const bool stall = a.test_stall && i == 0 && warp == 0 && blockIdx.x == 0 &&
                           blockIdx.y == 0 && blockIdx.z == 0;
        mbar_arrive_expect_tx_if(on && !bad && lane == 0, bar,
                                 SM::kStageBytes + (stall ? 16u : 0u));
        const bool mine = on && !bad && lane < 2;
        uint8_t* dst = st + (lane == 1 ? SM::kSlab : 0);
        const void* map = lane == 1 ? static_cast<const void*>(&tm_v) : &tm_k;
        if constexpr (D == 128)
            tma_load_4d_hint_if(mine, dst, map, 0, 0, 0, row / 8, bar, stream_policy);
        else
            tma_load_2d_hint_if(mine, dst, map, 0, row, bar, stream_policy);
    };

#pragma unroll
    for (int i = 0; i < kStages; ++i) issue(i, __shfl_sync(0xffffffffu, ids, i), i < my_count);

    // q^T as the B operand of the score MMA: lane holds head lane/4 (zero if >= G),
    // dims 16ks + 2(lane%4) + {0,1} (b0) and +8 (b1).
    const int qh = lane >> 2;
    const int qd = 2 * (lane & 3);
    uint32_t qb[KS][2];
    {
        const uint16_t* qrow = static_cast<const uint16_t*>(a.q) +
                               (static_cast<size_t>(seq) * a.num_q_heads + kvh * G + qh) * D;
#pragma unroll
        for (int ks = 0; ks < KS; ++ks) {
            if (qh < G) {
                qb[ks][0] = __ldg(reinterpret_cast<const uint32_t*>(qrow + 16 * ks + qd));
                qb[ks][1] = __ldg(reinterpret_cast<const uint32_t*>(qrow + 16 * ks + qd + 8));
            } else {
                qb[ks][0] = 0u;
                qb[ks][1] = 0u;
            }
        }
    }

    // O^T accumulators: m-tile mt, c0/c1 = (d = 16mt + lane/4, heads h0/h1),
    // c2/c3 = (d + 8, heads h0/h1); h0 = 2(lane%4), h1 = h0 + 1.
    float acc[KS][4];
#pragma unroll
    for (int mt = 0; mt < KS; ++mt)
#pragma unroll
        for (int e = 0; e < 4; ++e) acc[mt][e] = 0.f;
    float m_used[2] = {-INFINITY, -INFINITY};
    float l_part[2] = {0.f, 0.f};   // this lane's share of the denominators of h0, h1
    const float sl2 = a.scale_log2;
    const int t_lo = lane >> 2;     // score rows held: tokens t_lo and t_lo + 8

    // ldmatrix row addresses (per lane): matrix mi = lane / 8, row r = lane % 8.
    const int mi = lane >> 3;
    const int rr = lane & 7;
    const int k_tok = (mi & 1) * 8 + rr;     // K as A: tokens (mi&1)*8 + r, chunk 2ks + mi/2
    const int k_chk = mi >> 1;
    const int v_tok = (mi >> 1) * 8 + rr;    // V^T as A: tokens (mi>>1)*8 + r, chunk 2mt + mi&1
    const int v_chk = mi & 1;

    int failed_at = -1;
    for (int i = 0; i < my_count; ++i) {
        const int st_i = i % kStages;
        if (!mbar_wait_warp(&bars[st_i], (i / kStages) & 1, a.status)) {
            failed_at = i;
            break;
        }
        const uint32_t kbase = smem_u32(ring + st_i * SM::kStageBytes);
        const uint32_t vbase = kbase + SM::kSlab;
        const int blk = my_first + i * kWarps;
        const int valid = min(kBlk, L - blk * kBlk);

        const bool fuse = append && blk == nblk - 1;   // holds the new token, row valid - 1
        if (valid < kBlk || fuse) {
            uint8_t* stage = ring + st_i * SM::kStageBytes;
            // Rows past the context may hold anything (NaN included): zero their V so
            // that a zero probability contributes exactly zero.
            for (int idx = lane; idx < (kBlk - valid) * SM::kHalves * 8; idx += 32) {
                const int t = valid + idx / (SM::kHalves * 8);
                const int c = idx % (SM::kHalves * 8);
                *reinterpret_cast<uint4*>(stage + SM::kSlab +
                                          (slab_addr<D>(kbase, t, c) - kbase)) =
                    make_uint4(0, 0, 0, 0);
            }
            if (fuse) {
                // The new token: lane -> (K or V, 16-byte piece c) of its row; it replaces
                // the staged row and is stored into the pool slot (a plain copy, the same
                // bits kv_append writes).
                constexpr int kPieces = D / 8;
                const int phys = __ldg(bt + (blk >> a.chunk_shift));
                if (lane < 2 * kPieces) {
                    const int which = lane / kPieces;
                    const int c = lane % kPieces;
                    const uint4 x = __ldg(static_cast<const uint4*>(which ? a.v_new : a.k_new) +
                                          (static_cast<size_t>(seq) * a.num_kv_heads + kvh) *
                                              kPieces + c);
                    *reinterpret_cast<uint4*>(stage + which * SM::kSlab +
                                              (slab_addr<D>(kbase, valid - 1, c) - kbase)) = x;
                    if (phys >= 0 && phys < a.num_blocks) {
                        const size_t row =
                            ((((static_cast<size_t>(phys) * a.num_kv_heads + kvh)
                               << a.chunk_shift) + (blk & ((1 << a.chunk_shift) - 1))) * kBlk) +
                            valid - 1;
                        uint4* pool = static_cast<uint4*>(const_cast<void*>(which ? a.v_pool
                                                                                  : a.k_pool));
                        pool[row * kPieces + c] = x;
                    }
                }
            }
            fence_proxy_async_smem();
            __syncwarp();
        }

        // S^T = K . q^T
        float s[4] = {0.f, 0.f, 0.f, 0.f};
#pragma unroll
        for (int ks = 0; ks < KS; ++ks) {
            uint32_t a0, a1, a2, a3;
            ldsm_x4(slab_addr<D>(kbase, k_tok, 2 * ks + k_chk), a0, a1, a2, a3);
            mma_bf16(s, a0, a1, a2, a3, qb[ks][0], qb[ks][1]);
        }
#pragma unroll
        for (int e = 0; e < 4; ++e) {
            const int t = t_lo + ((e & 2) ? 8 : 0);
            s[e] = (t < valid) ? s[e] * sl2 : -INFINITY;
        }
        // per-head block max over the 16 tokens (lanes sharing lane % 4)
        float mx[2] = {fmaxf(s[0], s[2]), fmaxf(s[1], s[3])};
#pragma unroll
        for (int o = 4; o < 32; o <<= 1) {
            mx[0] = fmaxf(mx[0], __shfl_xor_sync(0xffffffffu, mx[0], o));
            mx[1] = fmaxf(mx[1], __shfl_xor_sync(0xffffffffu, mx[1], o));
        }
        float alpha[2];
        bool grow = false;
#pragma unroll
        for (int h = 0; h < 2; ++h) {
            const bool g = mx[h] > m_used[h] + kLazyRescale;
            const float m_cur = g ? mx[h] : m_used[h];
            alpha[h] = fast_exp2(m_used[h] - m_cur);
            m_used[h] = m_cur;
            grow |= g;
        }
        float p[4];
#pragma unroll
        for (int e = 0; e < 4; ++e) p[e] = fast_exp2(s[e] - m_used[e & 1]);
        l_part[0] = l_part[0] * alpha[0] + p[0] + p[2];
        l_part[1] = l_part[1] * alpha[1] + p[1] + p[3];
        if (__any_sync(0xffffffffu, grow)) {
#pragma unroll
            for (int mt = 0; mt < KS; ++mt) {
                acc[mt][0] *= alpha[0];
                acc[mt][1] *= alpha[1];
                acc[mt][2] *= alpha[0];
                acc[mt][3] *= alpha[1];
            }
        }
        // P^T fragments: [token][head] 8x8 tiles transposed in registers; hi + lo parts.
        const uint32_t h01 = pack_bf16x2(p[0], p[1]);
        const uint32_t h23 = pack_bf16x2(p[2], p[3]);
        const uint32_t l01 = pack_bf16x2(p[0] - bf16lo_to_f32(h01), p[1] - bf16hi_to_f32(h01));
        const uint32_t l23 = pack_bf16x2(p[2] - bf16lo_to_f32(h23), p[3] - bf16hi_to_f32(h23));
        const uint32_t bh0 = movm_t(h01), bh1 = movm_t(h23);
        const uint32_t bl0 = movm_t(l01), bl1 = movm_t(l23);
        // O^T += V^T . P^T
#pragma unroll
        for (int mt = 0; mt < KS; ++mt) {
            uint32_t a0, a1, a2, a3;
            ldsm_x4_t(slab_addr<D>(vbase, v_tok, 2 * mt + v_chk), a0, a1, a2, a3);
            mma_bf16(acc[mt], a0, a1, a2, a3, bh0, bh1);
            mma_bf16(acc[mt], a0, a1, a2, a3, bl0, bl1);
        }
        __syncwarp();
        const int nxt = i + kStages;
        if ((nxt & 31) == 0 && nxt < my_count) fetch_ids(nxt);
        issue(nxt, __shfl_sync(0xffffffffu, ids, nxt & 31), nxt < my_count);
    }
    if (failed_at >= 0) {
        for (int j = failed_at + 1; j < my_count && j < failed_at + kStages; ++j)
            mbar_wait_warp(&bars[j % kStages], (j / kStages) & 1, a.status);
    }

    // full denominators of h0, h1 over this warp's tokens
#pragma unroll
    for (int o = 4; o < 32; o <<= 1) {
        l_part[0] += __shfl_xor_sync(0xffffffffu, l_part[0], o);
        l_part[1] += __shfl_xor_sync(0xffffffffu, l_part[1], o);
    }
    __syncthreads();  // every warp is done with its ring: reuse it as merge scratch
    float* macc = reinterpret_cast<float*>(smem);            // [W][G][D]
    float* mm = macc + kWarps * G * D;                       // [W][G]
    float* ml = mm + kWarps * G;                             // [W][G]
    const int h0 = 2 * (lane & 3);
#pragma unroll
    for (int hh = 0; hh < 2; ++hh) {
        const int h = h0 + hh;
        if (h < G) {
#pragma unroll
            for (int mt = 0; mt < KS; ++mt) {
                macc[(warp * G + h) * D + 16 * mt + t_lo] = acc[mt][hh];
                macc[(warp * G + h) * D + 16 * mt + t_lo + 8] = acc[mt][2 + hh];
            }
            if (t_lo == 0) {
                mm[warp * G + h] = my_count > 0 ? m_used[hh] : -INFINITY;
                ml[warp * G + h] = my_count > 0 ? l_part[hh] : 0.f;
            }
        }
    }
    __syncthreads();

    const int nparts = a.max_parts + a.extra_parts;   // partial slots per row
    for (int idx = threadIdx.x; idx < G * D; idx += kThreads) {
        const int g = idx / D;
        const int d = idx % D;
        float M = -INFINITY;
#pragma unroll
        for (int w = 0; w < kWarps; ++w) M = fmaxf(M, mm[w * G + g]);
        float o = 0.f, l = 0.f;
#pragma unroll
        for (int w = 0; w < kWarps; ++w) {
            const float f = fast_exp2(mm[w * G + g] - M);
            o = fmaf(f, macc[(w * G + g) * D + d], o);
            l = fmaf(f, ml[w * G + g], l);
        }
        const size_t row = static_cast<size_t>(seq) * a.num_q_heads + kvh * G + g;
        if (nparts == 1) {
            static_cast<uint16_t*>(a.out)[row * D + d] =
                static_cast<uint16_t>(pack_bf16x2(o / l, 0.f) & 0xffffu);
        } else {
            const size_t pr = row * nparts + a.extra_parts + part;
            a.o_part[pr * D + d] = o / l;
            if (d == 0) {
                a.m_part[pr] = M;
                a.l_part[pr] = l;
            }
        }
    }
}

template <int D, int G>
cudaError_t launch_tc(const DecodeArgs& a, cudaStream_t stream) {
    using SM = TcSmem<D, G>;
    CUtensorMap mk, mv;
    const int64_t rows = a.num_blocks * a.num_kv_heads * (kBlk << a.chunk_shift);
    const bool maps_ok = D == 128 ? make_pool_block_map(&mk, a.k_pool, rows) &&
                                        make_pool_block_map(&mv, a.v_pool, rows)
                                  : make_pool_map(&mk, a.k_pool, rows, D) &&
                                        make_pool_map(&mv, a.v_pool, rows, D);
    if (!maps_ok) return cudaErrorInvalidValue;
    auto kern = decode_tc_kernel<D, G>;
    cudaError_t e =
        set_smem_once(reinterpret_cast<const void*>(kern), SM::kTotal);
    if (e != cudaSuccess) return e;
    if (a.max_parts > 0) {   // zero when a cascade decode has no private suffix at all
        dim3 grid(a.num_kv_heads, a.num_seqs, a.max_parts);
        e = launch_maybe_pdl(!a.no_pdl, kern, grid, dim3(kThreads), SM::kTotal, stream, mk, mv,
                             a);
        if (e != cudaSuccess) return e;
    }
    if (a.extra_parts == 0 && a.max_parts == 1) return e;  // output written directly
    if (a.defer_combine) return e;
    return launch_decode_combine(a, PKV_BF16, D, stream);
}

template <int D>
cudaError_t launch_tc_group(const DecodeArgs& a, int G, cudaStream_t stream) {
    switch (G) {
        case 1: return launch_tc<D, 1>(a, stream);
        case 2: return launch_tc<D, 2>(a, stream);
        case 4: return launch_tc<D, 4>(a, stream);
        case 8: return launch_tc<D, 8>(a, stream);
        default: return cudaErrorInvalidValue;
    }
}

}  // namespace

cudaError_t launch_paged_decode_tc(const DecodeArgs& a, int head_dim, int group,
                                   cudaStream_t stream) {
    if (head_dim == 128) return launch_tc_group<128>(a, group, stream);
    if (head_dim == 64) return launch_tc_group<64>(a, group, stream);
    return cudaErrorInvalidValue;
}

}  // namespace pkv
