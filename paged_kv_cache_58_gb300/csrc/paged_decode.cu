// Paged decode: one query token per sequence over a block-table-addressed KV pool.
//
// The attention kernel "walks the block table and gathers the relevant physical
// blocks" (Triptych "Paged Attention for Efficient Memory Management", body) and
// long contexts are split across thread blocks with a log-sum-exp merge (split-KV
// decode, aifetchly SGLang guide, "Integrating FlashInfer").  The arithmetic is
// ordinary softmax attention; only the addressing is paged.
//
// Grid: (partition, kv head, sequence).  A CTA owns `partition_chunks` consecutive
// 16-token chunks of one (sequence, kv head) -- a chunk is a 16-token block, or half
// of a 32-token one -- and serves the G = Hq / Hkv query heads that read that kv head,
// so each K/V byte is fetched from HBM once per step.  Inside the CTA each of the 4
// warps streams every 4th chunk of the partition through its own ring of
// shared-memory stages filled by 1-D bulk-async copies (one 16-token K slab and one V
// slab per stage, both contiguous in the pool layout), and keeps its own fp32
// online-softmax state; the 4 states are merged through shared memory at the end.
//
// Lane mapping for one 16-token block: the two half-warps take alternate token
// rows; lane c of a half-warp owns elements [c*NE, c*NE+NE) of D (NE = D/16).
// Scores: each lane forms G partial dot products, then a reduce-scatter over the
// 16 lanes (xor 8, 4, 2, 1; each step halves the number of values a lane keeps)
// leaves lane c holding the full score of head hl(c) = c / (16/G).  P.V: each lane
// accumulates acc[G][NE] for its D slice, fetching p of head g from lane g*(16/G).
#include <cuda_runtime.h>

#include "common.cuh"
#include "kernels.h"

namespace pkv {

namespace {

constexpr int kWarps = 4;
constexpr int kThreads = kWarps * 32;
constexpr int kStages = 3;
constexpr int kBlock = 16;

template <typename T, int NE>
PKV_DEVINL void load_chunk(const T* src, float (&x)[NE]) {
    if constexpr (sizeof(T) == 2) {
        if constexpr (NE == 8) {
            const uint4 w = *reinterpret_cast<const uint4*>(src);
            x[0] = bf16lo_to_f32(w.x); x[1] = bf16hi_to_f32(w.x);
            x[2] = bf16lo_to_f32(w.y); x[3] = bf16hi_to_f32(w.y);
            x[4] = bf16lo_to_f32(w.z); x[5] = bf16hi_to_f32(w.z);
            x[6] = bf16lo_to_f32(w.w); x[7] = bf16hi_to_f32(w.w);
        } else {
            const uint2 w = *reinterpret_cast<const uint2*>(src);
            x[0] = bf16lo_to_f32(w.x); x[1] = bf16hi_to_f32(w.x);
            x[2] = bf16lo_to_f32(w.y); x[3] = bf16hi_to_f32(w.y);
        }
    } else {
#pragma unroll
        for (int i = 0; i < NE; i += 4) {
            const float4 f = *reinterpret_cast<const float4*>(src + i);
            x[i] = f.x; x[i + 1] = f.y; x[i + 2] = f.z; x[i + 3] = f.w;
        }
    }
}

template <typename T>
PKV_DEVINL void store_elem(T* dst, float v);
template <>
PKV_DEVINL void store_elem<float>(float* dst, float v) { *dst = v; }
template <>
PKV_DEVINL void store_elem<uint16_t>(uint16_t* dst, float v) {
    *dst = static_cast<uint16_t>(pack_bf16x2(v, 0.f) & 0xffffu);
}

// Reduce-scatter of G per-lane partial sums over the 16 lanes of a half-warp.
// Returns the full sum of head (lane & 15) / (16 / G).
template <int G>
PKV_DEVINL float reduce_scatter16(float (&v)[G], int lane) {
    if constexpr (G == 1) {
        float a = v[0];
        a += __shfl_xor_sync(0xffffffffu, a, 8);
        a += __shfl_xor_sync(0xffffffffu, a, 4);
        a += __shfl_xor_sync(0xffffffffu, a, 2);
        a += __shfl_xor_sync(0xffffffffu, a, 1);
        return a;
    } else {
        constexpr int H = G / 2;
        const bool upper = (lane & 8) != 0;
        float w[H];
#pragma unroll
        for (int i = 0; i < H; ++i) {
            const float keep = upper ? v[i + H] : v[i];
            const float send = upper ? v[i] : v[i + H];
            w[i] = keep + __shfl_xor_sync(0xffffffffu, send, 8);
        }
        if constexpr (H == 1) {
            float a = w[0];
            a += __shfl_xor_sync(0xffffffffu, a, 4);
            a += __shfl_xor_sync(0xffffffffu, a, 2);
            a += __shfl_xor_sync(0xffffffffu, a, 1);
            return a;
        } else {
            constexpr int H2 = H / 2;
            const bool up2 = (lane & 4) != 0;
            float u[H2];
#pragma unroll
            for (int i = 0; i < H2; ++i) {
                const float keep = up2 ? w[i + H2] : w[i];
                const float send = up2 ? w[i] : w[i + H2];
                u[i] = keep + __shfl_xor_sync(0xffffffffu, send, 4);
            }
            if constexpr (H2 == 1) {
                float a = u[0];
                a += __shfl_xor_sync(0xffffffffu, a, 2);
                a += __shfl_xor_sync(0xffffffffu, a, 1);
                return a;
            } else {  // G == 8
                const bool up3 = (lane & 2) != 0;
                const float keep = up3 ? u[1] : u[0];
                const float send = up3 ? u[0] : u[1];
                float a = keep + __shfl_xor_sync(0xffffffffu, send, 2);
                a += __shfl_xor_sync(0xffffffffu, a, 1);
                return a;
            }
        }
    }
}

// Fused append: the new token, row `r` of chunk `blk` (of sequence `seq`, kv head
// `kvh`), replaces that row in the staged K and V slabs and is stored into its pool slot:
// a plain copy of the bits kv_append writes.  Lane p handles 16-byte pieces p, p + 32, ..
// of the K row then the V row (kPieces per row).  Kept out of line: it runs once per
// sequence and kv head, and inlined it costs the streaming loop registers.
template <int kPieces>
__device__ __noinline__ void append_row(const void* k_new, const void* v_new, void* k_pool,
                                        void* v_pool, uint8_t* stage, int slab_bytes, int phys,
                                        int64_t num_blocks, int num_kv_heads, int chunk_shift,
                                        int seq, int kvh, int blk, int r, int lane) {
    const size_t row = ((((static_cast<size_t>(phys) * num_kv_heads + kvh) << chunk_shift) +
                         (blk & ((1 << chunk_shift) - 1))) * kBlock) + r;
    const size_t src = (static_cast<size_t>(seq) * num_kv_heads + kvh) * kPieces;
    for (int p = lane; p < 2 * kPieces; p += 32) {
        const int which = p / kPieces;
        const int pc = p % kPieces;
        const uint4 x = __ldg(static_cast<const uint4*>(which ? v_new : k_new) + src + pc);
        reinterpret_cast<uint4*>(stage + which * slab_bytes)[r * kPieces + pc] = x;
        if (phys >= 0 && phys < num_blocks)
            static_cast<uint4*>(which ? v_pool : k_pool)[row * kPieces + pc] = x;
    }
    fence_proxy_async_smem();
}

template <typename T, int D, int G>
struct DecodeSmem {
    static constexpr int kSlab = kBlock * D * static_cast<int>(sizeof(T));
    static constexpr int kStageBytes = 2 * kSlab;
    static constexpr int kRing = kWarps * kStages * kStageBytes;
    static constexpr int kMergeAcc = kWarps * G * D * 4;
    static constexpr int kMergeML = 2 * kWarps * G * 4;
    static constexpr int kBars = kWarps * kStages * 8;
    static constexpr int kTotal = kRing + kMergeAcc + kMergeML + kBars;
};

template <typename T, int D, int G>
__global__ void __launch_bounds__(kThreads)
decode_split_kernel(const DecodeArgs a) {
    using SM = DecodeSmem<T, D, G>;
    constexpr int NE = D / 16;
    extern __shared__ __align__(128) uint8_t smem[];

    griddep_wait();
    griddep_launch_dependents();
    const int kvh = blockIdx.y;
    const int part = blockIdx.x;
    const int seq = blockIdx.z;   // table row
    const size_t qrow = static_cast<size_t>(seq);
    const int warp = threadIdx.x >> 5;
    const int lane = threadIdx.x & 31;
    const int hw = lane >> 4;   // half-warp: token parity
    const int c = lane & 15;    // D slice

    int L = a.context_lens[seq];
    const int span_end = a.chunk_offset + a.max_parts * a.partition_chunks;  // chunks covered
    const int max_chunks = a.max_blocks_per_seq << a.chunk_shift;
    bool append = a.k_new != nullptr;
    if (L > max_chunks * kBlock || L > span_end * kBlock) {
        if (part == 0 && threadIdx.x == 0) raise_status(a.status, PKV_ERR_OOB);
        L = min(max_chunks, span_end) * kBlock;
        append = false;   // the clamped end is not the new token
    }
    const int nblk = (L + kBlock - 1) / kBlock;
    const int b0 = a.chunk_offset + part * a.partition_chunks;
    if (L <= 0 || b0 >= nblk) {   // uniform over the CTA, before any barrier
        // A fused append in a cascade decode needs the newest token in the private
        // suffix; one inside the shared prefix is not stored: report it.
        if (append && part == 0 && threadIdx.x == 0 && L > 0 && nblk <= a.chunk_offset)
            raise_status(a.status, PKV_ERR_INVALID);
        // A context length below 1 is outside the contract (a query sees at least its own
        // key): report it, and give the sequence's rows zeros rather than stale memory.
        if (L <= 0 && part == 0 && threadIdx.x == 0) raise_status(a.status, PKV_ERR_INVALID);
        if (L <= 0 && part == 0 && a.chunk_offset == 0)
            zero_invalid_rows(a, seq, kvh, G, D, static_cast<int>(sizeof(T)));
        return;
    }
    const int b1 = min(nblk, b0 + a.partition_chunks);
    const int my_first = b0 + warp;
    const int my_count = my_first < b1 ? (b1 - my_first + kWarps - 1) / kWarps : 0;

    uint8_t* ring = smem + warp * kStages * SM::kStageBytes;
    float* macc = reinterpret_cast<float*>(smem + SM::kRing);             // [W][G][D]
    float* mm = reinterpret_cast<float*>(smem + SM::kRing + SM::kMergeAcc);  // [W][G]
    float* ml = mm + kWarps * G;                                          // [W][G]
    uint64_t* bars = reinterpret_cast<uint64_t*>(smem + SM::kRing + SM::kMergeAcc + SM::kMergeML) +
                     warp * kStages;

    const T* kpool = static_cast<const T*>(a.k_pool);
    const T* vpool = static_cast<const T*>(a.v_pool);
    const int32_t* bt = a.block_tables + static_cast<size_t>(seq) * a.max_blocks_per_seq;

    if (lane == 0) {
#pragma unroll
        for (int i = 0; i < kStages; ++i) mbar_init(&bars[i], 1);
        fence_mbar_init();
        fence_proxy_async_smem();
    }
    __syncwarp();

    // Physical ids of this warp's blocks, 32 at a time, one per lane.
    int ids = -1;
    auto fetch_ids = [&](int base) {
        const int i = base + lane;
        ids = (i < my_count) ? __ldg(bt + ((my_first + i * kWarps) >> a.chunk_shift)) : -1;
    };
    fetch_ids(0);

    const uint64_t stream_policy = l2_policy_evict_first();   // K/V are read once
    auto issue = [&](int i, int phys) {  // lane 0 only
        uint8_t* st = ring + (i % kStages) * SM::kStageBytes;
        uint64_t* bar = &bars[i % kStages];
        if (phys < 0 || phys >= a.num_blocks) {
            raise_status(a.status, PKV_ERR_OOB);
            mbar_arrive(bar);  // complete the phase without data; output is invalid
            return;
        }
        const int ci = my_first + i * kWarps;   // chunk: rows 16 (ci & mask) of its block
        const size_t off = (((static_cast<size_t>(phys) * a.num_kv_heads + kvh) << a.chunk_shift) +
                            (ci & ((1 << a.chunk_shift) - 1))) * kBlock * D;
        // test hook: 16 bytes more than the copies deliver (see DecodeArgs::test_stall)
        const bool stall = a.test_stall && i == 0 && warp == 0 && blockIdx.x == 0 &&
                           blockIdx.y == 0 && blockIdx.z == 0;
        mbar_arrive_expect_tx(bar, SM::kStageBytes + (stall ? 16u : 0u));
        bulk_g2s_hint(st, kpool + off, SM::kSlab, bar, stream_policy);
        bulk_g2s_hint(st + SM::kSlab, vpool + off, SM::kSlab, bar, stream_policy);
    };

    // Prologue: fill the ring.
#pragma unroll
    for (int i = 0; i < kStages; ++i) {
        const int id = __shfl_sync(0xffffffffu, ids, i);
        if (lane == 0 && i < my_count) issue(i, id);
    }

    // Query slice of the G heads, pre-scaled by scale * log2(e) so that scores
    // are in the exp2 domain.
    const int hq = a.num_q_heads;
    float qf[G][NE];
    {
        const T* qbase = static_cast<const T*>(a.q) +
                         (qrow * hq + kvh * G) * D + c * NE;
#pragma unroll
        for (int g = 0; g < G; ++g) {
            load_chunk<T, NE>(qbase + g * D, qf[g]);
#pragma unroll
            for (int e = 0; e < NE; ++e) qf[g][e] *= a.scale_log2;
        }
    }

    float acc[G][NE];
#pragma unroll
    for (int g = 0; g < G; ++g)
#pragma unroll
        for (int e = 0; e < NE; ++e) acc[g][e] = 0.f;
    float m_run = -INFINITY;  // running max of head hl (replicated over lanes of hl)
    float l_run = 0.f;
    constexpr int kHeadStride = 16 / G;
    const int src_base = lane & 16;

    int failed_at = -1;
    for (int i = 0; i < my_count; ++i) {
        const int st_i = i % kStages;
        if (!mbar_wait(&bars[st_i], (i / kStages) & 1, a.status)) {
            failed_at = i;
            break;
        }
        const T* K = reinterpret_cast<const T*>(ring + st_i * SM::kStageBytes);
        const T* V = reinterpret_cast<const T*>(ring + st_i * SM::kStageBytes + SM::kSlab);
        const int blk = my_first + i * kWarps;
        const int valid = min(kBlock, L - blk * kBlock);
        if (append && blk == nblk - 1) {
            append_row<D * static_cast<int>(sizeof(T)) / 16>(
                a.k_new, a.v_new, const_cast<void*>(a.k_pool), const_cast<void*>(a.v_pool),
                ring + st_i * SM::kStageBytes, SM::kSlab, __ldg(bt + (blk >> a.chunk_shift)),
                a.num_blocks, a.num_kv_heads, a.chunk_shift, seq, kvh, blk, valid - 1, lane);
            __syncwarp();
        }

        float sc[8];
#pragma unroll
        for (int r = 0; r < 8; ++r) {
            const int row = hw + 2 * r;
            float kf[NE];
            load_chunk<T, NE>(K + row * D + c * NE, kf);
            float part_[G];
#pragma unroll
            for (int g = 0; g < G; ++g) {
                float s = 0.f;
#pragma unroll
                for (int e = 0; e < NE; ++e) s = fmaf(qf[g][e], kf[e], s);
                part_[g] = s;
            }
            const float full = reduce_scatter16<G>(part_, lane);
            sc[r] = (row < valid) ? full : -INFINITY;
        }

        float bmax = sc[0];
#pragma unroll
        for (int r = 1; r < 8; ++r) bmax = fmaxf(bmax, sc[r]);
        bmax = fmaxf(bmax, __shfl_xor_sync(0xffffffffu, bmax, 16));
        const float m_new = fmaxf(m_run, bmax);
        const float alpha = fast_exp2(m_run - m_new);
        float psum = 0.f;
#pragma unroll
        for (int r = 0; r < 8; ++r) {
            sc[r] = fast_exp2(sc[r] - m_new);
            psum += sc[r];
        }
        psum += __shfl_xor_sync(0xffffffffu, psum, 16);
        l_run = l_run * alpha + psum;
        m_run = m_new;

#pragma unroll
        for (int g = 0; g < G; ++g) {
            const float ag = __shfl_sync(0xffffffffu, alpha, src_base | (g * kHeadStride));
#pragma unroll
            for (int e = 0; e < NE; ++e) acc[g][e] *= ag;
        }
#pragma unroll
        for (int r = 0; r < 8; ++r) {
            const int row = hw + 2 * r;
            float pg[G];
#pragma unroll
            for (int g = 0; g < G; ++g)
                pg[g] = __shfl_sync(0xffffffffu, sc[r], src_base | (g * kHeadStride));
            if (row < valid) {  // rows past the context may hold anything, even NaN
                float vf[NE];
                load_chunk<T, NE>(V + row * D + c * NE, vf);
#pragma unroll
                for (int g = 0; g < G; ++g)
#pragma unroll
                    for (int e = 0; e < NE; ++e) acc[g][e] = fmaf(pg[g], vf[e], acc[g][e]);
            }
        }
        __syncwarp();
        const int nxt = i + kStages;
        if ((nxt & 31) == 0 && nxt < my_count) fetch_ids(nxt);
        const int id = __shfl_sync(0xffffffffu, ids, nxt & 31);
        if (lane == 0 && nxt < my_count) issue(nxt, id);
    }
    if (failed_at >= 0) {
        // A copy never landed: wait (bounded) for the copies still in flight so none
        // lands after the CTA exits; the status word marks the output invalid.
        for (int j = failed_at + 1; j < my_count && j < failed_at + kStages; ++j)
            mbar_wait(&bars[j % kStages], (j / kStages) & 1, a.status);
    }

    // Fold the two half-warps (same D slice, different tokens).
#pragma unroll
    for (int g = 0; g < G; ++g)
#pragma unroll
        for (int e = 0; e < NE; ++e) acc[g][e] += __shfl_xor_sync(0xffffffffu, acc[g][e], 16);

    if (hw == 0) {
#pragma unroll
        for (int g = 0; g < G; ++g)
#pragma unroll
            for (int e = 0; e < NE; ++e) macc[(warp * G + g) * D + c * NE + e] = acc[g][e];
        if ((c % kHeadStride) == 0) {
            const int hl = c / kHeadStride;
            mm[warp * G + hl] = my_count > 0 ? m_run : -INFINITY;
            ml[warp * G + hl] = my_count > 0 ? l_run : 0.f;
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
        const int h = kvh * G + g;
        const size_t row = qrow * hq + h;
        if (nparts == 1) {
            store_elem<T>(static_cast<T*>(a.out) + row * D + d, o / l);
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

// Log-sum-exp merge of the partitions of one (sequence, query head):
// M = max m_p, w_p = l_p * 2^(m_p - M), out = sum w_p o_p / sum w_p.
// One warp per (sequence, query head); lane i owns elements [i*D/32, (i+1)*D/32)
// and the partials of all partitions are loaded 8 at a time so their latencies
// overlap.
constexpr int kCombineWarps = 4;

template <typename T, int D>
__global__ void __launch_bounds__(kCombineWarps * 32)
decode_combine_kernel(const DecodeArgs a) {
    griddep_wait();
    griddep_launch_dependents();
    constexpr int EL = D / 32;  // 4 (D 128) or 2 (D 64) elements per lane
    const int warp = threadIdx.x >> 5;
    const int lane = threadIdx.x & 31;
    const size_t row = static_cast<size_t>(blockIdx.x) * kCombineWarps + warp;  // seq*Hq + h
    if (row >= static_cast<size_t>(a.num_seqs) * a.num_q_heads) return;
    const int seq = static_cast<int>(row / a.num_q_heads);
    const int L = min(a.context_lens[seq], (a.max_blocks_per_seq << a.chunk_shift) * kBlock);
    const int nblk = (L + kBlock - 1) / kBlock;
    const int total = a.max_parts + a.extra_parts;   // partial slots per row
    const int np = a.extra_parts +
                   min(a.max_parts, max(0, (nblk - a.chunk_offset + a.partition_chunks - 1) /
                                               a.partition_chunks));
    if (np <= 0) return;
    const float* mp = a.m_part + row * total;
    const float* lp = a.l_part + row * total;
    const float* op = a.o_part + row * total * D + lane * EL;

    // One round trip for the common case: m and l of partials lane and lane + 32 and the
    // first 8 partial outputs are loaded together; the weights need the row max first.
    auto load_o = [&](int p, float (&v)[EL]) {
        const float* src = op + static_cast<size_t>(p) * D;
        if constexpr (EL == 4) {
            const float4 f = *reinterpret_cast<const float4*>(src);
            v[0] = f.x; v[1] = f.y; v[2] = f.z; v[3] = f.w;
        } else {
            const float2 f = *reinterpret_cast<const float2*>(src);
            v[0] = f.x; v[1] = f.y;
        }
    };
    const float m_a = lane < np ? mp[lane] : -INFINITY;
    const float l_a = lane < np ? lp[lane] : 0.f;
    float v0[8][EL];
#pragma unroll
    for (int u = 0; u < 8; ++u)
        if (u < np) load_o(u, v0[u]);
    float M = m_a;
    for (int p = lane + 32; p < np; p += 32) M = fmaxf(M, mp[p]);
#pragma unroll
    for (int o = 16; o > 0; o >>= 1) M = fmaxf(M, __shfl_xor_sync(0xffffffffu, M, o));

    float acc[EL];
#pragma unroll
    for (int e = 0; e < EL; ++e) acc[e] = 0.f;
    const float w_a = lane < np ? l_a * fast_exp2(m_a - M) : 0.f;
    float W = w_a;
#pragma unroll
    for (int u = 0; u < 8; ++u) {
        const float wu = __shfl_sync(0xffffffffu, w_a, u);
        if (u < np) {
#pragma unroll
            for (int e = 0; e < EL; ++e) acc[e] = fmaf(wu, v0[u][e], acc[e]);
        }
    }
    // Partials 8 .. np - 1 (long contexts), 8 loads in flight at a time.
    for (int base = 0; base < np; base += 32) {
        const int p = base + lane;
        const float w = base == 0 ? w_a : ((p < np) ? lp[p] * fast_exp2(mp[p] - M) : 0.f);
        if (base > 0) W += w;
        const int cnt = min(32, np - base);
        for (int u0 = base == 0 ? 8 : 0; u0 < cnt; u0 += 8) {
            float v[8][EL];
#pragma unroll
            for (int u = 0; u < 8; ++u)
                if (u0 + u < cnt) load_o(base + u0 + u, v[u]);
#pragma unroll
            for (int u = 0; u < 8; ++u) {
                const float wu = __shfl_sync(0xffffffffu, w, (u0 + u) & 31);
                if (u0 + u < cnt) {
#pragma unroll
                    for (int e = 0; e < EL; ++e) acc[e] = fmaf(wu, v[u][e], acc[e]);
                }
            }
        }
    }
#pragma unroll
    for (int o = 16; o > 0; o >>= 1) W += __shfl_xor_sync(0xffffffffu, W, o);
    const float inv = 1.f / W;
    T* dst = static_cast<T*>(a.out) + row * D + lane * EL;
#pragma unroll
    for (int e = 0; e < EL; ++e) store_elem<T>(dst + e, acc[e] * inv);
}

template <typename T, int D, int G>
cudaError_t launch_typed(const DecodeArgs& a, cudaStream_t stream) {
    using SM = DecodeSmem<T, D, G>;
    auto kern = decode_split_kernel<T, D, G>;
    cudaError_t e = set_smem_once(reinterpret_cast<const void*>(kern), SM::kTotal);
    if (e != cudaSuccess) return e;
    if (a.max_parts > 0) {   // zero when a cascade decode has no private suffix at all
        dim3 grid(a.max_parts, a.num_kv_heads, a.num_seqs);
        e = launch_maybe_pdl(!a.no_pdl, kern, grid, dim3(kThreads), SM::kTotal, stream, a);
        if (e != cudaSuccess) return e;
    }
    if (a.extra_parts == 0 && a.max_parts == 1) return e;  // output written directly
    if (a.defer_combine) return e;
    return launch_decode_combine(a, sizeof(T) == 2 ? PKV_BF16 : PKV_F32, D, stream);
}

template <typename T, int D>
cudaError_t launch_combine_typed(const DecodeArgs& a, cudaStream_t stream) {
    const size_t rows = static_cast<size_t>(a.num_seqs) * a.num_q_heads;
    const unsigned grid = static_cast<unsigned>((rows + kCombineWarps - 1) / kCombineWarps);
    return launch_pdl(decode_combine_kernel<T, D>, dim3(grid), dim3(kCombineWarps * 32), 0,
                      stream, a);
}

template <typename T, int D>
cudaError_t launch_group(const DecodeArgs& a, int G, cudaStream_t stream) {
    switch (G) {
        case 1: return launch_typed<T, D, 1>(a, stream);
        case 2: return launch_typed<T, D, 2>(a, stream);
        case 4: return launch_typed<T, D, 4>(a, stream);
        case 8: return launch_typed<T, D, 8>(a, stream);
        default: return cudaErrorInvalidValue;
    }
}

}  // namespace

cudaError_t launch_decode_combine(const DecodeArgs& a, int dtype, int head_dim,
                                  cudaStream_t stream) {
    if (dtype == PKV_BF16) {
        if (head_dim == 128) return launch_combine_typed<uint16_t, 128>(a, stream);
        if (head_dim == 64) return launch_combine_typed<uint16_t, 64>(a, stream);
    } else if (dtype == PKV_F32) {
        if (head_dim == 128) return launch_combine_typed<float, 128>(a, stream);
        if (head_dim == 64) return launch_combine_typed<float, 64>(a, stream);
    }
    return cudaErrorInvalidValue;
}

cudaError_t launch_paged_decode(const DecodeArgs& a, int dtype, int head_dim, int group,
                                cudaStream_t stream) {
    if (dtype == PKV_BF16) {
        if (head_dim == 128) return launch_group<uint16_t, 128>(a, group, stream);
        if (head_dim == 64) return launch_group<uint16_t, 64>(a, group, stream);
    } else if (dtype == PKV_F32) {
        if (head_dim == 128) return launch_group<float, 128>(a, group, stream);
        if (head_dim == 64) return launch_group<float, 64>(a, group, stream);
    }
    return cudaErrorInvalidValue;
}

}  // namespace pkv
