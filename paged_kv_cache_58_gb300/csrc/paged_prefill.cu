// Prefix-chunk causal prefill on the tcgen05 tensor cores.
//
// New query tokens of a request attend to the request's cached prefix plus the
// new tokens up to themselves; only the unseen suffix is computed while the
// cached K/V are reused from the pool (aitalk.it "RadixAttention: A Tree That
// Does Not Forget": compute only the unseen suffix; aifetchly SGLang guide,
// "Prefill Bypass").  K/V are gathered through the block table ("the kernel walks
// the block table", Triptych "Paged Attention for Efficient Memory Management").
//
// A query tile is 128 rows: TOK = 128 / G consecutive new tokens x the G query heads
// that share kv head `kvh` (rows token-major, heads inner), so every K/V tile staged
// for it serves all G heads.  A work item is a PAIR of adjacent query tiles, X = 0
// (tokens t0 .. t0 + TOK - 1) and X = 1 (the next TOK tokens; absent past the
// request's last token), of one request and kv head: both attend the same keys up to
// the causal limit, so each 128-key K/V tile staged in shared memory serves both, and
// the pair's two online softmaxes run side by side.  Per query tile X and KV tile j:
//   S_j = Q_X K_j^T  tcgen05.mma kind::f16 (bf16 in, fp32 accumulate) into the TMEM
//                    S/P buffer of X
//   softmax          warpgroup X, one thread per row: tcgen05.ld S_j, causal mask,
//                    exp2, row sums in fp32; P_j goes back over S_j in the same TMEM
//                    columns, as one bf16 value per weight (rounded to nearest) or as
//                    bf16 hi + lo parts (hi = P truncated, lo = the remainder
//                    truncated: hi + lo within 2^-14 of P)
//   O_X += P_j V_j   A = P from TMEM, B = V_j from shared memory, into the TMEM
//                    accumulator O_X (one P.V pass, or two for hi + lo)
// The split keeps the probabilities near fp32 precision: a single bf16 P is off by up
// to 2^-8 per weight, which rows attending only a few keys do not average away; with
// the split every output is within 2^-14 * max|v| of the exact weights' result.  A
// query tile whose rows all attend at least p_single_min_keys keys (1024 by default)
// keeps a single bf16 P, as FlashAttention-style kernels do: there the rounding errors
// of many weights average out (for N(0,1) data their effect on an output has a
// standard deviation near 2^-8 / sqrt(3 n / e) for n keys, about 1.2e-4 at n = 1024),
// and the P.V pass takes 8 MMAs instead of 16.
// The running max is updated lazily: O and l are rescaled only when a row's max grows
// by more than 2^8, which keeps P <= 256 and leaves the result exact.
//
// Ping-pong.  Within one query tile the chain S_j -> softmax -> P_j V_j -> S_{j+1}
// (which overwrites P_j) is serial; the pair's two chains interleave in the tensor
// pipe, so the pipe runs one tile's P.V and next S while the other tile's softmax
// works, and each softmax warpgroup has its own scheduler slots.  One warp issues
// each query tile's MMAs (S_j, then P_j V_j, then S_{j+1} once that P.V completed:
// MMAs with different accumulators are not ordered against each other).
//
// K/V staging.  One ring of shared-memory slots holds K_0, V_0, K_1, V_1, ... in turn
// (5 slots of 32 KB at head_dim 128); a slot is free again once both query tiles'
// MMAs that read it have run (the S products for a K slot, the P.V products for a V
// slot).  Each 16-token chunk of a tile (a 16-token block, or half of a 32-token
// one) arrives as ONE TMA box: at head_dim 128 a 4-D box (the chunk's 16 rows x 256 B
// viewed as 2 row groups x 2 column halves x 8 rows x 128 B, 128-byte swizzle), so a
// K/V tile lands as [8-key group][column half][8 rows][128 B]: a valid K-major operand
// (8-row atoms 2 KB apart) for S and MN-major operand (column halves 1 KB apart) for
// P.V; at head_dim 64 a 16-row x 64-column box, the tile one 64-column half with 8-row
// atoms 1 KB apart.  On the tile holding the last key a query tile needs, its P.V
// product skips the 16-key steps wholly past that key (P = 0 there); the V rows past
// the pair's last key (they may hold NaN from unused slots) are zeroed, once V has
// landed, by each issuer whose P.V reads them.
//
// Persistent CTAs.  A CTA pays a few microseconds outside its tile loop (barrier and
// TMEM set-up, the first gathers and S, the epilogue), which nothing overlaps when
// each SM runs one CTA; with at most 128 requests (and outside cascade mode) the grid
// is one CTA per SM and each works through a share of the items (see next_item), with
// the next item's Q, gathers and first S products under way while the softmax warps
// finish the current one.
//
// Warp roles (384 threads, three warpgroups): warps 0-3 softmax + epilogue of query
// tile 0, warps 4-7 the same for query tile 1 (warp w owns TMEM lanes 32 (w % 4) ..
// + 31), warp 8 barrier set-up + TMA producer, warp 9 TMEM owner + issuer of tile 0,
// warp 10 issuer of tile 1, warp 11 idle.  The softmax warpgroups take 216 registers
// a thread, the third warpgroup 72 (setmaxnreg).  TMEM columns: S/P of tiles 0 and 1
// at [0, 128) and [128, 256); their O at [256, 256 + D) and [256 + D, 256 + 2 D).
#include <atomic>
#include <cstdlib>

#include <cuda.h>
#include <cuda_runtime.h>

#include "common.cuh"
#include "kernels.h"
#include "tcgen05.cuh"

namespace pkv {

namespace {

constexpr int kRows = 128;                 // query rows per tile
constexpr int kKeys = 128;                 // keys per KV tile
constexpr int kChunk = 16;                 // tokens per staged chunk: a block, or half of one
constexpr int kHalf = kRows * 128;         // one 64-column half of a 128-row Q tile: 16 KB
constexpr int kMaxRing = 10;               // K/V ring slots at most (head_dim 64)
constexpr int kMaxSchedReqs = 128;         // persistent scheduling ranks up to 128 requests

// barrier indices: ring slot s full / empty; per query tile X (0, 1): S written, P
// written, P.V done, O read out, drain at exit.  BQ: the item's Q tiles landed;
// BQ_EMPTY: every S product of an item has run (the Q buffer may be reloaded).
constexpr int BFULL = 0, BEMPTY = kMaxRing, BQ = 2 * kMaxRing, BQ_EMPTY = BQ + 1,
              BS_FULL = BQ + 2, BP_FULL = BQ + 4, BPV_DONE = BQ + 6, BO_FREE = BQ + 8,
              BDRAIN = BQ + 10;
constexpr int kNumBars = BQ + 12;

// Shared-memory geometry for head_dim D (64 or 128).
template <int D>
struct Geom {
    static constexpr int kHalves = D / 64;                // 64-column halves of a row
    static constexpr int kQTile = kRows * D * 2;          // one Q tile
    static constexpr int kSlot = kKeys * D * 2;           // one K or V tile
    static constexpr int kRing = D == 128 ? 5 : kMaxRing; // ring slots
    static constexpr int kChunkBytes = kChunk * D * 2;    // 16 rows of one kv head
    static constexpr int kGroupBytes = 8 * D * 2;         // 8 key rows, every half
    static constexpr int kOffQ = 0;                       // Q tiles 0 and 1
    static constexpr int kOffRing = 2 * kQTile;
    static constexpr int kOffBar = kOffRing + kRing * kSlot;
    // barriers, then the TMEM address and abort flag, then the persistent schedule
    static constexpr int kOffSreq = kOffBar + kNumBars * 8 + 16;
    static constexpr int kOffOff = kOffSreq + kMaxSchedReqs * 2;
    static constexpr int kSmemBytes = kOffOff + (kMaxSchedReqs + 1) * 4 + 1024;  // + align slack
};
constexpr int kThreads = 384;
constexpr int kProducerWarp = 8;
constexpr int kMmaWarp = 9;                // issues query tile 0; owns TMEM (warp 10: tile 1)
constexpr uint32_t kTmemCols = 512;
constexpr uint32_t kTmemO = 256;           // O of tile X at kTmemO + X * D
constexpr float kLazyRescale = 8.0f;       // log2 units
constexpr float kNoMax = -1.0e30f;         // running max before a row saw a key
// Register split (setmaxnreg): the two softmax warpgroups and the third one.  Their sum
// over the 384 threads (2 x 128 x 216 + 128 x 72 = 64512) must not exceed what the
// launch provides (384 x the kernel's register count); the launcher checks it.
constexpr int kRegsSoftmax = 216;
constexpr int kRegsOther = 72;

struct Ctl {
    uint64_t* bars;
    volatile int* abort_flag;
    int* status;
};

// Bounded mbarrier wait of a converged warp, shared by all roles: every lane polls and a
// vote makes the outcome uniform (a completed phase stays completed), so the warp never
// diverges; reconverging a diverged warp costs hundreds of cycles while the scheduler is
// busy with the softmax.  Gives up when another role aborted or after the time budget
// (then raises PKV_ERR_TIMEOUT and aborts the CTA).
PKV_DEVINL bool wait_bar_warp(const Ctl& c, int idx, uint32_t parity, int lane) {
    uint64_t* bar = &c.bars[idx];
    if (__any_sync(0xffffffffu, mbar_try_wait(bar, parity))) return true;
    const unsigned long long t0 = globaltimer_ns();
    for (;;) {
        if (__any_sync(0xffffffffu, mbar_try_wait(bar, parity))) return true;
        if (__any_sync(0xffffffffu, *c.abort_flag != 0)) return false;
        if (__any_sync(0xffffffffu, globaltimer_ns() - t0 > kWaitBudgetNs)) {
            if (lane == 0) {
                raise_status(c.status, PKV_ERR_TIMEOUT);
                *c.abort_flag = 1;
            }
            __syncwarp();
            return false;
        }
    }
}

PKV_DEVINL void setmaxnreg_inc() {
    asm volatile("setmaxnreg.inc.sync.aligned.u32 %0;" ::"n"(kRegsSoftmax));
}
PKV_DEVINL void setmaxnreg_dec() {
    asm volatile("setmaxnreg.dec.sync.aligned.u32 %0;" ::"n"(kRegsOther));
}

// ------------------------------------------------------------------ work items
// An item is a pair of adjacent 128-row query tiles (2 m, 2 m + 1) of one request and
// kv head.  With `persistent` set the grid holds at most one CTA per SM, and CTA b
// works through the items k = i P + (b, or P - 1 - b for odd i), i = 0, 1, ... (P
// CTAs, a snake over the item list) of a list that ranks the requests by their key
// count, longest first, and within a request takes the pairs last-first: the longest
// items are spread over the CTAs first and each CTA's total comes out near the mean.
// Each role walks the same list, so barrier phases carry over from one item to the
// next and the next item's gathers and first S products start while the softmax warps
// finish the current one.  Otherwise CTA (x, y, z) takes the single item (pair x, kv
// head y, request z -- in cascade mode split z).

struct TileParams {   // one query tile of an item
    bool valid;       // the tile holds at least one of the request's new tokens
    int t0;           // its first token (cascade: first sequence)
    int max_lim;      // last key any of its rows sees
    int ntiles;       // KV tiles it reads: [j0, j0 + ntiles)
    bool p_single;    // one bf16 P per weight (else hi + lo)
};

struct ItemParams {
    int kvh, r, n, c, j0, ntiles, max_lim, qoff;
    TileParams x[2];
};

// Parameters of item (pair, kvh, r); false when it has no rows or no tile, or reads
// keys past its table (then PKV_ERR_OOB is raised when `report`).
template <int G>
PKV_DEVINL bool item_params(const PrefillArgs& a, int pair, int kvh, int r, bool report,
                            ItemParams& p) {
    constexpr int TOK = kRows / G;
    const bool cascade = a.cascade != 0;   // rows = sequences over the c shared keys
    p.kvh = kvh;
    p.r = r;
    p.n = cascade ? a.cascade_rows : __ldg(a.new_lens + r);
    p.c = cascade ? a.cascade_keys : __ldg(a.cached_lens + r);
    const int t0 = 2 * pair * TOK;
    if (t0 >= p.n) return false;
    const int L = cascade ? p.c : p.c + p.n;   // keys in the pool for this request
    if (p.c < 0 || L <= 0 || L > a.max_blocks_per_seq * a.block_size) {
        if (report) raise_status(a.status, PKV_ERR_OOB);
        return false;
    }
    // KV tiles [j0, j0 + ntiles): all of them, or in cascade mode the range of split r
    // (its partial goes to slot r; the host sizes the splits so that none is empty).
    p.j0 = cascade ? r * a.cascade_tiles_per_split : 0;
    p.ntiles = 0;
    p.max_lim = -1;
#pragma unroll
    for (int X = 0; X < 2; ++X) {
        TileParams& t = p.x[X];
        t.t0 = t0 + X * TOK;
        t.valid = t.t0 < p.n;
        const int i_last = min(t.t0 + TOK, p.n) - 1;
        t.max_lim = cascade ? p.c - 1 : p.c + i_last;
        t.ntiles = !t.valid ? 0
                   : cascade ? min(t.max_lim / kKeys + 1 - p.j0, a.cascade_tiles_per_split)
                             : t.max_lim / kKeys + 1;
        if (t.ntiles <= 0) t.valid = false;
        if (!t.valid) t.ntiles = 0;
        // Every row of the tile attends at least min_keys keys (its first token the fewest).
        const int min_keys = cascade ? p.c : p.c + t.t0 + 1;
        t.p_single = min_keys >= a.p_single_min_keys;
        if (t.valid) {
            p.ntiles = max(p.ntiles, t.ntiles);
            p.max_lim = max(p.max_lim, t.max_lim);
        }
    }
    if (p.ntiles <= 0) return false;
    p.qoff = cascade ? 0 : __ldg(a.q_offsets + r);
    return true;
}

// Persistent schedule in shared memory, right after the barriers, the TMEM address and
// the abort flag: sreq[rho] = the request of rank rho (most keys first), then off[rho] =
// its first item (off[R] = the item count).
constexpr int kSchedSreq = kNumBars * 8 + 16;                 // bytes past the barriers
constexpr int kSchedOff = kSchedSreq + kMaxSchedReqs * 2;

struct Sched {
    const uint64_t* bars;
    int R;
    bool persistent;
    PKV_DEVINL int sreq(int rho) const {
        return reinterpret_cast<const uint16_t*>(reinterpret_cast<const uint8_t*>(bars) +
                                                 kSchedSreq)[rho];
    }
    PKV_DEVINL int off(int rho) const {
        return reinterpret_cast<const int*>(reinterpret_cast<const uint8_t*>(bars) +
                                            kSchedOff)[rho];
    }
};

struct Cursor {
    int m = 0;     // the CTA's items visited
    int rho = 0;   // rank of the request holding the last one
};

// The CTA's next item; false when it has none left.
template <int G>
PKV_DEVINL bool next_item(const PrefillArgs& a, const Sched& s, Cursor& cur, bool report,
                          ItemParams& p) {
    if (!s.persistent) {
        if (cur.m++ > 0) return false;
        return item_params<G>(a, blockIdx.x, blockIdx.y, blockIdx.z, report, p);
    }
    const int P = gridDim.x;
    const int b = blockIdx.x;
    const int total = s.off(s.R);
    for (;;) {
        const int m = cur.m++;
        const int k = m * P + ((m & 1) ? P - 1 - b : b);
        if (k >= total) return false;
        while (s.off(cur.rho + 1) <= k) ++cur.rho;   // k grows with m
        const int rem = k - s.off(cur.rho);
        const int np = (s.off(cur.rho + 1) - s.off(cur.rho)) / a.num_kv_heads;
        if (item_params<G>(a, np - 1 - rem / a.num_kv_heads, rem % a.num_kv_heads,
                           s.sreq(cur.rho), report, p))
            return true;
    }
}

// Ring slot and phase parity of the K (v = 0) or V (v = 1) tile of the CTA's g-th KV tile.
template <int R>
PKV_DEVINL int ring_slot(int g, int v) { return (2 * g + v) % R; }
template <int R>
PKV_DEVINL uint32_t ring_par(int g, int v) { return static_cast<uint32_t>((2 * g + v) / R) & 1u; }

template <int D, int G>
__global__ void __launch_bounds__(kThreads, 1)
prefill_tcgen05_kernel(const __grid_constant__ CUtensorMap tm_q,
                       const __grid_constant__ CUtensorMap tm_k,
                       const __grid_constant__ CUtensorMap tm_v, const PrefillArgs a,
                       const int persistent, const int test_stall) {
    using GM = Geom<D>;
    constexpr int TOK = kRows / G;
    constexpr int R = GM::kRing;
    extern __shared__ uint8_t smem_raw[];
    uint8_t* smem = reinterpret_cast<uint8_t*>(
        (reinterpret_cast<uintptr_t>(smem_raw) + 1023) & ~static_cast<uintptr_t>(1023));

    const int warp = threadIdx.x >> 5;
    const int lane = threadIdx.x & 31;
    griddep_wait();
    griddep_launch_dependents();
    const bool cascade = a.cascade != 0;
    const int csh = a.block_size == 32 ? 1 : 0;   // log2 of chunks per block

    uint64_t* bars = reinterpret_cast<uint64_t*>(smem + GM::kOffBar);
    uint32_t* tmem_slot = reinterpret_cast<uint32_t*>(smem + GM::kOffBar + kNumBars * 8);
    volatile int* abort_flag = reinterpret_cast<volatile int*>(tmem_slot + 1);
    uint16_t* sreq = reinterpret_cast<uint16_t*>(smem + GM::kOffSreq);
    int* off = reinterpret_cast<int*>(smem + GM::kOffOff);
    Ctl ctl{bars, abort_flag, a.status};
    const Sched sch{bars, a.num_reqs, persistent != 0};

    if (sch.persistent) {
        // Rank the requests by key count (most first, ties by index) and lay out the
        // item list: rank rho holds ceil(n / (2 TOK)) query-tile pairs x the kv heads.
        const int Rq = a.num_reqs;
        for (int t = threadIdx.x; t < Rq; t += kThreads)   // off[] holds the key counts first
            off[t] = __ldg(a.cached_lens + t) + __ldg(a.new_lens + t);
        __syncthreads();
        for (int t = threadIdx.x; t < Rq; t += kThreads) {
            const int kt = off[t];
            int rank = 0;
            for (int u = 0; u < Rq; ++u) {
                const int ku = off[u];
                rank += (ku > kt) || (ku == kt && u < t);
            }
            sreq[rank] = static_cast<uint16_t>(t);
        }
        __syncthreads();
        if (warp == 0) {   // exclusive scan of the item counts over the ranks, 4 per lane
            int cnt[4], sum = 0;
#pragma unroll
            for (int e = 0; e < 4; ++e) {
                const int rho = lane * 4 + e;
                int v = 0;
                if (rho < Rq) {
                    const int nn = __ldg(a.new_lens + sreq[rho]);
                    v = nn > 0 ? (nn + 2 * TOK - 1) / (2 * TOK) * a.num_kv_heads : 0;
                }
                cnt[e] = v;
                sum += v;
            }
            int incl = sum;
#pragma unroll
            for (int o = 1; o < 32; o <<= 1) {
                const int y = __shfl_up_sync(0xffffffffu, incl, o);
                if (lane >= o) incl += y;
            }
            int run = incl - sum;
#pragma unroll
            for (int e = 0; e < 4; ++e) {
                const int rho = lane * 4 + e;
                if (rho < Rq) off[rho] = run;
                run += cnt[e];
                if (rho == Rq - 1) off[Rq] = run;
            }
        }
        __syncthreads();
    }

    if (warp == kProducerWarp) {
        if (lane == 0) {
            mbar_init(&bars[BQ], 1);
            mbar_init(&bars[BQ_EMPTY], 2);
            for (int st = 0; st < R; ++st) {
                mbar_init(&bars[BFULL + st], 1);
                mbar_init(&bars[BEMPTY + st], 2);   // both query tiles' products
            }
            for (int X = 0; X < 2; ++X) {
                mbar_init(&bars[BS_FULL + X], 1);
                mbar_init(&bars[BP_FULL + X], 4);   // the tile's four softmax warps
                mbar_init(&bars[BPV_DONE + X], 1);
                mbar_init(&bars[BO_FREE + X], 4);
                mbar_init(&bars[BDRAIN + X], 1);
            }
            *abort_flag = 0;
            fence_mbar_init();
            prefetch_tmap(&tm_q);
            prefetch_tmap(&tm_k);
            prefetch_tmap(&tm_v);
        }
    } else if (warp == kMmaWarp) {
        tmem_alloc(tmem_slot, kTmemCols);
        tmem_relinquish();
    }
    tc_fence_before();
    __syncthreads();
    tc_fence_after();
    const uint32_t tmem = *tmem_slot;

    const uint32_t sQ = smem_u32(smem + GM::kOffQ);
    const uint32_t sRing = smem_u32(smem + GM::kOffRing);

    if (warp >= 8) {
    // Registers: this warpgroup hands part of its share to the two softmax warpgroups.
    setmaxnreg_dec();
    if (warp == kProducerWarp) {
        // ------------------------------------------------------------ TMA producer
        // The whole warp runs the loop: each lane prefetches the block id of one 16-token
        // chunk (32 chunks = 4 KV tiles per refill, independent loads), lane 0 sets the
        // byte counts and lane b < 8 issues the box of chunk b of the tile.  A chunk is
        // a whole block (block size 16) or rows 16 h .. 16 h + 15 of one (block size 32).
        // Ring slots and their phases count the CTA's tiles over all its items (g); the
        // Q tiles of an item are loaded once every S product of the previous item has run.
        Cursor cur;
        ItemParams p;
        int it = 0, g = 0;
        int issued = 0;   // K and V tiles issued into the ring (2 per KV tile)
        bool ok = true;
        while (ok && next_item<G>(a, sch, cur, lane == 0, p)) {
            const int32_t* bt =
                a.block_tables + static_cast<size_t>(cascade ? 0 : p.r) * a.max_blocks_per_seq;
            const int nchunks = p.max_lim / kChunk + 1;
            if (it >= 1 && !wait_bar_warp(ctl, BQ_EMPTY, (it - 1) & 1, lane)) break;
            // Test hook (zero in normal use): CTA 0 arms its first Q barrier for 16 bytes
            // more than the Q copies deliver, so the issuers' wait for it runs out of time
            // (PKV_ERR_TIMEOUT) while the copies still land.
            const bool stall = test_stall && it == 0 && blockIdx.x == 0 && blockIdx.y == 0 &&
                               blockIdx.z == 0;
            if (lane == 0) {
                const bool two = p.x[1].valid;
                mbar_arrive_expect_tx(&bars[BQ], (two ? 2 : 1) * GM::kQTile + (stall ? 16u : 0u));
#pragma unroll
                for (int X = 0; X < 2; ++X) {
                    if (X == 0 || two) {
#pragma unroll
                        for (int h = 0; h < GM::kHalves; ++h)
                            tma_load_3d(smem + GM::kOffQ + X * GM::kQTile + h * kHalf, &tm_q,
                                        64 * h, p.kvh * G, p.qoff + p.x[X].t0, &bars[BQ]);
                    }
                }
            }
            ++it;
            int ids = 0;
            for (int jt = 0; jt < p.ntiles; ++jt, ++g) {
                constexpr int kPerTile = kKeys / kChunk;   // 8 chunks per KV tile
                if ((jt & 3) == 0) {
                    const int i = (p.j0 + jt) * kPerTile + lane;
                    ids = (i < nchunks) ? __ldg(bt + (i >> csh)) : 0;
                }
                const int nb = min(kPerTile, nchunks - (p.j0 + jt) * kPerTile);
                int phys = __shfl_sync(0xffffffffu, ids, ((jt & 3) * kPerTile) + (lane & 7));
                if (phys < 0 || phys >= a.num_blocks) {
                    if (lane < nb) raise_status(a.status, PKV_ERR_OOB);
                    phys = 0;  // keep the byte count; the output is flagged invalid
                }
                const int chunk = (p.j0 + jt) * kPerTile + (lane & 7);
                const int row = (phys * a.num_kv_heads + p.kvh) * a.block_size +
                                (chunk & ((1 << csh) - 1)) * kChunk;
                // K then V of tile g, each into the next ring slot once both query tiles'
                // products that read its previous contents have run.  The warp stays
                // converged: lane 0 sets the byte count and lanes b < nb issue the boxes
                // through predicated instructions.
#pragma unroll
                for (int v = 0; v < 2; ++v) {
                    const int s = ring_slot<R>(g, v);
                    if (issued >= R &&
                        !wait_bar_warp(ctl, BEMPTY + s, ring_par<R>(g, v) ^ 1u, lane)) {
                        ok = false;
                        break;
                    }
                    mbar_arrive_expect_tx_if(lane == 0, &bars[BFULL + s], nb * GM::kChunkBytes);
                    uint8_t* dst = smem + GM::kOffRing + s * GM::kSlot + lane * GM::kChunkBytes;
                    const void* map = v ? static_cast<const void*>(&tm_v) : &tm_k;
                    if constexpr (D == 128)
                        tma_load_4d_if(lane < nb, dst, map, 0, 0, 0, row / 8, &bars[BFULL + s]);
                    else
                        tma_load_2d_if(lane < nb, dst, map, 0, row, &bars[BFULL + s]);
                    ++issued;
                }
                if (!ok) break;
            }
        }
        // Drain (also after an abort): wait, bounded, until the last copy issued into
        // every slot has landed, so that no TMA write into shared memory outlives the
        // CTA.  No later copy goes into those slots, so the phases cannot move on.
        if (it >= 1) mbar_wait_warp(&bars[BQ], (it - 1) & 1, a.status);
        for (int s = 0; s < R; ++s) {
            if (issued > s) {
                const int last = s + R * ((issued - 1 - s) / R);   // ring index of its last use
                mbar_wait_warp(&bars[BFULL + s], static_cast<uint32_t>(last / R) & 1u, a.status);
            }
        }
    } else if (warp == kMmaWarp || warp == kMmaWarp + 1) {
        // ------------------------------------------------------------ MMA issuers
        // Warp kMmaWarp + X issues query tile X: for its KV tiles j: S_j into its S/P
        // buffer, then O_X += P_j V_j once the softmax has written P_j there, then S_{j+1}
        // into the same buffer once that P.V has completed.  A KV tile of the item past
        // this tile's last (or every tile, when the pair has no tile X) is only waited
        // for and released, so that each ring slot's phase needs both issuers and no
        // issuer runs a phase ahead.  Each issuing warp shares its scheduler with two
        // softmax warps and gets only the issue slots they leave free, so the loop is
        // short: the whole warp runs it converged (all lanes poll, then one leader lane
        // issues through predicated instructions), and the descriptors are precomputed
        // halves plus constant offsets.  Across items: an item's first P.V into O_X waits
        // until the softmax warps have read O_X out for the last item in which tile X had
        // tiles (BO_FREE + X, one phase per such item), and once this tile's last S of an
        // item has run it signals that the Q buffer may take the next item's Q (BQ_EMPTY;
        // an issuer without tiles in the item just arrives).  Both issuers wait for every
        // phase of BQ, tiles or not, so that no parity wait can fall two phases behind.
        constexpr uint32_t idesc_qk = idesc_bf16_f32(kRows, kKeys, false, false);
        constexpr uint32_t idesc_pv = idesc_bf16_f32(kRows, D, false, true);
        constexpr uint32_t hi_q = smem_desc_sw128_hi(1024);          // Q: 8-row atoms 1 KB apart
        constexpr uint32_t hi_kv = smem_desc_sw128_hi(GM::kGroupBytes);  // K/V: 8-key groups
        const int X = warp - kMmaWarp;
        const uint32_t lo_q = smem_desc_sw128_lo(sQ + X * GM::kQTile, 16);
        const uint32_t lo_k = smem_desc_sw128_lo(sRing, 16);
        const uint32_t lo_v = smem_desc_sw128_lo(sRing, 1024);       // V: column halves 1 KB apart
        const uint32_t tS = tmem + X * 128;
        const uint32_t tO = tmem + kTmemO + X * D;
        const bool leader = elect_one();   // issues every MMA and commit of this tile
        Cursor cur;
        ItemParams p;
        int it = 0, g0 = 0;
        uint32_t use = 0;     // this tile's KV tiles over all items (S/P buffer phases)
        uint32_t o_use = 0;   // items in which this tile had KV tiles (O_X read-outs)
        bool ok = true;
        while (ok && next_item<G>(a, sch, cur, false, p)) {
            ok = wait_bar_warp(ctl, BQ, it & 1, lane);
            const TileParams tp = X ? p.x[1] : p.x[0];   // selects, not a local-memory index
            bool o_free = o_use == 0;   // O_X read out after its last item
            for (int j = 0; ok && j < p.ntiles; ++j) {
                const int g = g0 + j;
                const int sk = ring_slot<R>(g, 0), sv = ring_slot<R>(g, 1);
                if (j >= tp.ntiles) {   // not read by this tile: release once landed
                    if (!wait_bar_warp(ctl, BFULL + sk, ring_par<R>(g, 0), lane)) { ok = false; break; }
                    mbar_arrive_if(leader, &bars[BEMPTY + sk]);
                    if (!wait_bar_warp(ctl, BFULL + sv, ring_par<R>(g, 1), lane)) { ok = false; break; }
                    mbar_arrive_if(leader, &bars[BEMPTY + sv]);
                    continue;
                }
                // S_j: K_j landed, and P of this buffer's previous tile consumed by its P.V.
                if (!wait_bar_warp(ctl, BFULL + sk, ring_par<R>(g, 0), lane)) { ok = false; break; }
                if (use >= 1 && !wait_bar_warp(ctl, BPV_DONE + X, (use - 1) & 1, lane)) {
                    ok = false;
                    break;
                }
                tc_fence_after();
                {
                    const uint32_t lk = lo_k + ((sk * GM::kSlot) >> 4);
#pragma unroll
                    for (int ks = 0; ks < D / 16; ++ks) {
                        const uint32_t kc = ((ks & 3) * 32) >> 4;   // 16 columns = 32 B
                        umma_bf16_if(leader, tS,
                                     desc_join(lo_q + (((ks >> 2) * kHalf) >> 4) + kc, hi_q),
                                     desc_join(lk + (((ks >> 2) * 1024) >> 4) + kc, hi_kv),
                                     idesc_qk, ks > 0);
                    }
                    umma_commit_if(leader, &bars[BS_FULL + X]);
                    umma_commit_if(leader, &bars[BEMPTY + sk]);
                    if (j + 1 == tp.ntiles) umma_commit_if(leader, &bars[BQ_EMPTY]);   // last S
                }
                // O_X += P_j V_j: P_j written, V_j landed, O_X read out (first tile).
                if (!wait_bar_warp(ctl, BP_FULL + X, use & 1, lane)) { ok = false; break; }
                if (!wait_bar_warp(ctl, BFULL + sv, ring_par<R>(g, 1), lane)) { ok = false; break; }
                if (!o_free) {
                    if (!wait_bar_warp(ctl, BO_FREE + X, (o_use - 1) & 1, lane)) {
                        ok = false;
                        break;
                    }
                    o_free = true;
                }
                // Keys past the last one this tile needs are masked for every row (P = 0):
                // the P.V product skips the 16-key steps that lie wholly past that key.
                // Rows past the pair's last key may hold anything (NaN in unused slots,
                // stale data where no block was loaded this tile): where this product
                // reads them (its last step is the pair's), they are zeroed, now that V_j
                // has landed, so that 0 * V stays 0.  Both issuers may zero the same rows;
                // both write zeros, which leaves the other's product reading zeros.
                const int kbase = (p.j0 + j) * kKeys;
                const int nvalid = min(kKeys, tp.max_lim - kbase + 1);   // >= 1
                const int ksteps = (nvalid + 15) >> 4;
                const int nvalid_pair = min(kKeys, p.max_lim - kbase + 1);
                if (nvalid_pair < ksteps * 16) {
                    const uint4 z = make_uint4(0, 0, 0, 0);
                    // rows nvalid_pair .. 16 ksteps - 1, 8 pieces per 128-byte half: lane =
                    // piece 8 rows apart so that each store instruction touches 8 rows of an atom
                    const int rows = ksteps * 16 - nvalid_pair;
                    for (int t = lane; t < rows * 8 * GM::kHalves; t += 32) {
                        const int row = nvalid_pair + t / (8 * GM::kHalves);
                        const int hh = (t / 8) % GM::kHalves;
                        const int jj = t & 7;
                        uint8_t* vrow = smem + GM::kOffRing + sv * GM::kSlot +
                                        (row >> 3) * GM::kGroupBytes + (row & 7) * 128;
                        *reinterpret_cast<uint4*>(vrow + hh * 1024 + ((jj ^ (row & 7)) << 4)) = z;
                    }
                    fence_proxy_async_smem();
                    __syncwarp();
                }
                tc_fence_after();
                {
                    const uint32_t lv = lo_v + ((sv * GM::kSlot) >> 4);
                    // V as the MN-major B operand: 16 keys = two 8-key groups.
#pragma unroll
                    for (int ks = 0; ks < kKeys / 16; ++ks) {
                        const uint64_t bv = desc_join(lv + ((ks * 2 * GM::kGroupBytes) >> 4), hi_kv);
                        umma_bf16_ta_if(leader && ks < ksteps, tO, tS + ks * 8, bv, idesc_pv,
                                        (j >= 1) || (ks > 0));
                        if (!tp.p_single)
                            umma_bf16_ta_if(leader && ks < ksteps, tO, tS + 64 + ks * 8, bv,
                                            idesc_pv, true);
                    }
                    umma_commit_if(leader, &bars[BPV_DONE + X]);
                    umma_commit_if(leader, &bars[BEMPTY + sv]);
                }
                ++use;
            }
            if (!ok) break;
            if (tp.ntiles == 0)
                mbar_arrive_if(leader, &bars[BQ_EMPTY]);   // no S in this item
            else
                ++o_use;
            g0 += p.ntiles;
            ++it;
        }
        // Drain (also after an abort): every MMA this tile issued completes before
        // the TMEM is freed at the end of the kernel.
        umma_commit_if(leader, &bars[BDRAIN + X]);
        mbar_wait_warp(&bars[BDRAIN + X], 0, a.status);
    }
    } else {
        setmaxnreg_inc();
        // ------------------------------------------------------------ softmax + epilogue
        const int X = warp >> 2;                  // query tile of this warpgroup
        const int row = threadIdx.x & 127;        // == TMEM lane
        const uint32_t lane_addr = static_cast<uint32_t>((warp & 3) * 32) << 16;
        const uint32_t tS = tmem + lane_addr + X * 128;
        const uint32_t tO = tmem + lane_addr + kTmemO + X * D;
        const float sl2 = a.scale_log2;
        Cursor cur;
        ItemParams p;
        uint32_t par = 0;   // parity of this tile's KV tiles over all items
        bool ok = true;
        bool have = next_item<G>(a, sch, cur, false, p);
        while (ok && have) {
        const TileParams tp = X ? p.x[1] : p.x[0];   // selects, not a local-memory index
        const int tok = tp.t0 + row / G;
        const bool row_valid = tok < p.n;
        const size_t orow_idx = static_cast<size_t>(p.qoff + tok) * a.num_q_heads +
                                p.kvh * G + row % G;
        const int lim = cascade ? p.c - 1 : (row_valid ? p.c + tok : p.c + p.n - 1);  // last key seen
        const bool p_single = tp.p_single;
        const int ntiles = tp.ntiles;
        float m_run = kNoMax;   // running max (log2 domain) and row sum
        float l_run = 0.f;
        for (int jt = 0; jt < ntiles; ++jt) {
            if (!wait_bar_warp(ctl, BS_FULL + X, par, lane)) { ok = false; break; }
            tc_fence_after();
            float x[kKeys];
#pragma unroll
            for (int q = 0; q < 4; ++q)
                tmem_ld32(tS + q * 32, *reinterpret_cast<float(*)[32]>(&x[q * 32]));
            tmem_wait_ld();

            const int kbase = (p.j0 + jt) * kKeys;
            if (kbase + kKeys - 1 > lim) {
#pragma unroll
                for (int k = 0; k < kKeys; ++k) x[k] = (kbase + k <= lim) ? x[k] : -INFINITY;
            }
            // Row max over 4 independent chains of three-input max.
            float m4[4];
#pragma unroll
            for (int u = 0; u < 4; ++u) m4[u] = -INFINITY;
#pragma unroll
            for (int k = 0; k < kKeys; k += 2)
                m4[(k >> 1) & 3] = fmax3(m4[(k >> 1) & 3], x[k], x[k + 1]);
            const float mx = fmaxf(fmaxf(m4[0], m4[1]), fmaxf(m4[2], m4[3]));
            const float m_tile = mx * sl2;   // scale > 0: max commutes with scaling
            const bool grow = m_tile > m_run + kLazyRescale;
            const float m_cur = grow ? m_tile : m_run;
            // 1 unless grow; 0 when the row had no key yet.  A row with no key in this
            // tile keeps m_cur finite (kNoMax at worst), so its p are exp2(-inf) = 0.
            const float alpha = fast_exp2(m_run - m_cur);
            // P_jt over S_jt in the same buffer (S is already in registers), written 32
            // keys at a time so that few packed values are live and the exp chains of a
            // chunk overlap.
            float rs8[8];
#pragma unroll
            for (int u = 0; u < 8; ++u) rs8[u] = 0.f;
            if (p_single) {
                // One bf16 P per weight (round to nearest) in columns [0, 64).
#pragma unroll
                for (int q = 0; q < kKeys / 32; ++q) {
                    uint32_t ph[16];
#pragma unroll
                    for (int e = 0; e < 16; ++e) {
                        const int k = q * 32 + 2 * e;
                        float a0, a1;
                        ffma2(a0, a1, x[k], x[k + 1], sl2, sl2, -m_cur, -m_cur);
                        const float p0 = fast_exp2(a0);
                        const float p1 = fast_exp2(a1);
                        const int u = (e & 3) * 2;
                        // row sums by fma with 1 (exact, one rounding as an add)
                        ffma2(rs8[u], rs8[u + 1], p0, p1, 1.f, 1.f, rs8[u], rs8[u + 1]);
                        ph[e] = pack_bf16x2(p0, p1);
                    }
                    tmem_st16(tS + q * 16, ph);
                }
            } else {
                // hi (P truncated to bf16) in columns [0, 64), lo (the exact remainder
                // P - hi, truncated) in [64, 128): hi + lo within 2^-14 of P, from byte
                // permutes instead of conversions.
#pragma unroll
                for (int q = 0; q < kKeys / 32; ++q) {
                    uint32_t phi[16], plo[16];
#pragma unroll
                    for (int e = 0; e < 16; ++e) {
                        const int k = q * 32 + 2 * e;
                        float a0, a1;
                        ffma2(a0, a1, x[k], x[k + 1], sl2, sl2, -m_cur, -m_cur);
                        const float p0 = fast_exp2(a0);
                        const float p1 = fast_exp2(a1);
                        const int u = (e & 3) * 2;
                        ffma2(rs8[u], rs8[u + 1], p0, p1, 1.f, 1.f, rs8[u], rs8[u + 1]);
                        phi[e] = pack_bf16x2_trunc(p0, p1);
                        float r0, r1;
                        ffma2(r0, r1, __uint_as_float(__float_as_uint(p0) & 0xffff0000u),
                              __uint_as_float(__float_as_uint(p1) & 0xffff0000u), -1.f, -1.f,
                              p0, p1);
                        plo[e] = pack_bf16x2_trunc(r0, r1);
                    }
                    tmem_st16(tS + q * 16, phi);
                    tmem_st16(tS + 64 + q * 16, plo);
                }
            }
            const float rs = ((rs8[0] + rs8[1]) + (rs8[2] + rs8[3])) +
                             ((rs8[4] + rs8[5]) + (rs8[6] + rs8[7]));
            l_run = l_run * alpha + rs;
            m_run = m_cur;
            // O_X is rescaled only when some row of the warp grew its max; here, after the
            // P stores (S no longer in registers) and before P is handed over, so that
            // the next P.V accumulates onto the rescaled O.  The previous P.V (tile
            // jt - 1) has completed already: S_jt waited for it before overwriting the
            // buffer; the wait below only makes that visible here.
            if (jt >= 1 && __any_sync(0xffffffffu, grow)) {
                if (!wait_bar_warp(ctl, BPV_DONE + X, par ^ 1u, lane)) {
                    ok = false;
                    break;
                }
                tc_fence_after();
#pragma unroll
                for (int q = 0; q < D / 32; ++q) {
                    float o[32];
                    tmem_ld32(tO + q * 32, o);
                    tmem_wait_ld();
#pragma unroll
                    for (int e = 0; e < 32; ++e) o[e] *= alpha;
                    tmem_st32(tO + q * 32, o);
                }
            }
            tmem_wait_st();
            tc_fence_before();
            __syncwarp();
            mbar_arrive_if(lane == 0, &bars[BP_FULL + X]);
            par ^= 1u;
        }
        if (!ok) break;
        // The next item's parameters, looked up now so that their loads overlap the
        // epilogue's waits rather than delay the next item's first tile.
        ItemParams pn;
        const bool have_next = next_item<G>(a, sch, cur, false, pn);
        if (ntiles > 0) {
            // ------------------------------------------------------------ epilogue
            // O = O_X / l; the tile's last P.V must have completed.
            if (!wait_bar_warp(ctl, BPV_DONE + X, par ^ 1u, lane)) break;
            tc_fence_after();
            const float inv = 1.f / l_run;
            uint16_t* orow = static_cast<uint16_t*>(a.out) + orow_idx * D;
            const size_t prow = orow_idx * a.max_parts_total + p.r;   // cascade: slot = split
            if (cascade && row_valid) {
                a.m_part[prow] = m_run;   // log2 domain, as the decode partials
                a.l_part[prow] = l_run;
            }
#pragma unroll
            for (int q = 0; q < D / 32; ++q) {
                float o[32];
                tmem_ld32(tO + q * 32, o);
                tmem_wait_ld();
#pragma unroll
                for (int e = 0; e < 32; ++e) o[e] *= inv;
                if (cascade && row_valid) {
                    float* dst = a.o_part + prow * D + q * 32;
#pragma unroll
                    for (int e = 0; e < 32; e += 4)
                        *reinterpret_cast<float4*>(dst + e) =
                            make_float4(o[e], o[e + 1], o[e + 2], o[e + 3]);
                } else if (row_valid) {
#pragma unroll
                    for (int e = 0; e < 32; e += 8) {
                        uint4 w;
                        w.x = pack_bf16x2(o[e], o[e + 1]);
                        w.y = pack_bf16x2(o[e + 2], o[e + 3]);
                        w.z = pack_bf16x2(o[e + 4], o[e + 5]);
                        w.w = pack_bf16x2(o[e + 6], o[e + 7]);
                        *reinterpret_cast<uint4*>(orow + q * 32 + e) = w;
                    }
                }
            }
            // O_X of this item is read out: the issuer may start the next item's P.V.
            tc_fence_before();
            __syncwarp();
            mbar_arrive_if(lane == 0, &bars[BO_FREE + X]);
        }
        p = pn;
        have = have_next;
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

// Test hook: PKV_TEST_PREFILL_STALL=1 makes one Q wait of the next prefill run out of
// time (read at each call; tests only).
int prefill_test_stall() {
    const char* v = std::getenv("PKV_TEST_PREFILL_STALL");
    return v && v[0] == '1' ? 1 : 0;
}

// Streaming multiprocessors of the current device (read once per device).
int sm_count() {
    static std::atomic<int> cached[64];   // 0: not read yet; host threads may race benignly
    int dev = 0;
    if (cudaGetDevice(&dev) != cudaSuccess || dev < 0 || dev >= 64) return 1;
    int v = cached[dev].load(std::memory_order_relaxed);
    if (v <= 0) {
        if (cudaDeviceGetAttribute(&v, cudaDevAttrMultiProcessorCount, dev) != cudaSuccess || v <= 0)
            return 1;
        cached[dev].store(v, std::memory_order_relaxed);
    }
    return v;
}

// The register split is only safe when the launch gives the CTA at least the registers
// the split hands out: 384 threads x the kernel's register count (ptxas).  Checked once
// per kernel and device; a kernel built with fewer registers is not launched.
template <typename K>
bool register_split_fits(K kern) {
    static std::atomic<int> ok_cached[64];   // 0 unknown, 1 fits, 2 does not
    int dev = 0;
    if (cudaGetDevice(&dev) != cudaSuccess || dev < 0 || dev >= 64) return false;
    int v = ok_cached[dev].load(std::memory_order_relaxed);
    if (v == 0) {
        cudaFuncAttributes attr{};
        if (cudaFuncGetAttributes(&attr, reinterpret_cast<const void*>(kern)) != cudaSuccess)
            return false;
        const int need = 2 * 128 * kRegsSoftmax + 128 * kRegsOther;
        v = attr.numRegs * kThreads >= need ? 1 : 2;
        ok_cached[dev].store(v, std::memory_order_relaxed);
    }
    return v == 1;
}

template <int D, int G>
cudaError_t launch_g(const PrefillArgs& a, cudaStream_t stream) {
    using GM = Geom<D>;
    CUtensorMap mq, mk, mv;
    const int64_t rows = a.num_blocks * a.num_kv_heads * a.block_size;
    const bool pool_ok = D == 128 ? make_pool_block_map(&mk, a.k_pool, rows) &&
                                        make_pool_block_map(&mv, a.v_pool, rows)
                                  : make_pool_map(&mk, a.k_pool, rows, D) &&
                                        make_pool_map(&mv, a.v_pool, rows, D);
    if (!pool_ok || !make_q_group_map(&mq, a.q, a.total_new, a.num_q_heads, D, G, kRows / G))
        return cudaErrorInvalidValue;
    auto kern = prefill_tcgen05_kernel<D, G>;
    if (!register_split_fits(kern)) return cudaErrorNotSupported;
    cudaError_t e =
        set_smem_once(reinterpret_cast<const void*>(kern), GM::kSmemBytes);
    if (e != cudaSuccess) return e;
    constexpr int TOK = kRows / G;
    const int pairs = (a.max_new + 2 * TOK - 1) / (2 * TOK);
    // Persistent CTAs walking the ranked item list, at most one per SM; not for the
    // cascade's prefix pass, which is meant to hold few SMs beside the suffix decode.
    const int persistent = (!a.cascade && a.num_reqs <= kMaxSchedReqs) ? 1 : 0;
    dim3 grid(pairs, a.num_kv_heads, a.num_reqs);
    if (persistent) {
        const int64_t items = static_cast<int64_t>(pairs) * a.num_kv_heads * a.num_reqs;
        grid = dim3(static_cast<unsigned>(items < sm_count() ? items : sm_count()), 1, 1);
    }
    return launch_pdl(kern, grid, dim3(kThreads), GM::kSmemBytes, stream, mq, mk, mv, a,
                      persistent, prefill_test_stall());
}

template <int D>
cudaError_t launch_d(const PrefillArgs& a, int group, cudaStream_t stream) {
    switch (group) {
        case 1: return launch_g<D, 1>(a, stream);
        case 2: return launch_g<D, 2>(a, stream);
        case 4: return launch_g<D, 4>(a, stream);
        case 8: return launch_g<D, 8>(a, stream);
        default: return cudaErrorNotSupported;
    }
}

}  // namespace

cudaError_t launch_paged_prefill(const PrefillArgs& a, int group, cudaStream_t stream) {
    if (a.block_size != 16 && a.block_size != 32) return cudaErrorNotSupported;
    if (a.head_dim == 128) return launch_d<128>(a, group, stream);
    if (a.head_dim == 64) return launch_d<64>(a, group, stream);
    return cudaErrorNotSupported;
}

}  // namespace pkv
