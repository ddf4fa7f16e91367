// Prefix-chunk causal prefill on the tcgen05 tensor cores.
//
// New query tokens of a request attend to the request's cached prefix plus the
// new tokens up to themselves; only the unseen suffix is computed while the
// cached K/V are reused from the pool (aitalk.it "RadixAttention: A Tree That
// Does Not Forget": compute only the unseen suffix; aifetchly SGLang guide,
// "Prefill Bypass").  K/V are gathered through the block table ("the kernel walks
// the block table", Triptych "Paged Attention for Efficient Memory Management").
//
// A work item is one 128-row query tile: TOK = 128 / G consecutive new tokens x the G
// query heads that share kv head `kvh` (rows token-major, heads inner), so every K/V
// tile staged for it serves all G heads.  Per 128-key KV tile j:
//   S_j = Q K_j^T  tcgen05.mma kind::f16 (bf16 in, fp32 accumulate) into the TMEM
//                  S/P buffer g % 3 (g: the tile's index over the CTA's items)
//   softmax        two threads per row, each on half of the tile's keys (warps w and
//                  12 + w share TMEM lane quarter w): tcgen05.ld S_j, causal mask,
//                  exp2, row sums in fp32; P_j is split into bf16 hi + lo parts (hi = P
//                  truncated, lo = the remainder truncated: hi + lo within 2^-14 of P)
//                  and stored back over S_j in the same TMEM buffer (keys 64h..64h+63
//                  at columns 64h.., hi in 32 columns and lo in the next 32)
//   O += P_j V_j   two tcgen05.mma passes (A = P hi, then P lo, from TMEM; B = V_j
//                  from shared memory) into the item's TMEM accumulator O
// The split keeps the probabilities near fp32 precision: a single bf16 P is off by up
// to 2^-8 per weight, which rows attending only a few keys do not average away; with
// the split every output is within 2^-14 * max|v| of the exact weights' result.  A
// tile whose rows all attend at least p_single_min_keys keys (1024 by default) keeps a
// single bf16 P, rounded to nearest, as FlashAttention-style kernels do: there the
// rounding errors of many weights average out (for N(0,1) data their effect on an
// output has a standard deviation near 2^-8 / sqrt(3 n / e) for n keys, about 1.2e-4
// at n = 1024), and the P.V pass takes 8 MMAs instead of 16.
// The running max is updated lazily: O and l are rescaled only when a row's max
// grows by more than 2^8, which keeps P <= 256 and leaves the result exact.  With a
// single P, an item's tiles after its first take the exponentials against the running
// max first and skip the max pass when every row sum stays below 2^8 (no row grew).
//
// Three S/P buffers, one accumulator.  KV tile g of the CTA (counted over its items) is
// scored into TMEM S/P buffer g % 3; P_g goes back over S_g in the same buffer, and
// O += P_g V_g accumulates into one O for the item, so S_{g+3} may overwrite the buffer
// only once P_g V_g has run.  While the softmax works on tile g, the tensor pipe runs
// P_{g-1} V_{g-1} and the S products of up to two tiles ahead, so the chain S -> softmax
// -> P.V -> S of one buffer has two softmax passes to complete in.  One warp issues the
// S products, another the P.V products: MMAs into different accumulators are not
// ordered against each other, so each waits on the barriers of its own inputs.  K and
// V stages (3 each, tile g in stage g % 3) are released when their S and P.V have run,
// so the gathers of later tiles are in flight.  Each 16-token chunk of a tile (a
// 16-token block, or half of a 32-token one) arrives as ONE TMA box: at head_dim 128 a
// 4-D box (the chunk's 16 rows x 256 B viewed as 2 row groups x 2 column halves x 8
// rows x 128 B, 128-byte swizzle), so a K/V tile lands as [8-key group][column half]
// [8 rows][128 B]: a valid K-major operand (8-row atoms 2 KB apart) for S and MN-major
// operand (column halves 1 KB apart) for P.V; at head_dim 64 a 16-row x 64-column box,
// the tile one 64-column half with 8-row atoms 1 KB apart.  On the tile holding the
// last key a query tile needs, the P.V product skips the 16-key steps wholly past that
// key (P = 0 there), and the issuer zeroes the V rows of its last step past it (they
// may hold NaN from unused slots) once V has landed.
//
// Persistent CTAs.  A CTA pays about 5 us outside its tile loop (barrier and TMEM set-up,
// the first gathers and S, the epilogue), which nothing overlaps when each SM runs one
// CTA; with at most 128 requests (and outside cascade mode) the grid is one CTA per SM
// and each works through a share of the query tiles (the work items below), with the
// next item's Q, gathers and first S products under way while the softmax warps finish
// the current one.
//
// Measured costs per 128-key tile on GB300 (clock64 traces, isolated probes, and copies
// of this kernel with parts of the work removed): the 16 N = 128 MMAs of a single-P
// tile take the tensor pipe 1024 cycles (64 each at full rate), the softmax about 1450
// cycles on its two warpgroups, and a warp issuing TMA boxes about 100 cycles per box:
// with all 16 boxes of a tile from one warp the kernel took 0.372 ms on the 16 x
// 512-token batch with no softmax work at all, with K and V from two warps 0.308 ms.
// Shared memory serves about 160 KB a tile (S reads Q and K, P.V reads V, the copies
// write K and V) at up to 128 B a cycle.  A warp that issues MMAs gets only the issue
// slots its scheduler's softmax warps leave free, which is why the issue loops are short.
//
// Warp roles (512 threads, four warpgroups): warps 0-3 and 12-15 softmax (warps w and
// 12 + w own TMEM lanes 32w..32w+31, keys 0-63 and 64-127 of each tile; the partners
// agree per tile through a 64-thread named barrier), warp 4 barrier set-up + Q and K
// copies, warp 5 TMEM owner + S issuer, warp 6 P.V issuer, warp 7 V copies, warps 8-11
// epilogue (warp 8 + q reads lanes 32q..32q+31).  At the end of an item the softmax
// warps hand the rows' 1 / l to the epilogue warps through shared memory and go on with
// the next item; the epilogue warps wait for the item's last P.V product, read the
// accumulator out, store the output and release the accumulator.  Registers
// (setmaxnreg): softmax 192 a thread, copies and issuers 64, epilogue 64.  TMEM
// columns: S/P buffers at [0, 128), [128, 256) and [256, 384); O at [384, 384 + D).
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
constexpr int kHalf = kRows * 128;         // one 64-column half of the 128-row Q tile: 16 KB
constexpr int kStagesK = 3;                // K stages: freed right after S = Q K^T
constexpr int kStagesV = 3;                // V stages: freed after P.V
constexpr int kNumBars = 28;

constexpr int kMaxSchedReqs = 128;   // persistent scheduling ranks up to 128 requests

// Shared-memory geometry for head_dim D (64 or 128).
template <int D>
struct Geom {
    static constexpr int kHalves = D / 64;                // 64-column halves of a row
    static constexpr int kQBytes = kRows * D * 2;         // Q tile
    static constexpr int kTileBytes = kKeys * D * 2;      // one K or V stage
    static constexpr int kChunkBytes = kChunk * D * 2;    // 16 rows of one kv head
    static constexpr int kGroupBytes = 8 * D * 2;         // 8 key rows, every half
    static constexpr int kOffQ = 0;
    static constexpr int kOffK = kOffQ + kQBytes;
    static constexpr int kOffV = kOffK + kStagesK * kTileBytes;
    static constexpr int kOffBar = kOffV + kStagesV * kTileBytes;
    // barriers, then the TMEM address and abort flag, then the persistent schedule, then
    // the rows' 1 / l for the epilogue warps
    static constexpr int kOffSreq = kOffBar + kNumBars * 8 + 16;
    static constexpr int kOffOff = kOffSreq + kMaxSchedReqs * 2;
    static constexpr int kOffCoef = kOffOff + (kMaxSchedReqs + 1) * 4;
    // (the row coefficients, then an exchange array of the two softmax halves)
    static constexpr int kSmemBytes = kOffCoef + 2 * kRows * 4 + 1024;  // + align slack
};
constexpr int kSoftmaxWarps = 4;
constexpr int kProducerWarp = 4;
constexpr int kMmaWarp = 5;                // issues the S products; owns TMEM
constexpr int kPvWarp = 6;                 // issues the P.V products
constexpr int kProducerVWarp = 7;          // V copies (warp 4: Q and K copies)
constexpr int kEpilogueWarp = 8;           // warps 8-11: epilogue
constexpr int kSoftmaxBWarp = 12;          // warps 12-15: softmax, keys 64-127 of a tile
constexpr int kThreads = 512;
// Register split (setmaxnreg) of the four warpgroups: two softmax, copies + issuers,
// epilogue.  The sum over the 512 threads (128 x (2 x 192 + 64 + 64) = 65536) must not
// exceed what the launch provides (512 x the kernel's register count); the launcher
// checks it.
constexpr int kRegsSoftmax = 192;
constexpr int kRegsIssue = 64;
constexpr int kRegsEpilogue = 64;
constexpr uint32_t kTmemCols = 512;
constexpr int kSBufs = 3;                  // S/P buffers; buffer b at TMEM column 128 b
constexpr uint32_t kTmemO = 384;           // the O accumulator
static_assert(kStagesK == kSBufs && kStagesV == kSBufs, "tile g uses stage and buffer g % 3");
constexpr float kLazyRescale = 8.0f;       // log2 units
constexpr float kLazyLimit = 256.0f;       // 2^kLazyRescale
constexpr float kNoMax = -1.0e30f;         // running max before an item's first tile

// barrier indices: K/V stages and S/P buffers (the CTA's tile g uses stage and buffer
// g % 3).  BQ_EMPTY: every S of an item has run (the Q buffer may be reloaded); BO_FREE:
// the epilogue warps have read O out for an item; BEPI: the softmax warps have written an
// item's row coefficients; BCOEF_FREE: the epilogue warps have read them; BDRAIN: per
// issuing warp, at exit.
constexpr int BQ = 0, BK_FULL = 1, BK_EMPTY = 4, BV_FULL = 7, BV_EMPTY = 10, BS_FULL = 13,
              BP_FULL = 16, BPV_DONE = 19, BDRAIN = 22, BQ_EMPTY = 24, BO_FREE = 25,
              BEPI = 26, BCOEF_FREE = 27;

PKV_DEVINL void setmaxnreg_softmax() {
    asm volatile("setmaxnreg.inc.sync.aligned.u32 %0;" ::"n"(kRegsSoftmax));
}
PKV_DEVINL void setmaxnreg_issue() {
    asm volatile("setmaxnreg.dec.sync.aligned.u32 %0;" ::"n"(kRegsIssue));
}
PKV_DEVINL void setmaxnreg_epilogue() {
    asm volatile("setmaxnreg.dec.sync.aligned.u32 %0;" ::"n"(kRegsEpilogue));
}

// Named barrier `id` of the two partner softmax warps (64 threads).
PKV_DEVINL void pair_sync(uint32_t id) {
    asm volatile("bar.sync %0, 64;" ::"r"(id) : "memory");
}
// The same barrier, returning whether `v` holds for all 64 threads.
PKV_DEVINL bool pair_all(uint32_t id, bool v) {
    uint32_t r;
    asm volatile(
        "{\n\t.reg .pred p, q;\n\tsetp.ne.u32 p, %1, 0;\n\t"
        "bar.red.and.pred q, %2, 64, p;\n\tselp.u32 %0, 1, 0, q;\n\t}"
        : "=r"(r)
        : "r"(static_cast<uint32_t>(v)), "r"(id)
        : "memory");
    return r != 0;
}

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

// ------------------------------------------------------------------ work items
// An item is one 128-row query tile of one request and kv head.  With `persistent`
// set the grid holds at most one CTA per SM, and CTA b works through the items k =
// m P + (b, or P - 1 - b for odd m), m = 0, 1, ... (P CTAs, a snake over the item list)
// of a list that ranks the requests by their key count, longest first, and within a
// request takes the query tiles last-first: the longest items are spread over the CTAs
// first and each CTA's total comes out near the mean.  Each role walks the same list, so
// barrier phases carry over from one item to the next and the next item's gathers and
// first S products start while the softmax warps finish the current one.  Otherwise
// CTA (x, y, z) takes the single item (query tile x, kv head y, request z -- in
// cascade mode split z).

struct ItemParams {
    int kvh, r, n, c, t0, max_lim, j0, ntiles, qoff, qrow0;
    bool p_single;
};

// Parameters of item (qt, kvh, r); false when it has no rows (t0 >= n), no tile, or
// keys past its table (then PKV_ERR_OOB is raised when `report`).
template <int G>
PKV_DEVINL bool item_params(const PrefillArgs& a, int qt, int kvh, int r, bool report,
                            ItemParams& p) {
    constexpr int TOK = kRows / G;
    const bool cascade = a.cascade != 0;   // rows = sequences over the c shared keys
    p.kvh = kvh;
    p.r = r;
    p.n = cascade ? a.cascade_rows : __ldg(a.new_lens + r);
    p.c = cascade ? a.cascade_keys : __ldg(a.cached_lens + r);
    p.t0 = qt * TOK;
    if (p.t0 >= p.n) return false;
    const int L = cascade ? p.c : p.c + p.n;   // keys in the pool for this request
    if (p.c < 0 || L <= 0 || L > a.max_blocks_per_seq * a.block_size) {
        if (report) raise_status(a.status, PKV_ERR_OOB);
        return false;
    }
    const int i_last = min(p.t0 + TOK, p.n) - 1;
    p.max_lim = cascade ? p.c - 1 : p.c + i_last;   // last key any row of the tile sees
    // KV tiles [j0, j0 + ntiles): all of them, or in cascade mode the range of split r
    // (its partial goes to slot r; the host sizes the splits so that none is empty).
    p.j0 = cascade ? r * a.cascade_tiles_per_split : 0;
    p.ntiles = cascade ? min(p.max_lim / kKeys + 1 - p.j0, a.cascade_tiles_per_split)
                       : p.max_lim / kKeys + 1;
    if (p.ntiles <= 0) return false;
    p.qoff = cascade ? 0 : __ldg(a.q_offsets + r);
    p.qrow0 = p.qoff + p.t0;   // first token row of the tile in q / out
    // Every row of the tile attends at least min_keys keys (its first token the fewest).
    const int min_keys = cascade ? p.c : p.c + p.t0 + 1;
    p.p_single = min_keys >= a.p_single_min_keys;
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
        const int nq = (s.off(cur.rho + 1) - s.off(cur.rho)) / a.num_kv_heads;
        if (item_params<G>(a, nq - 1 - rem / a.num_kv_heads, rem % a.num_kv_heads,
                           s.sreq(cur.rho), report, p))
            return true;
    }
}

template <int D, int G>
__global__ void __launch_bounds__(kThreads, 1)
prefill_tcgen05_kernel(const __grid_constant__ CUtensorMap tm_q,
                       const __grid_constant__ CUtensorMap tm_k,
                       const __grid_constant__ CUtensorMap tm_v, const PrefillArgs a,
                       const int persistent, const int test_stall) {
    using GM = Geom<D>;
    constexpr int TOK = kRows / G;
    extern __shared__ uint8_t smem_raw[];
    uint8_t* smem = reinterpret_cast<uint8_t*>(
        (reinterpret_cast<uintptr_t>(smem_raw) + 1023) & ~static_cast<uintptr_t>(1023));

    griddep_wait();
    griddep_launch_dependents();
    const int warp = threadIdx.x >> 5;
    const int lane = threadIdx.x & 31;
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
        // item list: rank rho holds ceil(n / TOK) query tiles x the kv heads.
        const int R = a.num_reqs;
        for (int t = threadIdx.x; t < R; t += kThreads)   // off[] holds the key counts first
            off[t] = __ldg(a.cached_lens + t) + __ldg(a.new_lens + t);
        __syncthreads();
        for (int t = threadIdx.x; t < R; t += kThreads) {
            const int kt = off[t];
            int rank = 0;
            for (int u = 0; u < R; ++u) {
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
                if (rho < R) {
                    const int nn = __ldg(a.new_lens + sreq[rho]);
                    v = nn > 0 ? (nn + TOK - 1) / TOK * a.num_kv_heads : 0;
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
                if (rho < R) off[rho] = run;
                run += cnt[e];
                if (rho == R - 1) off[R] = run;
            }
        }
        __syncthreads();
    }

    if (warp == kProducerWarp) {
        if (lane == 0) {
            mbar_init(&bars[BQ], 1);
            mbar_init(&bars[BQ_EMPTY], 1);
            mbar_init(&bars[BO_FREE], 4);   // the epilogue warps
            mbar_init(&bars[BEPI], kSoftmaxWarps);
            mbar_init(&bars[BCOEF_FREE], 4);
            for (int st = 0; st < kSBufs; ++st) {
                mbar_init(&bars[BK_FULL + st], 1);
                mbar_init(&bars[BK_EMPTY + st], 1);
                mbar_init(&bars[BV_FULL + st], 1);
                mbar_init(&bars[BV_EMPTY + st], 1);
                mbar_init(&bars[BS_FULL + st], 1);
                mbar_init(&bars[BP_FULL + st], 2 * kSoftmaxWarps);
                mbar_init(&bars[BPV_DONE + st], 1);
            }
            mbar_init(&bars[BDRAIN + 0], 1);
            mbar_init(&bars[BDRAIN + 1], 1);
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
    const uint32_t sK = smem_u32(smem + GM::kOffK);
    const uint32_t sV = smem_u32(smem + GM::kOffV);

    if (warp >= kSoftmaxWarps && warp < kEpilogueWarp) {
    setmaxnreg_issue();
    if (warp == kProducerWarp || warp == kProducerVWarp) {
        // ------------------------------------------------------------ TMA producers
        // Warp 4 copies Q and K, warp 7 V: a warp spends about 100 cycles per box it
        // issues, and one warp issuing both K and V (16 boxes per KV tile) set the pace of
        // the whole kernel.  Each warp runs the loop whole: each lane prefetches the block
        // id of one 16-token chunk (32 chunks = 4 KV tiles per refill, independent loads),
        // lane 0 sets the byte counts and lane b < 8 issues the box of chunk b of the
        // tile.  A chunk is a whole block (block size 16) or rows 16 h .. 16 h + 15 of one
        // (block size 32).  Stages and their phases count the CTA's tiles over all its
        // items (g); the Q of an item is loaded once every S product of the previous item
        // has run.
        const bool doqk = warp == kProducerWarp;
        Cursor cur;
        ItemParams p;
        int it = 0, g = 0;
        int k_issued = 0, v_issued = 0;   // tiles whose K / V copies were issued
        bool ok = true;
        while (ok && next_item<G>(a, sch, cur, lane == 0, p)) {
            const int32_t* bt =
                a.block_tables + static_cast<size_t>(cascade ? 0 : p.r) * a.max_blocks_per_seq;
            const int nchunks = p.max_lim / kChunk + 1;
            if (doqk && it >= 1 && !wait_bar_warp(ctl, BQ_EMPTY, (it - 1) & 1, lane)) break;
            // Test hook (zero in normal use): CTA 0 arms its first Q barrier for 16 bytes
            // more than the Q copy delivers, so the issuers' wait for it runs out of time
            // (PKV_ERR_TIMEOUT) while the copy still lands.
            const bool stall = test_stall && it == 0 && blockIdx.x == 0 && blockIdx.y == 0 &&
                               blockIdx.z == 0;
            if (doqk && lane == 0) {
                mbar_arrive_expect_tx(&bars[BQ], GM::kQBytes + (stall ? 16u : 0u));
#pragma unroll
                for (int h = 0; h < GM::kHalves; ++h)
                    tma_load_3d(smem + GM::kOffQ + h * kHalf, &tm_q, 64 * h, p.kvh * G, p.qrow0,
                                &bars[BQ]);
            }
            ++it;
            int ids = 0;
            for (int jt = 0; jt < p.ntiles; ++jt, ++g) {
                constexpr int kPerTile = kKeys / kChunk;   // 8 chunks per KV tile
                if ((jt & 3) == 0) {
                    const int i = (p.j0 + jt) * kPerTile + lane;
                    ids = (i < nchunks) ? __ldg(bt + (i >> csh)) : 0;
                }
                const int sk = g % kStagesK;
                const int sv = g % kStagesV;
                const int nb = min(kPerTile, nchunks - (p.j0 + jt) * kPerTile);
                int phys = __shfl_sync(0xffffffffu, ids, ((jt & 3) * kPerTile) + (lane & 7));
                if (phys < 0 || phys >= a.num_blocks) {
                    if (lane < nb) raise_status(a.status, PKV_ERR_OOB);
                    phys = 0;  // keep the byte count; the output is flagged invalid
                }
                const int chunk = (p.j0 + jt) * kPerTile + (lane & 7);
                const int row = (phys * a.num_kv_heads + p.kvh) * a.block_size +
                                (chunk & ((1 << csh) - 1)) * kChunk;
                // K of tile g: its stage is free once S of tile g - kStagesK has run.  The
                // warp stays converged: lane 0 sets the byte count and lanes b < nb issue
                // the boxes through predicated instructions.
                if (doqk && g >= kStagesK &&
                    !wait_bar_warp(ctl, BK_EMPTY + sk, ((g / kStagesK) - 1) & 1, lane)) {
                    ok = false;
                    break;
                }
                mbar_arrive_expect_tx_if(doqk && lane == 0, &bars[BK_FULL + sk], nb * GM::kChunkBytes);
                {
                    uint8_t* dst = smem + GM::kOffK + sk * GM::kTileBytes + lane * GM::kChunkBytes;
                    if constexpr (D == 128)
                        tma_load_4d_if(doqk && lane < nb, dst, &tm_k, 0, 0, 0, row / 8, &bars[BK_FULL + sk]);
                    else
                        tma_load_2d_if(doqk && lane < nb, dst, &tm_k, 0, row, &bars[BK_FULL + sk]);
                }
                k_issued += doqk;
                // V of tile g: its stage is free once P.V of tile g - kStagesV has run.
                if (!doqk && g >= kStagesV &&
                    !wait_bar_warp(ctl, BV_EMPTY + sv, ((g / kStagesV) - 1) & 1, lane)) {
                    ok = false;
                    break;
                }
                mbar_arrive_expect_tx_if(!doqk && lane == 0, &bars[BV_FULL + sv], nb * GM::kChunkBytes);
                {
                    uint8_t* dst = smem + GM::kOffV + sv * GM::kTileBytes + lane * GM::kChunkBytes;
                    if constexpr (D == 128)
                        tma_load_4d_if(!doqk && lane < nb, dst, &tm_v, 0, 0, 0, row / 8, &bars[BV_FULL + sv]);
                    else
                        tma_load_2d_if(!doqk && lane < nb, dst, &tm_v, 0, row, &bars[BV_FULL + sv]);
                }
                v_issued += !doqk;
            }
        }
        // Drain (also after an abort): wait, bounded, until the last copy issued into
        // every stage has landed, so that no TMA write into shared memory outlives the
        // CTA.  No later copy goes into those stages, so the phases cannot move on.
        if (doqk && it >= 1) mbar_wait_warp(&bars[BQ], (it - 1) & 1, a.status);
        for (int st = 0; st < kStagesK; ++st) {
            if (k_issued > st) {
                const int last = st + kStagesK * ((k_issued - 1 - st) / kStagesK);
                mbar_wait_warp(&bars[BK_FULL + st], (last / kStagesK) & 1, a.status);
            }
            if (v_issued > st) {
                const int last = st + kStagesV * ((v_issued - 1 - st) / kStagesV);
                mbar_wait_warp(&bars[BV_FULL + st], (last / kStagesV) & 1, a.status);
            }
        }
    } else if (warp == kMmaWarp) {
        // ------------------------------------------------------------ S issuer
        // S_g = Q K_g^T into S/P buffer g % 3 once K_g has landed and the buffer's
        // previous tile g - 3 has been consumed by its P.V product (P_{g-3} lies in the
        // same columns); at an item's first tile, once the item's Q has landed.  After an
        // item's last S it signals that the Q buffer may take the next item's Q
        // (BQ_EMPTY).  The issuing warps share their schedulers with softmax warps and
        // get only the issue slots those leave free, so the loops are short: the whole
        // warp runs them converged (all lanes poll, one leader lane issues through
        // predicated instructions) and the descriptors are precomputed halves plus
        // constant offsets.
        constexpr uint32_t idesc_qk = idesc_bf16_f32(kRows, kKeys, false, false);
        constexpr uint32_t hi_q = smem_desc_sw128_hi(1024);          // Q: 8-row atoms 1 KB apart
        constexpr uint32_t hi_kv = smem_desc_sw128_hi(GM::kGroupBytes);  // K: 8-key groups
        const uint32_t lo_q = smem_desc_sw128_lo(sQ, 16);
        const uint32_t lo_k = smem_desc_sw128_lo(sK, 16);
        const bool leader = elect_one();   // issues every MMA and commit of this warp
        Cursor cur;
        ItemParams p;
        int it = 0, g = 0;
        bool ok = true;
        while (ok && next_item<G>(a, sch, cur, false, p)) {
            ok = wait_bar_warp(ctl, BQ, it & 1, lane);
            for (int j = 0; ok && j < p.ntiles; ++j, ++g) {
                const int b = g % kSBufs;
                if (!wait_bar_warp(ctl, BK_FULL + b, (g / kSBufs) & 1, lane)) { ok = false; break; }
                if (g >= kSBufs &&
                    !wait_bar_warp(ctl, BPV_DONE + b, ((g / kSBufs) - 1) & 1, lane)) {
                    ok = false;
                    break;
                }
                tc_fence_after();
                const uint32_t tS = tmem + b * 128;
                const uint32_t lk = lo_k + ((b * GM::kTileBytes) >> 4);
#pragma unroll
                for (int ks = 0; ks < D / 16; ++ks) {
                    const uint32_t kc = ((ks & 3) * 32) >> 4;   // 16 columns = 32 B
                    umma_bf16_if(leader, tS,
                                 desc_join(lo_q + (((ks >> 2) * kHalf) >> 4) + kc, hi_q),
                                 desc_join(lk + (((ks >> 2) * 1024) >> 4) + kc, hi_kv),
                                 idesc_qk, ks > 0);
                }
                umma_commit_if(leader, &bars[BS_FULL + b]);
                umma_commit_if(leader, &bars[BK_EMPTY + b]);
                if (j + 1 == p.ntiles) umma_commit_if(leader, &bars[BQ_EMPTY]);   // last S
            }
            ++it;
        }
        // Drain (also after an abort): every MMA this warp issued completes before the
        // TMEM is freed at the end of the kernel.
        umma_commit_if(leader, &bars[BDRAIN + 0]);
        mbar_wait_warp(&bars[BDRAIN + 0], 0, a.status);
    } else if (warp == kPvWarp) {
        // ------------------------------------------------------------ P.V issuer
        // O += P_g V_g once the softmax warps have written P_g into buffer g % 3 and V_g
        // has landed; an item's first P.V overwrites O, once the epilogue warps have read
        // the previous item's O out (BO_FREE).  The P.V products all accumulate into the
        // one O and run in issue order.
        constexpr uint32_t idesc_pv = idesc_bf16_f32(kRows, D, false, true);
        constexpr uint32_t hi_kv = smem_desc_sw128_hi(GM::kGroupBytes);  // V: 8-key groups
        const uint32_t lo_v = smem_desc_sw128_lo(sV, 1024);          // V: column halves 1 KB apart
        const uint32_t tO = tmem + kTmemO;
        const bool leader = elect_one();
        Cursor cur;
        ItemParams p;
        int it = 0, g = 0;
        bool ok = true;
        while (ok && next_item<G>(a, sch, cur, false, p)) {
            for (int j = 0; ok && j < p.ntiles; ++j, ++g) {
                const int b = g % kSBufs;
                if (!wait_bar_warp(ctl, BP_FULL + b, (g / kSBufs) & 1, lane)) { ok = false; break; }
                if (!wait_bar_warp(ctl, BV_FULL + b, (g / kSBufs) & 1, lane)) { ok = false; break; }
                if (j == 0 && it >= 1 && !wait_bar_warp(ctl, BO_FREE, (it - 1) & 1, lane)) {
                    ok = false;
                    break;
                }
                // Keys past the last one this tile needs are masked for every row (P = 0),
                // but their V rows may hold anything (NaN in unused slots, stale data where
                // no block was loaded this tile).  The P.V product skips the 16-key steps
                // that lie wholly past that key, and the rows of the last step past it are
                // zeroed, now that V_g has landed, so that 0 * V stays 0.
                const int kbase = (p.j0 + j) * kKeys;
                const int nvalid = min(kKeys, p.max_lim - kbase + 1);   // >= 1
                const int ksteps = (nvalid + 15) >> 4;
                if (nvalid < ksteps * 16) {
                    const uint4 z = make_uint4(0, 0, 0, 0);
                    // rows nvalid .. 16 ksteps - 1, 8 pieces per 128-byte half: lane = piece
                    // 8 rows apart so that each store instruction touches 8 rows of an atom
                    const int rows = ksteps * 16 - nvalid;
                    for (int t = lane; t < rows * 8 * GM::kHalves; t += 32) {
                        const int row = nvalid + t / (8 * GM::kHalves);
                        const int hh = (t / 8) % GM::kHalves;
                        const int jj = t & 7;
                        uint8_t* vrow = smem + GM::kOffV + b * GM::kTileBytes +
                                        (row >> 3) * GM::kGroupBytes + (row & 7) * 128;
                        *reinterpret_cast<uint4*>(vrow + hh * 1024 + ((jj ^ (row & 7)) << 4)) = z;
                    }
                    fence_proxy_async_smem();
                    __syncwarp();
                }
                tc_fence_after();
                const uint32_t tS = tmem + b * 128;
                const uint32_t lv = lo_v + ((b * GM::kTileBytes) >> 4);
                // V as the MN-major B operand: 16 keys = two 8-key groups.
#pragma unroll
                for (int ks = 0; ks < kKeys / 16; ++ks) {
                    const uint64_t bv = desc_join(lv + ((ks * 2 * GM::kGroupBytes) >> 4), hi_kv);
                    // P of keys 16 ks .. 16 ks + 15: columns 64 h + 8 (ks % 4), h = ks / 4
                    // (the softmax half that wrote it), lo 32 columns further
                    const uint32_t tp = tS + (ks >> 2) * 64 + (ks & 3) * 8;
                    umma_bf16_ta_if(leader && ks < ksteps, tO, tp, bv, idesc_pv,
                                    (j > 0) || (ks > 0));
                    if (!p.p_single)
                        umma_bf16_ta_if(leader && ks < ksteps, tO, tp + 32, bv, idesc_pv, true);
                }
                umma_commit_if(leader, &bars[BPV_DONE + b]);
                umma_commit_if(leader, &bars[BV_EMPTY + b]);
            }
            ++it;
        }
        umma_commit_if(leader, &bars[BDRAIN + 1]);
        mbar_wait_warp(&bars[BDRAIN + 1], 0, a.status);
    }
    } else if (warp >= kEpilogueWarp && warp < kSoftmaxBWarp) {
        setmaxnreg_epilogue();
        // ------------------------------------------------------------ epilogue
        // Warp 8 + q reads TMEM lanes 32 q .. 32 q + 31 (its lane quarter).  Per item: once
        // the softmax warps have written the rows' coefficients 1 / l (BEPI) and the
        // item's last P.V product is done, O / l is stored, and the accumulator and the
        // coefficients are released for the next item.  The same item list as every role.
        const int q4 = warp & 3;
        const int row = q4 * 32 + lane;   // == TMEM lane
        const uint32_t lane_addr = static_cast<uint32_t>(q4 * 32) << 16;
        const float* coef = reinterpret_cast<const float*>(smem + GM::kOffCoef);
        Cursor cur;
        ItemParams p;
        int e = 0;   // items ended
        int g = 0;   // the CTA's tiles over all items
        while (next_item<G>(a, sch, cur, false, p)) {
            g += p.ntiles;
            const int gl = g - 1;   // the item's last tile
            bool fin = wait_bar_warp(ctl, BEPI, e & 1, lane);
            if (fin) fin = wait_bar_warp(ctl, BPV_DONE + gl % kSBufs, (gl / kSBufs) & 1, lane);
            if (!fin) break;
            tc_fence_after();
            const float c = coef[row];
            const int tok = p.t0 + row / G;
            const bool row_valid = tok < p.n;
            const size_t orow_idx = static_cast<size_t>(p.qoff + tok) * a.num_q_heads +
                                    p.kvh * G + row % G;
            uint16_t* orow = static_cast<uint16_t*>(a.out) + orow_idx * D;
            const size_t prow = orow_idx * a.max_parts_total + p.r;   // cascade: slot = split
#pragma unroll
            for (int q2 = 0; q2 < D / 32; ++q2) {
                float o[32];
                tmem_ld32(tmem + lane_addr + kTmemO + q2 * 32, o);
                tmem_wait_ld();
#pragma unroll
                for (int k = 0; k < 32; ++k) o[k] *= c;
                if (cascade && row_valid) {
                    float* dst = a.o_part + prow * D + q2 * 32;
#pragma unroll
                    for (int k = 0; k < 32; k += 4)
                        *reinterpret_cast<float4*>(dst + k) =
                            make_float4(o[k], o[k + 1], o[k + 2], o[k + 3]);
                } else if (row_valid) {
#pragma unroll
                    for (int k = 0; k < 32; k += 8) {
                        uint4 w;
                        w.x = pack_bf16x2(o[k], o[k + 1]);
                        w.y = pack_bf16x2(o[k + 2], o[k + 3]);
                        w.z = pack_bf16x2(o[k + 4], o[k + 5]);
                        w.w = pack_bf16x2(o[k + 6], o[k + 7]);
                        *reinterpret_cast<uint4*>(orow + q2 * 32 + k) = w;
                    }
                }
            }
            // O of this item and the coefficients are read: the P.V issuer may start the
            // next item's products, the softmax warps may write the next coefficients.
            tc_fence_before();
            __syncwarp();
            mbar_arrive_if(lane == 0, &bars[BO_FREE]);
            mbar_arrive_if(lane == 0, &bars[BCOEF_FREE]);
            ++e;
        }
    } else {
        setmaxnreg_softmax();
        // ------------------------------------------------------------ softmax
        // Two warpgroups: warps 0-3 take keys 0-63 of every KV tile, warps 12-15 keys
        // 64-127.  Warp w and warp 12 + w share TMEM lane quarter w % 4 (rows 32 w ..
        // 32 w + 31), one thread per row each, and run on the same scheduler, where each
        // hides the other's latencies.  The partners keep one running max per row and a
        // row sum each; they meet at named barrier 1 + w % 4 (64 threads) to agree, per
        // tile, whether the optimistic pass holds for the whole row and whether to go on
        // at all (every exit is joint, so neither can be left waiting at a barrier), to
        // exchange their tile maxima on the full pass, and to add their row sums at the
        // end of an item.  P of keys 64 h .. 64 h + 63 goes to columns 64 h .. (hi: 32
        // columns, lo: the next 32) of the buffer: each half stores only over the S it has
        // loaded itself.
        const int half = warp >= kSoftmaxBWarp ? 1 : 0;
        const int wq = warp & 3;
        const int row = wq * 32 + lane;           // == TMEM lane
        const uint32_t bar_id = 1 + wq;           // the partners' named barrier
        const uint32_t lane_addr = static_cast<uint32_t>(wq * 32) << 16;
        const uint32_t cbase = 64 * half;         // this half's S / P columns
        float* xch = reinterpret_cast<float*>(smem + GM::kOffCoef) + kRows;   // exchange
        const float sl2 = a.scale_log2;
        Cursor cur;
        ItemParams p;
        int g = 0;          // the CTA's tiles over all items
        int ended = 0;      // items handed over to the epilogue warps
        bool ok = true;
        bool have = next_item<G>(a, sch, cur, false, p);
        while (ok && have) {
        const int tok = p.t0 + row / G;
        const bool row_valid = tok < p.n;
        const size_t orow_idx = static_cast<size_t>(p.qoff + tok) * a.num_q_heads +
                                p.kvh * G + row % G;
        const int prow_slot = p.r;
        const int lim = cascade ? p.c - 1 : (row_valid ? p.c + tok : p.c + p.n - 1);  // last key seen
        const bool p_single = p.p_single;
        const int ntiles = p.ntiles;
        // Running max (log2 domain, the same in both halves) and this half's row sum.
        float m_run = kNoMax;
        float l_run = 0.f;
        for (int jt = 0; jt < ntiles; ++jt, ++g) {
            const int b = g % kSBufs;
            const uint32_t tS = tmem + lane_addr + b * 128 + cbase;
            const int kbase = (p.j0 + jt) * kKeys + 64 * half;   // this half's first key
            bool okw = wait_bar_warp(ctl, BS_FULL + b, (g / kSBufs) & 1, lane);
            float x[64];
            // Optimistic pass (one bf16 P, after an item's first tile): exponentials
            // against the running max, with no max pass.  A half-row sum below 2^8 bounds
            // each of its p below 2^8; when that holds for both halves of every row the
            // rows' maxima did not grow past the lazy threshold, and these are the P and
            // sums the full pass would compute.  Otherwise both halves load S again (still
            // intact: nothing was stored over it yet) and take the full pass.
            const bool try_fast = p_single && jt >= 1;
            bool good = false;
            uint32_t ph[32];
            float rs = 0.f;
            if (okw) {
                tc_fence_after();
                tmem_ld32(tS, *reinterpret_cast<float(*)[32]>(&x[0]));
                tmem_ld32(tS + 32, *reinterpret_cast<float(*)[32]>(&x[32]));
                tmem_wait_ld();
                if (kbase + 63 > lim) {
#pragma unroll
                    for (int k = 0; k < 64; ++k) x[k] = (kbase + k <= lim) ? x[k] : -INFINITY;
                }
                if (try_fast) {
                    float rs8[8];
#pragma unroll
                    for (int u = 0; u < 8; ++u) rs8[u] = 0.f;
#pragma unroll
                    for (int e = 0; e < 32; ++e) {
                        float a0, a1;
                        ffma2(a0, a1, x[2 * e], x[2 * e + 1], sl2, sl2, -m_run, -m_run);
                        const float p0 = fast_exp2(a0);
                        const float p1 = fast_exp2(a1);
                        const int u = (e & 3) * 2;
                        ffma2(rs8[u], rs8[u + 1], p0, p1, 1.f, 1.f, rs8[u], rs8[u + 1]);
                        ph[e] = pack_bf16x2(p0, p1);
                    }
                    rs = ((rs8[0] + rs8[1]) + (rs8[2] + rs8[3])) +
                         ((rs8[4] + rs8[5]) + (rs8[6] + rs8[7]));
                    good = rs < kLazyLimit;
                }
            }
            if (pair_all(bar_id, okw && good)) {
                tmem_st32(tS, *reinterpret_cast<const float(*)[32]>(&ph[0]));
                l_run += rs;
            } else {
                // Joint exit when either half failed its wait (or saw another role abort).
                if (!pair_all(bar_id, okw)) { ok = false; break; }
                if (try_fast) {
                    tmem_ld32(tS, *reinterpret_cast<float(*)[32]>(&x[0]));
                    tmem_ld32(tS + 32, *reinterpret_cast<float(*)[32]>(&x[32]));
                    tmem_wait_ld();
                    if (kbase + 63 > lim) {
#pragma unroll
                        for (int k = 0; k < 64; ++k)
                            x[k] = (kbase + k <= lim) ? x[k] : -INFINITY;
                    }
                }
                // Full pass.  This half's max over 4 independent chains of three-input
                // max; the partners exchange theirs through shared memory (half 0 writes,
                // half 1 takes the maximum of both and writes it back).
                float m4[4];
#pragma unroll
                for (int u = 0; u < 4; ++u) m4[u] = -INFINITY;
#pragma unroll
                for (int k = 0; k < 64; k += 2)
                    m4[(k >> 1) & 3] = fmax3(m4[(k >> 1) & 3], x[k], x[k + 1]);
                float mx = fmaxf(fmaxf(m4[0], m4[1]), fmaxf(m4[2], m4[3]));
                if (half == 0) xch[row] = mx;
                pair_sync(bar_id);
                if (half == 1) {
                    mx = fmaxf(mx, xch[row]);
                    xch[row] = mx;
                }
                pair_sync(bar_id);
                if (half == 0) mx = xch[row];
                const float m_tile = mx * sl2;   // scale > 0: max commutes with scaling
                const float m_used = m_run;
                const bool grow = m_tile > m_used + kLazyRescale;
                const float m_cur = grow ? m_tile : m_used;
                // 1 unless grow; 0 at the item's first tile.  A row with no key in this
                // tile keeps m_cur finite (kNoMax at worst), so its p are exp2(-inf) = 0.
                const float alpha = fast_exp2(m_used - m_cur);
                // O is rescaled only when some row of the warp grew its max (the partner
                // warp has the same rows, so it decides alike), once the P.V products
                // issued so far (the last one, of tile g - 1, completes last) are done;
                // each half rescales half of O's columns.  The item's first P.V overwrites
                // O, so its first tile needs none.  A failed wait is carried to the next
                // joint decision.
                if (jt >= 1 && __any_sync(0xffffffffu, grow)) {
                    const int gp = g - 1;
                    okw = wait_bar_warp(ctl, BPV_DONE + gp % kSBufs, (gp / kSBufs) & 1, lane);
                    if (okw) {
                        tc_fence_after();
#pragma unroll
                        for (int q = 0; q < D / 64; ++q) {
                            float o[32];
                            const uint32_t ta =
                                tmem + lane_addr + kTmemO + half * (D / 2) + q * 32;
                            tmem_ld32(ta, o);
                            tmem_wait_ld();
#pragma unroll
                            for (int e = 0; e < 32; ++e) o[e] *= alpha;
                            tmem_st32(ta, o);
                        }
                    }
                }
                float rs8[8];
#pragma unroll
                for (int u = 0; u < 8; ++u) rs8[u] = 0.f;
                if (p_single) {
                    // One bf16 P per weight (round to nearest) in 32 columns.
#pragma unroll
                    for (int e = 0; e < 32; ++e) {
                        float a0, a1;
                        ffma2(a0, a1, x[2 * e], x[2 * e + 1], sl2, sl2, -m_cur, -m_cur);
                        const float p0 = fast_exp2(a0);
                        const float p1 = fast_exp2(a1);
                        const int u = (e & 3) * 2;
                        // row sums by fma with 1 (exact, one rounding as an add)
                        ffma2(rs8[u], rs8[u + 1], p0, p1, 1.f, 1.f, rs8[u], rs8[u + 1]);
                        ph[e] = pack_bf16x2(p0, p1);
                    }
                    tmem_st32(tS, *reinterpret_cast<const float(*)[32]>(&ph[0]));
                } else {
                    // hi (p truncated to bf16) in 32 columns, lo (the exact remainder
                    // p - hi, truncated) in the next 32: hi + lo is within 2^-14 of p
                    // (relative), from byte permutes instead of conversions.
#pragma unroll
                    for (int q = 0; q < 2; ++q) {
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
                                  __uint_as_float(__float_as_uint(p1) & 0xffff0000u), -1.f,
                                  -1.f, p0, p1);
                            plo[e] = pack_bf16x2_trunc(r0, r1);
                        }
                        tmem_st16(tS + q * 16, phi);
                        tmem_st16(tS + 32 + q * 16, plo);
                    }
                }
                const float rsf = ((rs8[0] + rs8[1]) + (rs8[2] + rs8[3])) +
                                  ((rs8[4] + rs8[5]) + (rs8[6] + rs8[7]));
                l_run = l_run * alpha + rsf;
                m_run = m_cur;
            }
            tmem_wait_st();
            tc_fence_before();
            __syncwarp();
            mbar_arrive_if(lane == 0, &bars[BP_FULL + b]);
        }
        if (!ok) break;
        // The next item's parameters, looked up now so that their loads overlap the
        // hand-over below rather than delay the next item's first tile.
        ItemParams pn;
        const bool have_next = next_item<G>(a, sch, cur, false, pn);
        // ------------------------------------------------------------ hand-over
        // Half 1 passes its row sums to half 0 (the exchange array is free once both
        // passed the first barrier).  Half 0 writes 1 / l for the epilogue warps, which
        // scale O once the item's last P.V product is done, while the softmax warps go on
        // with the next item; the coefficients of the previous item must have been read
        // first (BCOEF_FREE).  Every row sees the item's first key, so l > 0.
        {
            pair_sync(bar_id);
            if (half == 1) xch[row] = l_run;
            pair_sync(bar_id);
            bool oke = true;
            if (half == 0) {
                const float l = l_run + xch[row];
                oke = ended == 0 || wait_bar_warp(ctl, BCOEF_FREE, (ended - 1) & 1, lane);
                if (oke) {
                    float* coef = reinterpret_cast<float*>(smem + GM::kOffCoef);
                    coef[row] = 1.f / l;
                    if (cascade && row_valid) {
                        const size_t prow = orow_idx * a.max_parts_total + prow_slot;
                        a.m_part[prow] = m_run;   // log2 domain, as the decode partials
                        a.l_part[prow] = l;
                    }
                    __syncwarp();
                    mbar_arrive_if(lane == 0, &bars[BEPI]);
                }
            }
            if (!pair_all(bar_id, oke)) break;
            ++ended;
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
        const int need = 128 * (2 * kRegsSoftmax + kRegsIssue + kRegsEpilogue);
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
    const int qtiles = (a.max_new + TOK - 1) / TOK;
    // Persistent CTAs walking the ranked item list, at most one per SM; not for the
    // cascade's prefix pass, which is meant to hold few SMs beside the suffix decode.
    const int persistent = (!a.cascade && a.num_reqs <= kMaxSchedReqs) ? 1 : 0;
    dim3 grid(qtiles, a.num_kv_heads, a.num_reqs);
    if (persistent) {
        const int64_t items = static_cast<int64_t>(qtiles) * a.num_kv_heads * a.num_reqs;
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
