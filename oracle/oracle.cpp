// Reference oracle for paged-KV attention.  TEST INFRASTRUCTURE ONLY.
//
// This file is a plain, slow, fp64 CPU statement of what the paged attention
// path computes.  Only the test suite, the smoke check and the CPU-baseline leg
// of the benchmark load it; the product library never links, loads or calls
// it, and it shares no code, header or table with the CUDA path.
//
// What it follows (page, section):
//  * "Paged Attention for Efficient Memory Management" (krlt.com Triptych day
//    152), body: the cache is cut into blocks of B tokens; each sequence holds a
//    block table mapping logical block indices to physical block ids in one
//    global pool; writes append in the current block; the attention kernel
//    "chases the block table".  The same page states that the scheme changes
//    layout only, not the attention scores.
//  * "PagedAttention and RadixAttention: Let's Talk About KV Cache" (aitalk.it),
//    section "PagedAttention: Memory Like an Operating System": the page table
//    is consulted at attention time to gather the blocks, and paging "does not
//    alter the attention algorithm".
//
// Because paging leaves the arithmetic untouched, the oracle is that plain
// definition written out: gather the sequence's K and V through the block
// table into contiguous fp64 arrays, then run max-subtracted softmax attention
// in fp64.  Readings of points the pages leave open:
//  * pool layout [num_blocks][num_kv_heads][block_size][head_dim], slot =
//    block * block_size + offset (the pages fix no layout);
//  * query head h reads kv head h / (Hq / Hkv) (contiguous GQA grouping);
//  * a decode query attends to all context_len keys, its own key included;
//  * prefill row i of a request with c cached tokens attends keys 0..c+i;
//  * a negative slot in kv_append means "skip this row" (padding).
//
// Element types: dtype 0 = IEEE fp32, dtype 1 = bfloat16 (upper 16 bits of an
// fp32).  Both widen to double exactly.

#include <atomic>
#include <cmath>
#include <cstdint>
#include <cstring>
#include <thread>
#include <vector>

namespace {

inline double load_elem(const void* base, int dtype, int64_t idx) {
    if (dtype == 0) {
        float f;
        std::memcpy(&f, static_cast<const char*>(base) + idx * 4, 4);
        return static_cast<double>(f);
    }
    uint16_t h;
    std::memcpy(&h, static_cast<const char*>(base) + idx * 2, 2);
    uint32_t w = static_cast<uint32_t>(h) << 16;
    float f;
    std::memcpy(&f, &w, 4);
    return static_cast<double>(f);
}

inline int elem_bytes(int dtype) { return dtype == 0 ? 4 : 2; }

struct PoolView {
    const void* k_pool;
    const void* v_pool;
    int dtype;
    int64_t num_blocks;
    int block_size;
    int num_kv_heads;
    int head_dim;
};

// Gather K and V of one kv head of one sequence, logical tokens [0, len),
// into contiguous row-major [len][head_dim] fp64 arrays.  Returns false when
// the block table points outside the pool.
bool gather_head(const PoolView& P, const int32_t* table_row, int64_t len, int kvh,
                 std::vector<double>& K, std::vector<double>& V) {
    const int D = P.head_dim;
    K.assign(static_cast<size_t>(len) * D, 0.0);
    V.assign(static_cast<size_t>(len) * D, 0.0);
    for (int64_t j = 0; j < len; ++j) {
        const int64_t logical = j / P.block_size;
        const int64_t offset = j % P.block_size;
        const int64_t phys = table_row[logical];
        if (phys < 0 || phys >= P.num_blocks) return false;
        const int64_t row = ((phys * P.num_kv_heads + kvh) * P.block_size + offset) * D;
        for (int d = 0; d < D; ++d) {
            K[j * D + d] = load_elem(P.k_pool, P.dtype, row + d);
            V[j * D + d] = load_elem(P.v_pool, P.dtype, row + d);
        }
    }
    return true;
}

// softmax(scale * q.K[j]) weighted sum of V[j] over keys j in [0, n), fp64.
void attend(const double* q, const std::vector<double>& K, const std::vector<double>& V,
            int64_t n, int D, double scale, double* out) {
    std::vector<double> x(static_cast<size_t>(n));
    double m = -INFINITY;
    for (int64_t j = 0; j < n; ++j) {
        double acc = 0.0;
        for (int d = 0; d < D; ++d) acc += q[d] * K[j * D + d];
        x[j] = scale * acc;
        if (x[j] > m) m = x[j];
    }
    double den = 0.0;
    for (int d = 0; d < D; ++d) out[d] = 0.0;
    for (int64_t j = 0; j < n; ++j) {
        const double p = std::exp(x[j] - m);
        den += p;
        for (int d = 0; d < D; ++d) out[d] += p * V[j * D + d];
    }
    for (int d = 0; d < D; ++d) out[d] /= den;
}

template <class F>
void parallel_for(int64_t n_items, int nthreads, F fn) {
    if (nthreads <= 0) nthreads = static_cast<int>(std::thread::hardware_concurrency());
    if (nthreads <= 0) nthreads = 1;
    if (nthreads > n_items) nthreads = static_cast<int>(n_items > 0 ? n_items : 1);
    std::atomic<int64_t> next{0};
    auto worker = [&]() {
        for (;;) {
            const int64_t i = next.fetch_add(1);
            if (i >= n_items) break;
            fn(i);
        }
    };
    if (nthreads == 1) {
        worker();
        return;
    }
    std::vector<std::thread> pool;
    for (int t = 0; t < nthreads; ++t) pool.emplace_back(worker);
    for (auto& th : pool) th.join();
}

}  // namespace

extern "C" {

// Scatter of new K/V rows into pool slots (the "append within the current
// block" write of the Triptych page).  A slot s names block s / block_size,
// offset s % block_size.  Returns the number of rows written, -1 when a slot
// lies past the pool.  Bytes are copied verbatim.
int64_t oracle_kv_append(int dtype, int64_t num_blocks, int block_size, int num_kv_heads,
                         int head_dim, const int64_t* slot_mapping, int64_t num_tokens,
                         const void* k, const void* v, void* k_pool, void* v_pool) {
    const int64_t row_bytes = static_cast<int64_t>(head_dim) * elem_bytes(dtype);
    int64_t written = 0;
    for (int64_t t = 0; t < num_tokens; ++t) {
        const int64_t slot = slot_mapping[t];
        if (slot < 0) continue;
        if (slot >= num_blocks * block_size) return -1;
        const int64_t blk = slot / block_size;
        const int64_t off = slot % block_size;
        for (int h = 0; h < num_kv_heads; ++h) {
            const int64_t src = (t * num_kv_heads + h) * row_bytes;
            const int64_t dst = ((blk * num_kv_heads + h) * block_size + off) * row_bytes;
            std::memcpy(static_cast<char*>(k_pool) + dst, static_cast<const char*>(k) + src, row_bytes);
            std::memcpy(static_cast<char*>(v_pool) + dst, static_cast<const char*>(v) + src, row_bytes);
            ++written;
        }
    }
    return written;
}

// Copy-on-write block copy: pool[dst] = pool[src] for every (src, dst) pair,
// all kv heads and slots of the block, in pair order.
int oracle_copy_blocks(int dtype, int64_t num_blocks, int block_size, int num_kv_heads,
                       int head_dim, const int32_t* pairs, int64_t num_pairs,
                       void* k_pool, void* v_pool) {
    const int64_t block_bytes =
        static_cast<int64_t>(num_kv_heads) * block_size * head_dim * elem_bytes(dtype);
    for (int64_t i = 0; i < num_pairs; ++i) {
        const int64_t src = pairs[2 * i], dst = pairs[2 * i + 1];
        if (src < 0 || src >= num_blocks || dst < 0 || dst >= num_blocks) return -1;
        std::memmove(static_cast<char*>(k_pool) + dst * block_bytes,
                     static_cast<char*>(k_pool) + src * block_bytes, block_bytes);
        std::memmove(static_cast<char*>(v_pool) + dst * block_bytes,
                     static_cast<char*>(v_pool) + src * block_bytes, block_bytes);
    }
    return 0;
}

// Gather one (sequence, kv head) into contiguous fp64 [len][head_dim] arrays.
int oracle_gather(int dtype, const void* k_pool, const void* v_pool, int64_t num_blocks,
                  int block_size, int num_kv_heads, int head_dim, const int32_t* table_row,
                  int64_t len, int kvh, double* k_out, double* v_out) {
    PoolView P{k_pool, v_pool, dtype, num_blocks, block_size, num_kv_heads, head_dim};
    std::vector<double> K, V;
    if (!gather_head(P, table_row, len, kvh, K, V)) return -1;
    std::memcpy(k_out, K.data(), K.size() * sizeof(double));
    std::memcpy(v_out, V.data(), V.size() * sizeof(double));
    return 0;
}

// Decode: one query token per sequence.  q and out are [S][Hq][D]; sequence s
// attends its first context_lens[s] tokens.  `want` ([S*Hq], may be null)
// selects which (s, h) rows to compute; others are left untouched.
int oracle_paged_decode(int dtype, const void* q, const void* k_pool, const void* v_pool,
                        int64_t num_blocks, int block_size, int num_kv_heads, int head_dim,
                        const int32_t* block_tables, int max_blocks_per_seq,
                        const int32_t* context_lens, int num_seqs, int num_q_heads, double scale,
                        const uint8_t* want, double* out, int nthreads) {
    if (num_kv_heads <= 0 || num_q_heads % num_kv_heads != 0) return -2;
    const int G = num_q_heads / num_kv_heads;
    const int D = head_dim;
    PoolView P{k_pool, v_pool, dtype, num_blocks, block_size, num_kv_heads, head_dim};
    std::atomic<int> err{0};
    parallel_for(static_cast<int64_t>(num_seqs) * num_kv_heads, nthreads, [&](int64_t item) {
        const int s = static_cast<int>(item / num_kv_heads);
        const int kvh = static_cast<int>(item % num_kv_heads);
        bool any = false;
        for (int g = 0; g < G; ++g)
            if (!want || want[static_cast<int64_t>(s) * num_q_heads + kvh * G + g]) any = true;
        if (!any) return;
        const int64_t len = context_lens[s];
        if (len <= 0 || len > static_cast<int64_t>(max_blocks_per_seq) * block_size) {
            err = -3;
            return;
        }
        std::vector<double> K, V;
        if (!gather_head(P, block_tables + static_cast<int64_t>(s) * max_blocks_per_seq, len, kvh,
                         K, V)) {
            err = -1;
            return;
        }
        std::vector<double> qv(D);
        for (int g = 0; g < G; ++g) {
            const int h = kvh * G + g;
            const int64_t row = static_cast<int64_t>(s) * num_q_heads + h;
            if (want && !want[row]) continue;
            for (int d = 0; d < D; ++d) qv[d] = load_elem(q, dtype, row * D + d);
            attend(qv.data(), K, V, len, D, scale, out + row * D);
        }
    });
    return err.load();
}

// Prefill of new tokens over a cached prefix.  Request r has cached_lens[r]
// tokens already in the pool and new_lens[r] new tokens whose K/V are in the
// pool too (written before the call); its query rows are q[q_offsets[r] + i],
// i < new_lens[r].  Row i attends keys 0 .. cached_lens[r] + i (causal,
// inclusive).  q/out are [N][Hq][D]; `want` ([N*Hq], may be null) selects rows.
int oracle_paged_prefill(int dtype, const void* q, const void* k_pool, const void* v_pool,
                         int64_t num_blocks, int block_size, int num_kv_heads, int head_dim,
                         const int32_t* block_tables, int max_blocks_per_seq,
                         const int32_t* cached_lens, const int32_t* new_lens,
                         const int32_t* q_offsets, int num_reqs, int num_q_heads, double scale,
                         const uint8_t* want, double* out, int nthreads) {
    if (num_kv_heads <= 0 || num_q_heads % num_kv_heads != 0) return -2;
    const int G = num_q_heads / num_kv_heads;
    const int D = head_dim;
    PoolView P{k_pool, v_pool, dtype, num_blocks, block_size, num_kv_heads, head_dim};
    std::atomic<int> err{0};
    parallel_for(static_cast<int64_t>(num_reqs) * num_kv_heads, nthreads, [&](int64_t item) {
        const int r = static_cast<int>(item / num_kv_heads);
        const int kvh = static_cast<int>(item % num_kv_heads);
        const int64_t c = cached_lens[r], n = new_lens[r];
        if (c < 0 || n < 0 || c + n > static_cast<int64_t>(max_blocks_per_seq) * block_size) {
            err = -3;
            return;
        }
        if (n == 0) return;
        bool any = false;
        for (int64_t i = 0; i < n && !any; ++i)
            for (int g = 0; g < G; ++g)
                if (!want || want[(q_offsets[r] + i) * num_q_heads + kvh * G + g]) any = true;
        if (!any) return;
        std::vector<double> K, V;
        if (!gather_head(P, block_tables + static_cast<int64_t>(r) * max_blocks_per_seq, c + n,
                         kvh, K, V)) {
            err = -1;
            return;
        }
        std::vector<double> qv(D);
        for (int64_t i = 0; i < n; ++i) {
            for (int g = 0; g < G; ++g) {
                const int h = kvh * G + g;
                const int64_t row = (q_offsets[r] + i) * num_q_heads + h;
                if (want && !want[row]) continue;
                for (int d = 0; d < D; ++d) qv[d] = load_elem(q, dtype, row * D + d);
                attend(qv.data(), K, V, c + i + 1, D, scale, out + row * D);
            }
        }
    });
    return err.load();
}

// Split-KV partial (the FlashInfer "split-KV decode" bullet of the aifetchly
// SGLang guide, section "Integrating FlashInfer"): attention of one fp64 query
// over contiguous keys [lo, hi) only.  Writes the normalised partial output
// o_part[D], the partial max m (of the scaled scores) and the partial
// denominator l = sum exp(x_j - m).
int oracle_attend_partial(const double* q, const double* K, const double* V, int64_t lo,
                          int64_t hi, int D, double scale, double* o_part, double* m_out,
                          double* l_out) {
    if (hi <= lo) return -1;
    double m = -INFINITY;
    std::vector<double> x(static_cast<size_t>(hi - lo));
    for (int64_t j = lo; j < hi; ++j) {
        double acc = 0.0;
        for (int d = 0; d < D; ++d) acc += q[d] * K[j * D + d];
        x[j - lo] = scale * acc;
        if (x[j - lo] > m) m = x[j - lo];
    }
    double l = 0.0;
    for (int d = 0; d < D; ++d) o_part[d] = 0.0;
    for (int64_t j = lo; j < hi; ++j) {
        const double p = std::exp(x[j - lo] - m);
        l += p;
        for (int d = 0; d < D; ++d) o_part[d] += p * V[j * D + d];
    }
    for (int d = 0; d < D; ++d) o_part[d] /= l;
    *m_out = m;
    *l_out = l;
    return 0;
}

// Log-sum-exp merge of P partials: M = max m_p, w_p = l_p exp(m_p - M),
// out = sum_p w_p o_p / sum_p w_p.
int oracle_lse_merge(int num_parts, int D, const double* o_parts, const double* m_parts,
                     const double* l_parts, double* out) {
    if (num_parts <= 0) return -1;
    double M = -INFINITY;
    for (int p = 0; p < num_parts; ++p)
        if (m_parts[p] > M) M = m_parts[p];
    double W = 0.0;
    for (int d = 0; d < D; ++d) out[d] = 0.0;
    for (int p = 0; p < num_parts; ++p) {
        const double w = l_parts[p] * std::exp(m_parts[p] - M);
        W += w;
        for (int d = 0; d < D; ++d) out[d] += w * o_parts[static_cast<int64_t>(p) * D + d];
    }
    for (int d = 0; d < D; ++d) out[d] /= W;
    return 0;
}

}  // extern "C"
