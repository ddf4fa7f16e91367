// Prefix reuse over the paged block pool: two index structures that point at
// blocks owned by the host allocator (aitalk.it "Two Layers, Not Two Rivals": the
// prefix index "simply points to blocks that are themselves managed by the paged
// allocator").
//
// 1. Chained block hashes (aitalk.it, same section; khotyn.com "PagedAttention"):
//    every full block gets a hash of its parent block's hash, its own tokens and
//    extra metadata, so equal prefixes produce equal hash chains.  A tenant salt
//    mixed into the hash keeps identical prompts of different tenants apart
//    (aitalk.it "Beyond the Two Techniques": cache salting).  Matching is at block
//    granularity.  Entries keep the tokens they stand for and a match compares
//    them, so a hash collision cannot share the wrong block.
//
// 2. A radix tree (compressed trie) of token sequences (aitalk.it "RadixAttention:
//    A Tree That Does Not Forget"; khotyn.com "RadixAttention"; aifetchly SGLang
//    guide, "Radix Tree Topology", "Dynamic Node Splitting", "LRU Leaf Eviction"):
//    edges carry token runs, nodes carry the physical blocks that hold those
//    positions; lookup returns the longest common prefix at token granularity;
//    insertion splits an edge where a new sequence diverges; nodes locked by active
//    requests are never evicted, and eviction removes least recently used unlocked
//    leaves until enough blocks are free, merging a parent left with one child.
//
// Both structures hold one allocator reference per block they point at, so cached
// blocks survive the sequences that produced them and return to the free list only
// when the index lets them go and no sequence uses them.
#include <algorithm>
#include <cstdint>
#include <list>
#include <memory>
#include <new>
#include <unordered_map>
#include <vector>

#include "../../include/pkv.h"
#include "alloc_internal.h"

namespace {

uint64_t mix64(uint64_t z) {  // splitmix64 finaliser
    z = (z ^ (z >> 30)) * 0xBF58476D1CE4E5B9ull;
    z = (z ^ (z >> 27)) * 0x94D049BB133111EBull;
    return z ^ (z >> 31);
}

}  // namespace

// ====================================================================== hash chain
struct pkv_pcache {
    struct Entry {
        int32_t block;
        uint64_t parent;
        uint64_t salt;
        std::vector<int32_t> tokens;
        std::list<uint64_t>::iterator lru;  // position in the LRU list (front = oldest)
    };
    pkv_alloc* alloc;
    std::unordered_map<uint64_t, Entry> map;
    std::list<uint64_t> lru;
};

extern "C" {

uint64_t pkv_block_hash(uint64_t parent_hash, uint64_t salt, const int32_t* tokens, int n,
                        uint64_t extra) {
    uint64_t h = mix64(parent_hash + 0x9E3779B97F4A7C15ull);
    h = mix64(h ^ salt);
    h = mix64(h ^ extra);
    for (int i = 0; i < n; ++i)
        h = mix64(h ^ (static_cast<uint64_t>(static_cast<uint32_t>(tokens[i])) |
                       (static_cast<uint64_t>(i) << 32)));
    return h;
}

pkv_pcache* pkv_pcache_create(pkv_alloc* a) {
    if (!a) return nullptr;
    pkv_pcache* pc = new (std::nothrow) pkv_pcache();
    if (pc) pc->alloc = a;
    return pc;
}

void pkv_pcache_destroy(pkv_pcache* pc) {
    if (!pc) return;
    for (auto& kv : pc->map) pc->alloc->release(kv.second.block);
    delete pc;
}

int pkv_pcache_match(pkv_pcache* pc, const int32_t* tokens, int64_t n, uint64_t salt,
                     int32_t* blocks_out, int max_blocks) {
    if (!pc || n < 0 || (n > 0 && !tokens) || max_blocks < 0 || (max_blocks > 0 && !blocks_out))
        return -1;
    const int B = pc->alloc->block_size;
    uint64_t parent = 0;
    int count = 0;
    for (int64_t start = 0; start + B <= n && count < max_blocks; start += B) {
        const uint64_t h = pkv_block_hash(parent, salt, tokens + start, B, 0);
        auto it = pc->map.find(h);
        if (it == pc->map.end()) break;
        const auto& e = it->second;
        if (e.parent != parent || e.salt != salt ||
            !std::equal(e.tokens.begin(), e.tokens.end(), tokens + start))
            break;
        pc->lru.splice(pc->lru.end(), pc->lru, e.lru);  // most recently used
        blocks_out[count++] = e.block;
        parent = h;
    }
    return count;
}

int pkv_pcache_insert(pkv_pcache* pc, int64_t seq_id, const int32_t* tokens, int64_t n,
                      uint64_t salt) {
    if (!pc || n < 0 || (n > 0 && !tokens)) return -1;
    auto sit = pc->alloc->seqs.find(seq_id);
    if (sit == pc->alloc->seqs.end() || sit->second.num_tokens < n) return -1;
    const auto& blocks = sit->second.blocks;
    const int B = pc->alloc->block_size;
    uint64_t parent = 0;
    int added = 0;
    for (int64_t start = 0, i = 0; start + B <= n; start += B, ++i) {
        const uint64_t h = pkv_block_hash(parent, salt, tokens + start, B, 0);
        auto it = pc->map.find(h);
        if (it == pc->map.end()) {
            pkv_pcache::Entry e;
            e.block = blocks[static_cast<size_t>(i)];
            e.parent = parent;
            e.salt = salt;
            e.tokens.assign(tokens + start, tokens + start + B);
            e.lru = pc->lru.insert(pc->lru.end(), h);
            pc->alloc->retain(e.block);
            pc->map.emplace(h, std::move(e));
            ++added;
        } else {
            pc->lru.splice(pc->lru.end(), pc->lru, it->second.lru);
        }
        parent = h;
    }
    return added;
}

int64_t pkv_pcache_evict(pkv_pcache* pc, int64_t min_free) {
    if (!pc) return -1;
    pkv_alloc* a = pc->alloc;
    int64_t freed = 0;
    for (auto it = pc->lru.begin();
         it != pc->lru.end() && static_cast<int64_t>(a->free_list.size()) < min_free;) {
        auto e = pc->map.find(*it);
        if (a->refcount[e->second.block] == 1) {  // only the cache holds it
            a->release(e->second.block);
            pc->map.erase(e);
            it = pc->lru.erase(it);
            ++freed;
        } else {
            ++it;
        }
    }
    return freed;
}

int64_t pkv_pcache_size(const pkv_pcache* pc) {
    return pc ? static_cast<int64_t>(pc->map.size()) : -1;
}

}  // extern "C"

// ====================================================================== radix tree
struct pkv_radix {
    struct Node {
        Node* parent = nullptr;
        std::vector<int32_t> tokens;          // edge label: positions [start, start + size)
        int64_t start = 0;                    // absolute position of tokens[0]
        std::vector<int32_t> blocks;          // blocks of positions [start, end), first one
                                              // is block index start / B
        std::unordered_map<int32_t, std::unique_ptr<Node>> children;  // by first token
        int64_t lock = 0;                     // active requests using this node
        uint64_t last_use = 0;
        int64_t end() const { return start + static_cast<int64_t>(tokens.size()); }
    };
    pkv_alloc* alloc;
    Node root;
    uint64_t clock = 0;
    int64_t nodes = 0;
    int64_t cached_tokens = 0;
};

namespace {

using RNode = pkv_radix::Node;

int64_t block_index(int64_t pos, int B) { return pos / B; }

// Blocks of positions [start, end) taken from a sequence's block table, one
// reference each.
void take_blocks(pkv_alloc* a, const std::vector<int32_t>& table, int64_t start, int64_t end,
                 std::vector<int32_t>& out) {
    const int B = a->block_size;
    out.clear();
    for (int64_t b = block_index(start, B); b <= block_index(end - 1, B); ++b) {
        const int32_t id = table[static_cast<size_t>(b)];
        a->retain(id);
        out.push_back(id);
    }
}

void release_blocks(pkv_alloc* a, std::vector<int32_t>& blocks) {
    for (int32_t b : blocks) a->release(b);
    blocks.clear();
}

// Split `n` so that it keeps its first `k` tokens; the rest moves to a new child
// that inherits n's children.  Blocks are divided by position; a block straddling
// the cut is referenced by both halves (one extra reference).
RNode* split(pkv_radix* t, RNode* n, int64_t k) {
    const int B = t->alloc->block_size;
    auto tail = std::make_unique<RNode>();
    tail->parent = n;
    tail->start = n->start + k;
    tail->tokens.assign(n->tokens.begin() + k, n->tokens.end());
    tail->children = std::move(n->children);
    for (auto& kv : tail->children) kv.second->parent = tail.get();
    tail->lock = n->lock;
    tail->last_use = n->last_use;
    const int64_t first_blk = block_index(n->start, B);
    const int64_t cut_first = block_index(tail->start, B) - first_blk;   // tail's first block
    const int64_t head_last = block_index(tail->start - 1, B) - first_blk;  // head's last block
    tail->blocks.assign(n->blocks.begin() + cut_first, n->blocks.end());
    if (head_last == cut_first) t->alloc->retain(n->blocks[static_cast<size_t>(cut_first)]);
    n->blocks.resize(static_cast<size_t>(head_last + 1));
    n->tokens.resize(static_cast<size_t>(k));
    n->children.clear();
    RNode* raw = tail.get();
    n->children.emplace(raw->tokens[0], std::move(tail));
    ++t->nodes;
    return raw;
}

// Merge `n` with its only child (edge compression after an eviction).
void merge_with_child(pkv_radix* t, RNode* n) {
    const int B = t->alloc->block_size;
    auto it = n->children.begin();
    std::unique_ptr<RNode> child = std::move(it->second);
    n->children.clear();
    const int64_t last_blk = block_index(n->end() - 1, B);
    const int64_t child_first = block_index(child->start, B);
    if (last_blk == child_first) {  // shared boundary block: keep the child's copy
        t->alloc->release(n->blocks.back());
        n->blocks.pop_back();
    }
    n->blocks.insert(n->blocks.end(), child->blocks.begin(), child->blocks.end());
    n->tokens.insert(n->tokens.end(), child->tokens.begin(), child->tokens.end());
    n->children = std::move(child->children);
    for (auto& kv : n->children) kv.second->parent = n;
    n->last_use = std::max(n->last_use, child->last_use);
    --t->nodes;
}

}  // namespace

extern "C" {

pkv_radix* pkv_radix_create(pkv_alloc* a) {
    if (!a) return nullptr;
    pkv_radix* t = new (std::nothrow) pkv_radix();
    if (t) t->alloc = a;
    return t;
}

static void radix_free(pkv_alloc* a, RNode* n) {
    for (auto& kv : n->children) radix_free(a, kv.second.get());
    release_blocks(a, n->blocks);
}

void pkv_radix_destroy(pkv_radix* t) {
    if (!t) return;
    radix_free(t->alloc, &t->root);
    delete t;
}

int64_t pkv_radix_match(pkv_radix* t, const int32_t* tokens, int64_t n, int32_t* blocks_out,
                        int max_blocks) {
    if (!t || n < 0 || (n > 0 && !tokens) || max_blocks < 0 || (max_blocks > 0 && !blocks_out))
        return -1;
    const int B = t->alloc->block_size;
    const uint64_t now = ++t->clock;
    RNode* node = &t->root;
    int64_t m = 0;
    while (m < n) {
        auto it = node->children.find(tokens[m]);
        if (it == node->children.end()) break;
        RNode* c = it->second.get();
        int64_t k = 0;
        while (k < static_cast<int64_t>(c->tokens.size()) && m + k < n && c->tokens[k] == tokens[m + k])
            ++k;
        c->last_use = now;
        // blocks of the matched positions [m, m + k) of this node; deeper nodes
        // overwrite a shared boundary block index with their own block
        const int64_t first = block_index(c->start, B);
        for (int64_t p = block_index(m, B); p <= block_index(m + k - 1, B); ++p)
            if (p < max_blocks) blocks_out[p] = c->blocks[static_cast<size_t>(p - first)];
        m += k;
        if (k < static_cast<int64_t>(c->tokens.size())) break;
        node = c;
    }
    return m;
}

pkv_status pkv_radix_insert(pkv_radix* t, int64_t seq_id, const int32_t* tokens, int64_t n) {
    if (!t || n < 0 || (n > 0 && !tokens)) return PKV_ERR_INVALID;
    auto sit = t->alloc->seqs.find(seq_id);
    if (sit == t->alloc->seqs.end() || sit->second.num_tokens < n) return PKV_ERR_NOT_FOUND;
    const auto& table = sit->second.blocks;
    const uint64_t now = ++t->clock;
    RNode* node = &t->root;
    int64_t m = 0;
    while (m < n) {
        auto it = node->children.find(tokens[m]);
        if (it == node->children.end()) {
            auto leaf = std::make_unique<RNode>();
            leaf->parent = node;
            leaf->start = m;
            leaf->tokens.assign(tokens + m, tokens + n);
            leaf->last_use = now;
            take_blocks(t->alloc, table, m, n, leaf->blocks);
            t->cached_tokens += n - m;
            node->children.emplace(tokens[m], std::move(leaf));
            ++t->nodes;
            return PKV_OK;
        }
        RNode* c = it->second.get();
        int64_t k = 0;
        while (k < static_cast<int64_t>(c->tokens.size()) && m + k < n && c->tokens[k] == tokens[m + k])
            ++k;
        c->last_use = now;
        if (k < static_cast<int64_t>(c->tokens.size())) split(t, c, k);
        m += k;
        node = c;
    }
    return PKV_OK;
}

pkv_status pkv_radix_lock(pkv_radix* t, const int32_t* tokens, int64_t n, int delta) {
    if (!t || n < 0 || (n > 0 && !tokens) || (delta != 1 && delta != -1)) return PKV_ERR_INVALID;
    RNode* node = &t->root;
    int64_t m = 0;
    std::vector<RNode*> path;
    while (m < n) {
        auto it = node->children.find(tokens[m]);
        if (it == node->children.end()) break;
        RNode* c = it->second.get();
        const int64_t len = static_cast<int64_t>(c->tokens.size());
        if (m + len > n || !std::equal(c->tokens.begin(), c->tokens.end(), tokens + m)) break;
        path.push_back(c);
        m += len;
        node = c;
    }
    if (m != n) return PKV_ERR_NOT_FOUND;  // lock whole nodes only: insert first
    for (RNode* c : path) {
        if (delta < 0 && c->lock == 0) return PKV_ERR_INVALID;
    }
    for (RNode* c : path) c->lock += delta;
    return PKV_OK;
}

static void collect_leaves(RNode* n, std::vector<RNode*>& out) {
    if (n->children.empty()) {
        out.push_back(n);
        return;
    }
    for (auto& kv : n->children) collect_leaves(kv.second.get(), out);
}

int64_t pkv_radix_evict(pkv_radix* t, int64_t min_free) {
    if (!t) return -1;
    pkv_alloc* a = t->alloc;
    int64_t evicted = 0;
    while (static_cast<int64_t>(a->free_list.size()) < min_free) {
        std::vector<RNode*> leaves;
        for (auto& kv : t->root.children) collect_leaves(kv.second.get(), leaves);
        RNode* victim = nullptr;
        for (RNode* l : leaves)
            if (l->lock == 0 && (!victim || l->last_use < victim->last_use)) victim = l;
        if (!victim) break;  // everything left is in use
        RNode* parent = victim->parent;
        t->cached_tokens -= static_cast<int64_t>(victim->tokens.size());
        release_blocks(a, victim->blocks);
        parent->children.erase(victim->tokens[0]);
        --t->nodes;
        ++evicted;
        if (parent != &t->root && parent->children.size() == 1 && parent->lock == 0 &&
            parent->children.begin()->second->lock == 0)
            merge_with_child(t, parent);
    }
    return evicted;
}

int64_t pkv_radix_num_nodes(const pkv_radix* t) { return t ? t->nodes : -1; }
int64_t pkv_radix_cached_tokens(const pkv_radix* t) { return t ? t->cached_tokens : -1; }

}  // extern "C"
