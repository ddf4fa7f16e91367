"""CPU tests of the prefix-reuse indexes over the host allocator (no GPU).

Chained block hashes and salting follow aitalk.it "Two Layers, Not Two Rivals" and
"Beyond the Two Techniques"; the radix tree, its node splitting, locking and LRU
leaf eviction follow aitalk.it "RadixAttention: A Tree That Does Not Forget",
khotyn.com "RadixAttention" and the aifetchly SGLang guide.  Golden figures are
in tests/golden/pages_figures.json with their sources.
"""
import json
import os
import random

import pytest

ROOT = os.path.dirname(os.path.dirname(os.path.abspath(__file__)))
GOLDEN = json.load(open(os.path.join(ROOT, "tests", "golden", "pages_figures.json")))
B = 16


@pytest.fixture(scope="module")
def pkv():
    from paged_kv_cache_58_gb300 import build
    build.build()
    import paged_kv_cache_58_gb300 as m
    return m


def new_seq(alloc, sid, n):
    alloc.add_seq(sid, 0)
    alloc.append(sid, n)


def refcount_total(alloc):
    return sum(alloc.refcount(b) for b in range(alloc.num_blocks))


# ---------------------------------------------------------------- block hashes
def test_hash_chain_equal_prefixes_equal_chains(pkv):
    a = list(range(16))
    h1 = pkv.block_hash(0, 0, a)
    assert h1 == pkv.block_hash(0, 0, a)
    assert pkv.block_hash(h1, 0, list(range(16, 32))) == pkv.block_hash(h1, 0,
                                                                          list(range(16, 32)))
    # a change in the parent (or the salt, or the tokens) changes the child hash
    assert pkv.block_hash(h1 ^ 1, 0, list(range(16, 32))) != pkv.block_hash(h1, 0,
                                                                              list(range(16, 32)))
    assert pkv.block_hash(0, 7, a) != h1
    b = a.copy()
    b[5] += 1
    assert pkv.block_hash(0, 0, b) != h1


def test_block_cache_reuses_full_blocks_only(pkv):
    g = GOLDEN["prefix_hit_1900_of_2000"]
    alloc = pkv.BlockAllocator(400)
    pc = pkv.PrefixCache(alloc)
    prompt = list(range(1000, 1000 + g["prompt_tokens"]))
    new_seq(alloc, 1, g["cached_tokens"])
    assert pc.insert(1, prompt[:g["cached_tokens"]]) == g["cached_tokens"] // B
    blocks = pc.match(prompt)
    assert len(blocks) * B == g["prompt_tokens"] - g["to_prefill_block_hash"]
    assert blocks == alloc.block_table([1], 200)[0].tolist()[:len(blocks)]
    # the new request shares those blocks and allocates the rest
    alloc.add_seq_shared(2, blocks, len(blocks) * B)
    assert all(alloc.refcount(b) == 3 for b in blocks)   # seq 1, seq 2, cache
    pc.close()
    alloc.close()


def test_salt_separates_tenants(pkv):
    alloc = pkv.BlockAllocator(64)
    pc = pkv.PrefixCache(alloc)
    prompt = list(range(64))
    new_seq(alloc, 1, 64)
    pc.insert(1, prompt, salt=111)
    assert len(pc.match(prompt, salt=111)) == 4
    assert pc.match(prompt, salt=222) == []
    assert pc.match(prompt) == []


def test_block_cache_eviction_keeps_blocks_in_use(pkv):
    alloc = pkv.BlockAllocator(10)
    pc = pkv.PrefixCache(alloc)
    new_seq(alloc, 1, 64)                       # 4 blocks
    pc.insert(1, list(range(64)))
    new_seq(alloc, 2, 32)                       # 2 blocks
    pc.insert(2, list(range(500, 532)))
    alloc.free_seq(2)                           # its blocks now live only in the cache
    assert alloc.num_free == 4
    assert pc.evict(6) == 2                     # drops seq 2's two cached blocks
    assert alloc.num_free == 6
    assert pc.evict(10) == 0                    # seq 1 still uses its blocks
    assert len(pc) == 4
    alloc.free_seq(1)
    assert pc.evict(10) == 4 and alloc.num_free == 10


# ---------------------------------------------------------------- radix tree
def test_radix_matches_1900_of_2000(pkv):
    g = GOLDEN["prefix_hit_1900_of_2000"]
    alloc = pkv.BlockAllocator(400)
    rt = pkv.RadixTree(alloc)
    prompt = list(range(7, 7 + g["prompt_tokens"]))
    new_seq(alloc, 1, g["cached_tokens"])
    rt.insert(1, prompt[:g["cached_tokens"]])
    m, blocks = rt.match(prompt)
    assert m == g["cached_tokens"]
    assert g["prompt_tokens"] - m == g["to_prefill_radix"]
    table = alloc.block_table([1], 200)[0].tolist()
    assert blocks == table[:len(blocks)]
    # share the matched blocks (the last one partial) and append the rest: the shared
    # partial block is copied first
    alloc.add_seq_shared(2, blocks, m)
    slots, cow = alloc.append(2, g["prompt_tokens"] - m)
    assert cow is not None and cow[0] == blocks[-1]
    assert alloc.seq_len(2) == g["prompt_tokens"]


def test_radix_multi_turn_agent_prefills(pkv):
    g = GOLDEN["multi_turn_agent_prefills"]
    alloc = pkv.BlockAllocator(2000)
    rt = pkv.RadixTree(alloc)
    rng = random.Random(0)
    conversation = [rng.randrange(32000) for _ in range(g["turn_prompt_tokens"][-1])]
    computed = []
    for turn, n in enumerate(g["turn_prompt_tokens"]):
        prompt = conversation[:n]
        m, blocks = rt.match(prompt)
        computed.append(n - m)
        alloc.add_seq_shared(turn, blocks, m)
        alloc.append(turn, n - m)
        rt.insert(turn, prompt)
        alloc.free_seq(turn)             # the tree keeps the blocks
    assert computed == g["computed_with_prefix_reuse"]
    assert sum(computed) == g["turn_prompt_tokens"][-1]


def test_radix_split_and_branch(pkv):
    """Three users share a system prompt; the tree stores it once and branches."""
    alloc = pkv.BlockAllocator(200)
    rt = pkv.RadixTree(alloc)
    system = list(range(100))
    questions = [list(range(1000 * (u + 1), 1000 * (u + 1) + 37)) for u in range(3)]
    for u, qtok in enumerate(questions):
        prompt = system + qtok
        m, blocks = rt.match(prompt)
        assert m == (0 if u == 0 else len(system))
        alloc.add_seq_shared(u, blocks, m)
        alloc.append(u, len(prompt) - m)
        rt.insert(u, prompt)
    assert rt.num_nodes == 4                          # shared prefix + 3 leaves
    assert rt.cached_tokens == len(system) + 3 * 37
    for u, qtok in enumerate(questions):              # each branch maps to its own blocks
        m, blocks = rt.match(system + qtok)
        assert m == len(system) + 37
        assert blocks == alloc.block_table([u], 20)[0].tolist()[:len(blocks)]


def test_radix_lru_eviction_protects_locked_and_shared(pkv):
    """The walk-through of the RadixAttention figure: two sessions share a system
    prompt; under memory pressure the least recently used, unlocked leaf goes first
    and the shared prefix stays."""
    alloc = pkv.BlockAllocator(40)
    rt = pkv.RadixTree(alloc)
    system = list(range(64))                          # 4 blocks
    s1 = system + list(range(500, 500 + 96))          # + 6 blocks
    s2 = system + list(range(900, 900 + 96))
    for sid, toks in ((1, s1), (2, s2)):
        m, blocks = rt.match(toks)
        alloc.add_seq_shared(sid, blocks, m)
        alloc.append(sid, len(toks) - m)
        rt.insert(sid, toks)
    rt.lock(s2, +1)                                   # session 2 is still running
    alloc.free_seq(1)
    alloc.free_seq(2)
    free0 = alloc.num_free
    assert rt.evict(free0 + 1) == 1                   # session 1's leaf (unlocked) goes
    assert rt.match(s1)[0] == len(system)             # its private part is gone ...
    assert rt.match(s2)[0] == len(s2)                 # ... session 2 and the prefix stay
    assert rt.evict(alloc.num_blocks) == 0            # all that is left is locked
    rt.lock(s2, -1)
    assert rt.evict(alloc.num_blocks) >= 1
    assert rt.num_nodes == 0 and alloc.num_free == alloc.num_blocks


def test_radix_random_workload_refcounts(pkv):
    """Random prompts over a 5-token vocabulary (many shared prefixes, splits and
    merges).  A content model records which token every slot holds (writes at append,
    whole-block copies at copy-on-write); every match must return blocks that hold the
    matched prompt, and references must balance at the end."""
    rng = random.Random(5)
    alloc = pkv.BlockAllocator(3000, seed=9)
    rt = pkv.RadixTree(alloc)
    vocab = 5
    content = {}
    live = []

    def check_match(prompt):
        m, blocks = rt.match(prompt)
        for p in range(m):
            assert content[blocks[p // B]][p % B] == prompt[p], (p, m)
        return m, blocks

    for sid in range(200):
        n = rng.randrange(1, 120)
        prompt = [rng.randrange(vocab) for _ in range(n)]
        m, blocks = check_match(prompt)
        assert 0 <= m <= n
        alloc.add_seq_shared(sid, blocks, m)
        slots, cow = alloc.append(sid, n - m)
        if cow is not None:
            content[cow[1]] = list(content[cow[0]])
        for i, slot in enumerate(slots):
            content.setdefault(slot // B, [None] * B)[slot % B] = prompt[m + i]
        rt.insert(sid, prompt)
        assert check_match(prompt)[0] == n
        live.append(sid)
        if rng.random() < 0.4:
            alloc.free_seq(live.pop(rng.randrange(len(live))))
        if rng.random() < 0.2:
            rt.evict(rng.randrange(alloc.num_blocks))
        for _ in range(3):       # probe random prompts against the tree
            check_match([rng.randrange(vocab) for _ in range(rng.randrange(1, 130))])
        assert alloc.num_free + sum(1 for b in range(alloc.num_blocks)
                                    if alloc.refcount(b) > 0) == alloc.num_blocks
    for sid in live:
        alloc.free_seq(sid)
    rt.evict(alloc.num_blocks)
    assert alloc.num_free == alloc.num_blocks and refcount_total(alloc) == 0
