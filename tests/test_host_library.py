"""CPU-only checks of libpkv: exported symbols, host allocator invariants, page figures.

No kernel is launched here; the library is loaded and only its host functions run.
"""
import ctypes
import json
import os
import re

import numpy as np
import pytest

ROOT = os.path.dirname(os.path.dirname(os.path.abspath(__file__)))
GOLDEN = os.path.join(ROOT, "tests", "golden", "pages_figures.json")


@pytest.fixture(scope="module")
def pkv():
    from paged_kv_cache_58_gb300 import build
    build.build()
    import paged_kv_cache_58_gb300 as m
    return m


def declared_functions():
    names = set()
    inc = os.path.join(ROOT, "include")
    for f in os.listdir(inc):
        if f.endswith(".h"):
            text = open(os.path.join(inc, f)).read()
            text = re.sub(r"/\*.*?\*/", "", text, flags=re.S)
            names.update(re.findall(r"\b(pkv_\w+)\s*\(", text))
    return sorted(names)


def test_library_exports_every_declared_function(pkv):
    names = declared_functions()
    assert len(names) >= 20
    lib = pkv.lib()
    missing = [n for n in names if not hasattr(lib, n)]
    assert not missing, missing


def test_status_strings(pkv):
    lib = pkv.lib()
    assert lib.pkv_status_string(0) == b"ok"
    assert lib.pkv_status_string(5).startswith(b"slot")
    assert lib.pkv_version() >= 100


def test_pool_bytes_and_llama70b_figure(pkv):
    g = json.load(open(GOLDEN))["kv_bytes_per_token_llama31_70b"]
    sh = g["shape_used"]
    import torch
    one_block = pkv.pool_bytes(1, sh["kv_heads"], sh["head_dim"], torch.bfloat16)
    assert one_block == 16 * sh["kv_heads"] * sh["head_dim"] * 2
    per_token = 2 * sh["layers"] * one_block / 16           # K and V, all layers
    assert per_token == 327680
    assert round(per_token / 2**20, 2) == g["mb_per_token"]
    assert abs(per_token * g["context_tokens"] / 2**30 - g["context_gb"]) < 1.0


def test_sixty_token_response_takes_four_blocks(pkv):
    g = json.load(open(GOLDEN))["sixty_token_response"]
    a = pkv.BlockAllocator(100)
    a.add_seq(1, 0)
    for _ in range(g["tokens"]):
        a.append(1, 1)
    assert a.seq_num_blocks(1) == g["blocks"]
    assert a.seq_num_blocks(1) * g["block_size"] - g["tokens"] <= g["max_idle_slots"]
    assert a.num_free == 100 - g["blocks"]


def _invariants(a, seqs):
    B = a.block_size
    held = {}
    used = set()
    for sid in seqs:
        n = a.seq_num_blocks(sid)
        L = a.seq_len(sid)
        assert 0 <= n * B - L < B or (L == 0 and n == 0), (sid, n, L)
        row = a.block_table([sid], max(n, 1))[0].tolist()
        for b in row[:n]:
            held[b] = held.get(b, 0) + 1
            used.add(b)
    for b, cnt in held.items():
        assert a.refcount(b) == cnt
    assert a.num_free + len(used) == a.num_blocks


@pytest.mark.parametrize("block_size", [16, 32])
def test_random_workload_waste_bound_and_conservation(pkv, block_size):
    g = json.load(open(GOLDEN))["waste_bound"]
    assert g["max_partial_blocks_per_sequence"] == 1
    rng = np.random.default_rng(0)
    a = pkv.BlockAllocator(4000, block_size=block_size, seed=3)
    live = []
    nxt = 0
    for step in range(600):
        op = rng.random()
        if op < 0.3 or not live:
            a.add_seq(nxt, int(rng.integers(0, 200)))
            live.append(nxt)
            nxt += 1
        elif op < 0.45:
            parent = live[int(rng.integers(len(live)))]
            a.fork(parent, nxt)
            live.append(nxt)
            nxt += 1
        elif op < 0.85:
            sid = live[int(rng.integers(len(live)))]
            a.append(sid, int(rng.integers(1, 40)))
        else:
            sid = live.pop(int(rng.integers(len(live))))
            a.free_seq(sid)
        if step % 50 == 0:
            _invariants(a, live)
    _invariants(a, live)
    for sid in live:
        a.free_seq(sid)
    assert a.num_free == 4000
    assert all(a.refcount(b) == 0 for b in range(4000))


def test_fork_shares_then_cow_on_partial_block(pkv):
    a = pkv.BlockAllocator(10)
    a.add_seq(0, 20)                        # blocks 0, 1 (block 1 holds 4 tokens)
    assert a.block_table([0], 3)[0].tolist() == [0, 1, -1]
    a.fork(0, 1)
    assert a.refcount(0) == 2 and a.refcount(1) == 2 and a.num_free == 8
    slots, cow = a.append(1, 1)
    assert cow == (1, 2)                   # private copy of the shared partial block
    assert slots == [2 * 16 + 4]
    assert a.refcount(1) == 1 and a.refcount(2) == 1 and a.refcount(0) == 2
    slots, cow = a.append(0, 1)            # parent's block 1 is private again
    assert cow is None and slots == [1 * 16 + 4]
    a.free_seq(0)
    assert a.refcount(0) == 1 and a.refcount(1) == 0
    a.free_seq(1)
    assert a.num_free == 10


def test_fork_at_block_boundary_needs_no_copy(pkv):
    a = pkv.BlockAllocator(10)
    a.add_seq(0, 32)
    a.fork(0, 1)
    slots, cow = a.append(1, 3)
    assert cow is None
    assert slots == [2 * 16, 2 * 16 + 1, 2 * 16 + 2]


def test_out_of_blocks_leaves_state_unchanged(pkv):
    import paged_kv_cache_58_gb300 as m
    a = pkv.BlockAllocator(4)
    a.add_seq(0, 50)                        # 4 blocks
    with pytest.raises(m.PkvError) as e:
        a.add_seq(1, 1)
    assert e.value.status == 6
    with pytest.raises(m.PkvError):
        a.append(0, 15)
    assert a.seq_len(0) == 50 and a.num_free == 0
    slots, _ = a.append(0, 14)              # fills the last block exactly
    assert len(slots) == 14 and a.seq_len(0) == 64


def test_seeded_free_order(pkv):
    a0 = pkv.BlockAllocator(64)
    a0.add_seq(0, 64 * 16)
    assert a0.block_table([0], 64)[0].tolist() == list(range(64))
    a1 = pkv.BlockAllocator(64, seed=7)
    a1.add_seq(0, 64 * 16)
    t1 = a1.block_table([0], 64)[0].tolist()
    assert sorted(t1) == list(range(64)) and t1 != list(range(64))
    a2 = pkv.BlockAllocator(64, seed=7)
    a2.add_seq(0, 64 * 16)
    assert a2.block_table([0], 64)[0].tolist() == t1


def test_unknown_ids_and_small_tables(pkv):
    import paged_kv_cache_58_gb300 as m
    a = pkv.BlockAllocator(8)
    a.add_seq(0, 40)
    with pytest.raises(m.PkvError):
        a.add_seq(0, 1)
    with pytest.raises(m.PkvError):
        a.fork(5, 6)
    with pytest.raises(m.PkvError):
        a.block_table([0], 2)
    with pytest.raises(m.PkvError):
        a.free_seq(9)


def test_decode_workspace_and_partition_policy(pkv):
    # 8B-shaped batch: 64 sequences up to 4096 tokens -> 1024-token partitions
    assert pkv.auto_partition(64, 32, 4096) == 64
    ws = pkv.decode_workspace_bytes(64, 32, 128, 4096)
    assert ws == 64 * 32 * 4 * (128 + 2) * 4
    # 70B-shaped batch: 131072 tokens -> at most 64 partitions
    pb = pkv.auto_partition(16, 64, 131072)
    assert pb == 128 and -(-8192 // pb) == 64
    # a single short sequence needs no workspace
    assert pkv.decode_workspace_bytes(1, 8, 128, 64) == 0
    # 32-token blocks: the same 1024-token partitions (32 blocks), the same workspace
    assert pkv.auto_partition(64, 32, 4096, block_size=32) == 32
    assert pkv.decode_workspace_bytes(64, 32, 128, 4096, block_size=32) == ws
    assert pkv.auto_partition(16, 64, 131072, block_size=32) == 64
    # other block sizes are not supported
    assert pkv.auto_partition(64, 32, 4096, block_size=8) == 0


def test_decode_step_layout(pkv):
    """Packed host layout of a decode step: 256-byte aligned arrays in order, sizes from
    the shapes; the staging adds the output and the split-KV workspace."""
    d = pkv.PoolDesc(32768, 16, 8, 128, 1)
    lay = pkv.StepLayout()
    assert pkv.lib().pkv_decode_step_layout(ctypes.byref(d), 64, 32, 256, ctypes.byref(lay)) == 0
    offs = [lay.q, lay.k_new, lay.v_new, lay.block_tables, lay.context_lens, lay.bytes]
    assert all(o % 256 == 0 for o in offs) and offs == sorted(offs)
    assert lay.q == 0 and lay.k_new >= 64 * 32 * 128 * 2
    assert lay.v_new - lay.k_new >= 64 * 8 * 128 * 2
    assert lay.context_lens - lay.block_tables >= 64 * 256 * 4
    assert lay.bytes - lay.context_lens >= 64 * 4
    staging = pkv.lib().pkv_paged_decode_append_host_staging_bytes(ctypes.byref(d), 64, 32,
                                                                   256, 4096, 0)
    assert staging == lay.bytes + 64 * 32 * 128 * 2 + pkv.decode_workspace_bytes(64, 32, 128,
                                                                                 4096)
    assert pkv.lib().pkv_decode_step_layout(ctypes.byref(d), -1, 32, 256,
                                            ctypes.byref(lay)) == 1


def test_prefill_step_layout(pkv):
    """Packed host layout of a prefill step: the copied part (q, tables, lengths,
    offsets) first, then the new rows and slots, 256-byte aligned; the staging adds the
    output."""
    d = pkv.PoolDesc(32768, 16, 8, 128, 1)
    lay = pkv.PrefillLayout()
    assert pkv.lib().pkv_prefill_step_layout(ctypes.byref(d), 16, 8192, 32, 513,
                                             ctypes.byref(lay)) == 0
    offs = [lay.q, lay.block_tables, lay.cached_lens, lay.new_lens, lay.q_offsets,
            lay.copied_bytes, lay.v_new, lay.slot_mapping, lay.bytes]
    assert all(o % 256 == 0 for o in offs) and offs == sorted(offs)
    assert lay.q == 0 and lay.block_tables >= 8192 * 32 * 128 * 2
    assert lay.cached_lens - lay.block_tables >= 16 * 513 * 4
    assert lay.copied_bytes - lay.q_offsets >= 17 * 4 and lay.k_new == lay.copied_bytes
    assert lay.v_new - lay.k_new >= 8192 * 8 * 128 * 2
    assert lay.bytes - lay.slot_mapping >= 8192 * 8
    staging = pkv.lib().pkv_paged_prefill_append_host_staging_bytes(ctypes.byref(d), 16, 8192,
                                                                    32, 513)
    assert staging == lay.bytes + 8192 * 32 * 128 * 2
    assert pkv.lib().pkv_prefill_step_layout(ctypes.byref(d), -1, 8192, 32, 513,
                                             ctypes.byref(lay)) == 1


def test_auto_partition_is_a_multiple_of_four_chunks():
    """The library's split-KV partition size, in 16-token chunks, is a multiple of 4 (one
    chunk per warp per step, and whole 32-token blocks) and at least 8, over a grid of
    batch shapes; in 32-token blocks it is half that."""
    import itertools
    import paged_kv_cache_58_gb300 as pkv
    for s, hq, ctx in itertools.product([1, 2, 3, 7, 16, 64, 256, 4096], [1, 8, 32, 64],
                                        [1, 17, 1000, 4096, 70000, 73728, 131072, 1 << 20]):
        pc = pkv.auto_partition(s, hq, ctx, block_size=16)
        assert pc % 4 == 0 and pc >= 8, (s, hq, ctx, pc)
        assert pkv.auto_partition(s, hq, ctx, block_size=32) * 2 == pc
