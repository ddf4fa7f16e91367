"""GPU parity of kv_append + paged_decode against the fp64 oracle (through the C ABI)."""
import dataclasses

import numpy as np
import pytest
import torch

import synth
from tests.helpers import check_attention, oracle_decode_case, pool_equal

pytestmark = pytest.mark.gpu


@pytest.fixture(scope="module")
def pkv():
    if not torch.cuda.is_available():
        pytest.skip("no CUDA device")
    import paged_kv_cache_58_gb300 as m
    from paged_kv_cache_58_gb300 import build
    build.build()
    return m


@pytest.fixture(params=["tc", "simt"])
def kernel(request, monkeypatch):
    """bf16 decode kernel under test: tensor-core (default) or CUDA-core."""
    if request.param == "simt":
        monkeypatch.setenv("PKV_DECODE_KERNEL", "simt")
    else:
        monkeypatch.delenv("PKV_DECODE_KERNEL", raising=False)
    return request.param


def run_decode(pkv, case, partition_blocks=0):
    pkv.kv_append(case.k_pool, case.v_pool, case.slot_mapping, case.k_new, case.v_new)
    out = pkv.paged_decode(case.q, case.k_pool, case.v_pool, case.block_tables,
                           case.context_lens, case.scale, max_context=case.max_context,
                           partition_blocks=partition_blocks)
    torch.cuda.synchronize()
    assert pkv.read_device_status() == 0
    return out


def small(wl_key, **over):
    return dataclasses.replace(synth.WORKLOADS[wl_key], **over)


def test_tiny_published_config(pkv, oracle_mod):
    case = synth.build_case("tiny", "cuda")
    ref, kp, vp = oracle_decode_case(oracle_mod, case)
    out = run_decode(pkv, case)
    assert pool_equal(case.k_pool, kp) and pool_equal(case.v_pool, vp)
    check_attention(out, ref)


@pytest.mark.parametrize("pb", [1, 2, 3])
def test_tiny_split_partitions(pkv, oracle_mod, pb):
    case = synth.build_case("tiny", "cuda")
    ref, _, _ = oracle_decode_case(oracle_mod, case)
    check_attention(run_decode(pkv, case, partition_blocks=pb), ref)


EDGE_LENS = [1, 2, 15, 16, 17, 31, 32, 33, 63, 64, 65, 127, 128, 129, 500, 1000]


@pytest.mark.parametrize("hq,hkv,d", [(32, 8, 128), (64, 8, 128), (16, 8, 128), (8, 8, 128),
                                      (32, 8, 64), (8, 1, 64)])
@pytest.mark.parametrize("pb", [0, 1, 5])
def test_edge_lengths_bf16(pkv, oracle_mod, hq, hkv, d, pb, kernel):
    wl = small("8b", num_q_heads=hq, num_kv_heads=hkv, head_dim=d, num_blocks=512)
    case = synth.build_case(wl, "cuda", lengths=EDGE_LENS, seed=hq * 7 + d + pb)
    ref, kp, vp = oracle_decode_case(oracle_mod, case)
    out = run_decode(pkv, case, partition_blocks=pb)
    assert pool_equal(case.k_pool, kp) and pool_equal(case.v_pool, vp)
    check_attention(out, ref)


@pytest.mark.parametrize("hq,hkv", [(4, 4), (8, 2), (32, 4)])
def test_fp32_shapes(pkv, oracle_mod, hq, hkv):
    wl = small("tiny", num_q_heads=hq, num_kv_heads=hkv, head_dim=128, num_blocks=256)
    case = synth.build_case(wl, "cuda", lengths=[1, 16, 17, 200, 333], seed=hq + hkv)
    ref, _, _ = oracle_decode_case(oracle_mod, case)
    check_attention(run_decode(pkv, case, partition_blocks=2), ref)


def test_llama3_8b_decode_full(pkv, oracle_mod, kernel):
    """Published 8B-shaped batch at full size, every output vs the oracle."""
    case = synth.build_case("8b", "cuda")
    ref, kp, vp = oracle_decode_case(oracle_mod, case)
    out = run_decode(pkv, case)
    assert pool_equal(case.k_pool, kp) and pool_equal(case.v_pool, vp)
    check_attention(out, ref)


def test_llama31_70b_long_decode_full(pkv, published_decode_ref, kernel):
    """Published 70B long-context batch at full size (16 sequences of U[16384, 131072]
    tokens, 64 / 8 heads, split-KV partitions): every output against the oracle."""
    ref = published_decode_ref("70b")
    case = synth.build_case("70b", "cuda")
    out = run_decode(pkv, case)
    assert ref.size == 16 * 64 * 128
    check_attention(out, ref)


def test_shared_prefix_decode_full(pkv, published_decode_ref, kernel):
    """Published shared-prefix batch: 256 sequences on the same 256 prefix blocks; every
    output against the oracle."""
    ref = published_decode_ref("shared")
    case = synth.build_case("shared", "cuda")
    bt = case.block_tables.cpu()
    assert (bt[:, :256] == bt[0, :256]).all()
    out = run_decode(pkv, case)
    assert ref.size == 256 * 32 * 128
    check_attention(out, ref)


def test_shared_prefix_equals_copied_prefix_on_gpu(pkv, kernel):
    """Same bits whether the prefix blocks are shared or copied per sequence."""
    wl = small("shared", num_seqs=6, num_blocks=4096)
    case = synth.build_case(wl, "cuda", lengths=[64, 100, 1024, 65, 300, 17])
    out_shared = run_decode(pkv, case, partition_blocks=32).clone()
    bt = case.block_tables.clone()
    free = torch.ones(case.k_pool.shape[0], dtype=torch.bool)
    free[bt[bt >= 0].long().cpu()] = False
    free_ids = torch.nonzero(free).flatten()
    pos = 0
    pairs = []
    for s in range(bt.shape[0]):
        for j in range(256):
            pairs.append((int(bt[s, j]), int(free_ids[pos])))
            bt[s, j] = int(free_ids[pos])
            pos += 1
    pkv.copy_blocks(case.k_pool, case.v_pool, torch.tensor(pairs, dtype=torch.int32,
                                                           device="cuda"))
    out_copied = pkv.paged_decode(case.q, case.k_pool, case.v_pool, bt, case.context_lens,
                                  case.scale, max_context=case.max_context, partition_blocks=32)
    torch.cuda.synchronize()
    assert pkv.read_device_status() == 0
    assert torch.equal(out_shared.view(torch.int16), out_copied.view(torch.int16))


def test_permuted_placement_same_bits(pkv, kernel):
    """Moving every block to another physical id leaves the output bits unchanged."""
    wl = small("8b", num_seqs=5, num_blocks=2048)
    case = synth.build_case(wl, "cuda", lengths=[700, 33, 4096, 1, 1500], seed=77)
    out_a = run_decode(pkv, case).clone()
    nb = case.k_pool.shape[0]
    perm = torch.randperm(nb, generator=torch.Generator().manual_seed(5)).cuda()
    k2 = torch.empty_like(case.k_pool)
    v2 = torch.empty_like(case.v_pool)
    k2[perm] = case.k_pool
    v2[perm] = case.v_pool
    bt = case.block_tables.clone()
    m = bt >= 0
    bt[m] = perm[bt[m].long()].int()
    out_b = pkv.paged_decode(case.q, k2, v2, bt, case.context_lens, case.scale,
                             max_context=case.max_context)
    torch.cuda.synchronize()
    assert torch.equal(out_a.view(torch.int16), out_b.view(torch.int16))


def test_workspace_too_small_is_rejected(pkv):
    case = synth.build_case("tiny", "cuda")
    ws = torch.empty(16, dtype=torch.uint8, device="cuda")
    with pytest.raises(pkv.PkvError) as e:
        pkv.paged_decode(case.q, case.k_pool, case.v_pool, case.block_tables, case.context_lens,
                         case.scale, max_context=case.max_context, partition_blocks=1,
                         workspace=ws)
    assert e.value.status == 6


def test_out_of_range_block_id_raises_status(pkv):
    """A table entry past the pool is skipped by the kernel and reported (no fault)."""
    wl = small("8b", num_seqs=2, num_blocks=64)
    case = synth.build_case(wl, "cuda", lengths=[40, 20], seed=9)
    bt = case.block_tables.clone()
    bt[0, 1] = 64          # one past the last block
    pkv.paged_decode(case.q, case.k_pool, case.v_pool, bt, case.context_lens, case.scale,
                     max_context=case.max_context)
    assert pkv.read_device_status() == 5
    assert pkv.read_device_status() == 0


def test_zero_context_length_is_reported_and_zeroed(pkv, kernel):
    """A context length of 0 is outside the contract (a query sees at least its own
    key): the kernel reports PKV_ERR_INVALID and writes zeros to that sequence's rows;
    the other sequences are decoded as usual, with or without split-KV partitions."""
    wl = small("8b", num_seqs=3, num_blocks=256)
    for pb in (0, 1):
        case = synth.build_case(wl, "cuda", lengths=[40, 20, 300], seed=19)
        pkv.kv_append(case.k_pool, case.v_pool, case.slot_mapping, case.k_new, case.v_new)
        torch.cuda.synchronize()
        ref = pkv.paged_decode(case.q, case.k_pool, case.v_pool, case.block_tables,
                               case.context_lens, case.scale, max_context=case.max_context,
                               partition_blocks=pb)
        torch.cuda.synchronize()
        assert pkv.read_device_status() == 0
        lens = case.context_lens.clone()
        lens[1] = 0
        out = torch.full_like(case.q, float("nan"))
        pkv.paged_decode(case.q, case.k_pool, case.v_pool, case.block_tables, lens, case.scale,
                         max_context=case.max_context, partition_blocks=pb, out=out)
        torch.cuda.synchronize()
        assert pkv.read_device_status() == 1
        assert pkv.read_device_status() == 0
        assert torch.equal(out[1], torch.zeros_like(out[1]))
        assert torch.equal(out[0::2].view(torch.int16), ref[0::2].view(torch.int16))
