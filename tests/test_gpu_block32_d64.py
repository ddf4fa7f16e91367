"""GPU parity of the 32-token-block and head_dim-64 paths against the fp64 oracle (C ABI).

Pool blocks of 32 tokens are walked by every kernel as two 16-token chunks; the tcgen05
prefill (and with it the cascade decode's prefix pass) is templated on head_dim 64 and
128.  The pages allow blocks of 16 or 32 tokens (Triptych page, "Paged Attention for
Efficient Memory Management")."""
import dataclasses

import numpy as np
import pytest
import torch

import synth
from tests.helpers import (case_single_p, check_attention, oracle_decode_case,
                           oracle_prefill_case, pool_equal, to_f64)
from tests.test_gpu_prefill import custom_case, run_prefill

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


LENS32 = [1, 2, 16, 17, 31, 32, 33, 47, 48, 63, 64, 65, 100, 500, 1000, 2049]


@pytest.mark.parametrize("hq,hkv,d", [(32, 8, 128), (8, 2, 64), (64, 8, 128)])
@pytest.mark.parametrize("pb", [0, 1, 3])
def test_decode_block32_bf16(pkv, oracle_mod, hq, hkv, d, pb, kernel):
    wl = dataclasses.replace(synth.WORKLOADS["8b"], num_q_heads=hq, num_kv_heads=hkv,
                             head_dim=d, num_blocks=512, block_size=32)
    case = synth.build_case(wl, "cuda", lengths=LENS32, seed=hq + d + pb)
    ref, kp, vp = oracle_decode_case(oracle_mod, case)
    out = run_decode(pkv, case, partition_blocks=pb)
    assert pool_equal(case.k_pool, kp) and pool_equal(case.v_pool, vp)   # kv_append, B = 32
    check_attention(out, ref)


@pytest.mark.parametrize("pb", [0, 1, 2])
def test_decode_block32_fp32(pkv, oracle_mod, pb):
    wl = dataclasses.replace(synth.WORKLOADS["tiny"], block_size=32, num_blocks=64)
    case = synth.build_case(wl, "cuda", lengths=[17, 33, 5, 64, 65, 100], seed=7 + pb)
    ref, kp, vp = oracle_decode_case(oracle_mod, case)
    out = run_decode(pkv, case, partition_blocks=pb)
    assert pool_equal(case.k_pool, kp) and pool_equal(case.v_pool, vp)
    check_attention(out, ref)


def relay_block32(case16, seed):
    """The same logical K/V and queries laid out in a 32-token-block pool with its own
    random placement."""
    S = case16.q.shape[0]
    nb16, hkv, _, d = case16.k_pool.shape
    lens = case16.context_lens.cpu().tolist()
    nblk = [-(-L // 32) for L in lens]
    g = torch.Generator().manual_seed(seed)
    nb = sum(nblk) + 3
    perm = torch.randperm(nb, generator=g)
    kp = torch.full((nb, hkv, 32, d), float("nan"), dtype=case16.k_pool.dtype, device="cuda")
    vp = torch.full_like(kp, float("nan"))
    bt = torch.full((S, max(nblk)), -1, dtype=torch.int32)
    pos = 0
    bt16 = case16.block_tables.cpu()
    for s in range(S):
        bt[s, :nblk[s]] = perm[pos:pos + nblk[s]].to(torch.int32)
        pos += nblk[s]
        j = torch.arange(lens[s])
        src_b = bt16[s, j // 16].long().cuda()
        src_o = (j % 16).cuda()
        dst_b = bt[s, j // 32].long().cuda()
        dst_o = (j % 32).cuda()
        kp[dst_b, :, dst_o, :] = case16.k_pool[src_b, :, src_o, :]
        vp[dst_b, :, dst_o, :] = case16.v_pool[src_b, :, src_o, :]
    return kp, vp, bt.cuda()


@pytest.mark.parametrize("pb16", [2, 4, 64])
def test_block32_same_bits_as_block16(pkv, kernel, pb16):
    """Blocks of 32 are walked as the same 16-token chunks as blocks of 16, in the same
    order and with the same partitions (pb16 chunks = pb16 / 2 blocks): the outputs
    are bit-identical."""
    wl = dataclasses.replace(synth.WORKLOADS["8b"], num_blocks=1024)
    case = synth.build_case(wl, "cuda", lengths=[1, 33, 100, 1000, 2049, 4000], seed=21)
    out16 = run_decode(pkv, case, partition_blocks=pb16)
    kp, vp, bt = relay_block32(case, seed=22)
    out32 = pkv.paged_decode(case.q, kp, vp, bt, case.context_lens, case.scale,
                             max_context=case.max_context, partition_blocks=pb16 // 2)
    torch.cuda.synchronize()
    assert pkv.read_device_status() == 0
    assert torch.equal(out16, out32)


@pytest.mark.parametrize("d,bs", [(64, 16), (64, 32), (128, 32)])
@pytest.mark.parametrize("hq,hkv", [(32, 8), (8, 8), (16, 2)])
def test_prefill_d64_and_block32(pkv, oracle_mod, d, bs, hq, hkv):
    cached = [0, 100, 1000, 16, 33, 1500]
    new = [37, 64, 300, 1, 128, 200]
    case = custom_case(hq, hkv, cached, new, seed=d + bs + hq, head_dim=d, block_size=bs)
    ref, kp, vp = oracle_prefill_case(oracle_mod, case)
    out = run_prefill(pkv, case)
    assert pool_equal(case.k_pool, kp) and pool_equal(case.v_pool, vp)
    check_attention(out, ref, single_p=case_single_p(case))


@pytest.mark.parametrize("d,bs", [(64, 16), (64, 32), (128, 32)])
def test_prefill_edges_d64_block32(pkv, oracle_mod, d, bs):
    for cached, new in (([0], [1]), ([0], [129]), ([31], [1]), ([32], [33]), ([4095], [257])):
        case = custom_case(32, 8, cached, new, seed=cached[0] + new[0] + d, head_dim=d,
                           block_size=bs)
        ref, _, _ = oracle_prefill_case(oracle_mod, case)
        check_attention(run_prefill(pkv, case), ref, single_p=case_single_p(case))


@pytest.mark.parametrize("d,bs,hq,hkv", [(64, 16, 8, 2), (128, 16, 32, 8), (64, 32, 4, 4),
                                         (128, 32, 8, 1)])
def test_prefill_fp32(pkv, oracle_mod, d, bs, hq, hkv):
    """fp32 pools: the tiled CUDA-core prefill, causal, fp32 throughout."""
    case = custom_case(hq, hkv, [0, 100, 33, 1], [37, 64, 17, 1], seed=d + bs + hq,
                       head_dim=d, block_size=bs, dtype=torch.float32)
    ref, kp, vp = oracle_prefill_case(oracle_mod, case)
    out = run_prefill(pkv, case)
    assert pool_equal(case.k_pool, kp) and pool_equal(case.v_pool, vp)
    max_abs, _ = check_attention(out, ref)
    assert max_abs < 1e-5   # fp32 arithmetic throughout


@pytest.mark.parametrize("d,bs,hq,hkv", [(128, 16, 32, 8), (64, 32, 16, 8), (128, 32, 8, 8),
                                         (64, 16, 64, 8)])
def test_prefill_fp32_multi_tile(pkv, oracle_mod, d, bs, hq, hkv):
    """fp32 pools over several 64-row query tiles and 64-key KV tiles: ragged last tiles,
    cached prefixes off every tile and block boundary, a one-token request, G 1 to 8."""
    case = custom_case(hq, hkv, [0, 1000, 65, 4095, 63], [129, 300, 64, 1, 77],
                       seed=7 * d + bs + hq, head_dim=d, block_size=bs, dtype=torch.float32)
    ref, kp, vp = oracle_prefill_case(oracle_mod, case)
    out = run_prefill(pkv, case)
    assert pool_equal(case.k_pool, kp) and pool_equal(case.v_pool, vp)
    max_abs, _ = check_attention(out, ref)
    assert max_abs < 1e-5   # fp32 arithmetic throughout


@pytest.mark.parametrize("d,bs,hq,prefix,suffixes,pb", [
    (128, 32, 32, 64, [1, 33, 100, 31], 0),
    (64, 16, 8, 160, [5, 300, 1], 2),
    (64, 32, 16, 128, [1, 31, 64, 700], 1),
])
def test_cascade_d64_and_block32(pkv, oracle_mod, d, bs, hq, prefix, suffixes, pb):
    wl = dataclasses.replace(synth.WORKLOADS["shared"], num_seqs=len(suffixes), num_q_heads=hq,
                             head_dim=d, shared_prefix=prefix, num_blocks=512, block_size=bs)
    case = synth.build_case(wl, "cuda", lengths=suffixes, seed=prefix + hq + d)
    ref, _, _ = oracle_decode_case(oracle_mod, case)
    pkv.kv_append(case.k_pool, case.v_pool, case.slot_mapping, case.k_new, case.v_new)
    prefix_blocks = case.block_tables[0, :prefix // bs].contiguous()
    casc = pkv.paged_decode_cascade(case.q, case.k_pool, case.v_pool, prefix_blocks, prefix,
                                    case.block_tables, case.context_lens, case.scale,
                                    max_context=case.max_context, partition_blocks=pb)
    torch.cuda.synchronize()
    assert pkv.read_device_status() == 0
    check_attention(casc, ref)


def test_copy_blocks_block32_bit_exact(pkv, oracle_mod):
    g = torch.Generator().manual_seed(5)
    kp = torch.randn((12, 4, 32, 64), generator=g).to(torch.bfloat16).cuda()
    vp = torch.randn((12, 4, 32, 64), generator=g).to(torch.bfloat16).cuda()
    pairs = torch.tensor([[1, 7], [3, 0], [11, 4]], dtype=torch.int32)
    hk, hv = synth.host_bits(kp), synth.host_bits(vp)
    oracle_mod.copy_blocks(pairs.numpy(), hk, hv)
    pkv.copy_blocks(kp, vp, pairs.cuda())
    torch.cuda.synchronize()
    assert pkv.read_device_status() == 0
    assert pool_equal(kp, hk) and pool_equal(vp, hv)
