"""GPU parity of kv_append, copy_blocks and the allocator-driven CoW flow (C ABI)."""
import numpy as np
import pytest
import torch

import synth
from tests.helpers import check_attention, pool_equal

pytestmark = pytest.mark.gpu


@pytest.fixture(scope="module")
def pkv():
    if not torch.cuda.is_available():
        pytest.skip("no CUDA device")
    import paged_kv_cache_58_gb300 as m
    from paged_kv_cache_58_gb300 import build
    build.build()
    return m


@pytest.mark.parametrize("kernel", ["pow2", "generic"])
@pytest.mark.parametrize("dtype,d,hkv", [(torch.bfloat16, 128, 8), (torch.bfloat16, 64, 2),
                                         (torch.float32, 128, 4), (torch.float32, 64, 1),
                                         (torch.bfloat16, 128, 3)])
def test_kv_append_bit_exact(pkv, oracle_mod, dtype, d, hkv, kernel, monkeypatch):
    """Both append kernels (the general one normally runs only past 2^31 chunks; the
    test hook sends these calls to it) against the oracle scatter, bit for bit."""
    if kernel == "generic":
        monkeypatch.setenv("PKV_TEST_APPEND_GENERIC", "1")
    g = torch.Generator().manual_seed(d + hkv)
    nb, T = 40, 300
    kp = torch.randn((nb, hkv, 16, d), generator=g).to(dtype).cuda()
    vp = torch.randn((nb, hkv, 16, d), generator=g).to(dtype).cuda()
    slots = torch.randperm(nb * 16, generator=g)[:T]
    slots[::7] = -1                        # padding rows are skipped
    k = torch.randn((T, hkv, d), generator=g).to(dtype).cuda()
    v = torch.randn((T, hkv, d), generator=g).to(dtype).cuda()
    hk, hv = synth.host_bits(kp), synth.host_bits(vp)
    oracle_mod.kv_append(slots.numpy(), synth.host_bits(k), synth.host_bits(v), hk, hv)
    pkv.kv_append(kp, vp, slots.cuda(), k, v)
    torch.cuda.synchronize()
    assert pkv.read_device_status() == 0
    assert pool_equal(kp, hk) and pool_equal(vp, hv)


def test_kv_append_prefill_sized(pkv, oracle_mod):
    """The 8192-token append of the prefix-cached prefill workload, bit-exact."""
    case = synth.build_case("prefill", "cuda")
    hk, hv = synth.host_bits(case.k_pool), synth.host_bits(case.v_pool)
    oracle_mod.kv_append(synth.host_bits(case.slot_mapping), synth.host_bits(case.k_new),
                         synth.host_bits(case.v_new), hk, hv)
    pkv.kv_append(case.k_pool, case.v_pool, case.slot_mapping, case.k_new, case.v_new)
    torch.cuda.synchronize()
    assert pkv.read_device_status() == 0
    assert pool_equal(case.k_pool, hk) and pool_equal(case.v_pool, hv)


def test_kv_append_empty_is_noop(pkv):
    kp = torch.zeros((4, 1, 16, 64), dtype=torch.bfloat16, device="cuda")
    vp = torch.zeros_like(kp)
    e = torch.empty((0, 1, 64), dtype=torch.bfloat16, device="cuda")
    pkv.kv_append(kp, vp, torch.empty(0, dtype=torch.int64, device="cuda"), e, e)
    torch.cuda.synchronize()
    assert not kp.any()


def test_kv_append_out_of_range_slot_reported(pkv):
    kp = torch.zeros((4, 1, 16, 64), dtype=torch.bfloat16, device="cuda")
    vp = torch.zeros_like(kp)
    k = torch.ones((2, 1, 64), dtype=torch.bfloat16, device="cuda")
    pkv.kv_append(kp, vp, torch.tensor([3, 64], dtype=torch.int64, device="cuda"), k, k)
    assert pkv.read_device_status() == 5
    assert kp[0, 0, 3].eq(1).all() and kp.sum().item() == 64


def test_copy_blocks_bit_exact(pkv, oracle_mod):
    g = torch.Generator().manual_seed(3)
    kp = torch.randn((20, 8, 16, 128), generator=g).to(torch.bfloat16).cuda()
    vp = torch.randn((20, 8, 16, 128), generator=g).to(torch.bfloat16).cuda()
    pairs = torch.tensor([[1, 7], [3, 0], [19, 4]], dtype=torch.int32)
    hk, hv = synth.host_bits(kp), synth.host_bits(vp)
    oracle_mod.copy_blocks(pairs.numpy(), hk, hv)
    pkv.copy_blocks(kp, vp, pairs.cuda())
    torch.cuda.synchronize()
    assert pkv.read_device_status() == 0
    assert pool_equal(kp, hk) and pool_equal(vp, hv)


def test_fork_append_cow_keeps_parent_view(pkv, oracle_mod):
    """Allocator-driven flow: fork mid-block, append to the child (CoW), decode both."""
    torch.manual_seed(0)
    hkv, hq, d, nb = 8, 32, 128, 64
    alloc = pkv.BlockAllocator(nb, seed=11)
    kp = torch.full((nb, hkv, 16, d), float("nan"), dtype=torch.bfloat16, device="cuda")
    vp = torch.full_like(kp, float("nan"))
    # parent holds 37 tokens (3 blocks, last one partial)
    alloc.add_seq(0, 0)
    slots, cow = alloc.append(0, 37)
    assert cow is None
    k = torch.randn((37, hkv, d)).to(torch.bfloat16).cuda()
    v = torch.randn((37, hkv, d)).to(torch.bfloat16).cuda()
    pkv.kv_append(kp, vp, torch.tensor(slots, device="cuda"), k, v)
    alloc.fork(0, 1)
    last = alloc.block_table([0], 4)[0, 2].item()
    assert alloc.refcount(last) == 2
    # child diverges: its write must go to a private copy of the shared partial block
    cslots, cow = alloc.append(1, 1)
    assert cow is not None and cow[0] == last and alloc.refcount(last) == 1
    pkv.copy_blocks(kp, vp, torch.tensor([cow], dtype=torch.int32, device="cuda"))
    kn = torch.randn((1, hkv, d)).to(torch.bfloat16).cuda()
    vn = torch.randn((1, hkv, d)).to(torch.bfloat16).cuda()
    pkv.kv_append(kp, vp, torch.tensor(cslots, device="cuda"), kn, vn)
    # parent appends too (its block is private again: no CoW)
    pslots, pcow = alloc.append(0, 1)
    assert pcow is None
    kn2 = torch.randn((1, hkv, d)).to(torch.bfloat16).cuda()
    vn2 = torch.randn((1, hkv, d)).to(torch.bfloat16).cuda()
    pkv.kv_append(kp, vp, torch.tensor(pslots, device="cuda"), kn2, vn2)
    bt = alloc.block_table([0, 1], 4).cuda()
    lens = torch.tensor([38, 38], dtype=torch.int32, device="cuda")
    q = torch.randn((2, hq, d)).to(torch.bfloat16).cuda()
    out = pkv.paged_decode(q, kp, vp, bt, lens, 0.088, max_context=38)
    torch.cuda.synchronize()
    assert pkv.read_device_status() == 0
    ref = oracle_mod.paged_decode(synth.host_bits(q), synth.host_bits(kp), synth.host_bits(vp),
                                  bt.cpu().numpy(), lens.cpu().numpy(), 0.088)
    check_attention(out, ref)
    # each sequence sees its own token 37
    K0, _ = oracle_mod.gather(synth.host_bits(kp), synth.host_bits(vp), bt[0].cpu().numpy(), 38, 0)
    K1, _ = oracle_mod.gather(synth.host_bits(kp), synth.host_bits(vp), bt[1].cpu().numpy(), 38, 0)
    np.testing.assert_array_equal(K0[:37], K1[:37])
    np.testing.assert_array_equal(K0[37], kn2[0, 0].float().cpu().numpy())
    np.testing.assert_array_equal(K1[37], kn[0, 0].float().cpu().numpy())
    alloc.close()
