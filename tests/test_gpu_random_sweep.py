"""Seeded random sweep of the decode family on the GPU: for each drawn configuration
(sequences, GQA group, head_dim, block size, partition size, context lengths from 1 up),
the fused call and kv_append + paged_decode give the same output bits and pools, both
match the fp64 oracle, on the tensor-core and the CUDA-core kernels."""
import dataclasses

import numpy as np
import pytest
import torch

import synth
from tests.helpers import case_single_p, check_attention, oracle_decode_case, pool_equal

pytestmark = pytest.mark.gpu


@pytest.fixture(scope="module")
def pkv():
    if not torch.cuda.is_available():
        pytest.skip("no CUDA device")
    import paged_kv_cache_58_gb300 as m
    from paged_kv_cache_58_gb300 import build
    build.build()
    return m


def draw(i):
    rng = np.random.default_rng(1000 + i)
    hkv = int(rng.choice([1, 2, 4, 8]))
    g = int(rng.choice([1, 2, 4, 8]))
    d = int(rng.choice([64, 128]))
    bs = int(rng.choice([16, 32]))
    s = int(rng.integers(1, 9))
    lens = [int(x) for x in rng.choice(
        [1, 2, 15, 16, 17, 31, 32, 33, 63, 64, 65, 127, 128, 129, 511, 1023, 1025, 2047, 3000],
        size=s)]
    pb = int(rng.choice([0, 1, 2, 3, 8]))
    kernel = str(rng.choice(["tc", "simt"]))
    return hkv, g, d, bs, lens, pb, kernel


@pytest.mark.parametrize("i", range(24))
def test_random_decode_config(pkv, oracle_mod, monkeypatch, i):
    hkv, g, d, bs, lens, pb, kernel = draw(i)
    if kernel == "simt":
        monkeypatch.setenv("PKV_DECODE_KERNEL", "simt")
    else:
        monkeypatch.delenv("PKV_DECODE_KERNEL", raising=False)
    nb = sum(-(-L // bs) for L in lens) + 64
    wl = dataclasses.replace(synth.WORKLOADS["8b"], num_seqs=len(lens), num_q_heads=hkv * g,
                             num_kv_heads=hkv, head_dim=d, block_size=bs, num_blocks=nb)
    a = synth.build_case(wl, "cuda", lengths=lens, seed=2000 + i)
    b = synth.build_case(wl, "cuda", lengths=lens, seed=2000 + i)
    ref, kp, vp = oracle_decode_case(oracle_mod, a)
    out_f = pkv.paged_decode_append(a.q, a.k_pool, a.v_pool, a.k_new, a.v_new, a.block_tables,
                                    a.context_lens, a.scale, max_context=a.max_context,
                                    partition_blocks=pb)
    pkv.kv_append(b.k_pool, b.v_pool, b.slot_mapping, b.k_new, b.v_new)
    out_s = pkv.paged_decode(b.q, b.k_pool, b.v_pool, b.block_tables, b.context_lens, b.scale,
                             max_context=b.max_context, partition_blocks=pb)
    torch.cuda.synchronize()
    assert pkv.read_device_status() == 0
    assert pool_equal(a.k_pool, kp) and pool_equal(a.v_pool, vp)
    assert torch.equal(a.k_pool.view(torch.uint8), b.k_pool.view(torch.uint8))
    assert torch.equal(out_f.view(torch.uint8), out_s.view(torch.uint8))
    check_attention(out_f, ref)


def draw_prefill(i):
    rng = np.random.default_rng(3000 + i)
    hkv = int(rng.choice([1, 2, 8]))
    g = int(rng.choice([1, 2, 4, 8]))
    d = int(rng.choice([64, 128]))
    bs = int(rng.choice([16, 32]))
    r = int(rng.integers(1, 5))
    cached = [int(x) for x in rng.choice([0, 1, 15, 16, 100, 127, 128, 1000, 1024, 1500, 2100],
                                         size=r)]
    new = [int(x) for x in rng.choice([1, 2, 31, 32, 33, 100, 129, 300], size=r)]
    return hkv, g, d, bs, cached, new


@pytest.mark.parametrize("i", range(16))
def test_random_prefill_config(pkv, oracle_mod, i):
    """tcgen05 prefill on drawn (requests, cached and new lengths, GQA group, head_dim,
    block size): rows with 1024 keys or more take the single-P path, others the split."""
    from tests.helpers import oracle_prefill_case
    from tests.test_gpu_prefill import custom_case, run_prefill
    hkv, g, d, bs, cached, new = draw_prefill(i)
    nb = sum(-(-(c + n) // bs) for c, n in zip(cached, new)) + 64
    case = custom_case(hkv * g, hkv, cached, new, seed=4000 + i, num_blocks=nb, head_dim=d,
                       block_size=bs)
    ref, kp, vp = oracle_prefill_case(oracle_mod, case)
    out = run_prefill(pkv, case)
    assert pool_equal(case.k_pool, kp) and pool_equal(case.v_pool, vp)
    check_attention(out, ref, single_p=case_single_p(case))
