"""GPU parity of the shared-prefix cascade decode (C ABI) against the fp64 oracle
and against the plain paged decode."""
import dataclasses

import numpy as np
import pytest
import torch

import synth
from tests.helpers import check_attention, oracle_decode_case

pytestmark = pytest.mark.gpu


@pytest.fixture(scope="module")
def pkv():
    if not torch.cuda.is_available():
        pytest.skip("no CUDA device")
    import paged_kv_cache_58_gb300 as m
    from paged_kv_cache_58_gb300 import build
    build.build()
    return m


def run_both(pkv, case, prefix_len, partition_blocks=0):
    pkv.kv_append(case.k_pool, case.v_pool, case.slot_mapping, case.k_new, case.v_new)
    prefix_blocks = case.block_tables[0, :prefix_len // 16].contiguous()
    casc = pkv.paged_decode_cascade(case.q, case.k_pool, case.v_pool, prefix_blocks, prefix_len,
                                    case.block_tables, case.context_lens, case.scale,
                                    max_context=case.max_context,
                                    partition_blocks=partition_blocks)
    plain = pkv.paged_decode(case.q, case.k_pool, case.v_pool, case.block_tables,
                             case.context_lens, case.scale, max_context=case.max_context)
    torch.cuda.synchronize()
    assert pkv.read_device_status() == 0
    return casc, plain


def test_shared_prefix_published_config_cascade(pkv, published_decode_ref):
    """Published shared-prefix batch (256 sequences on one 4096-token prefix, private
    suffixes U[64, 1024]): every output of the cascade and of the plain decode against
    the oracle.  The prefix pass attends 4096 keys per row, so it keeps one bf16 P."""
    ref = published_decode_ref("shared")
    case = synth.build_case("shared", "cuda")
    casc, plain = run_both(pkv, case, 4096)
    assert ref.size == 256 * 32 * 128
    check_attention(casc, ref, single_p=True)
    check_attention(plain, ref)


@pytest.mark.parametrize("hq,prefix,suffixes,pb", [
    (32, 16, [1, 15, 16, 17, 100], 0),
    (32, 160, [1, 2, 300, 64, 1000], 2),
    (8, 64, [5, 33, 1, 200], 1),
    (64, 512, [1, 700, 31], 0),
    (16, 32, [129, 1, 17], 3),
])
def test_cascade_small_cases(pkv, oracle_mod, hq, prefix, suffixes, pb):
    wl = dataclasses.replace(synth.WORKLOADS["shared"], num_seqs=len(suffixes), num_q_heads=hq,
                             shared_prefix=prefix, num_blocks=1024)
    case = synth.build_case(wl, "cuda", lengths=suffixes, seed=prefix + hq)
    ref, _, _ = oracle_decode_case(oracle_mod, case)
    casc, _ = run_both(pkv, case, prefix, pb)
    check_attention(casc, ref, single_p=prefix >= 1024)


def test_cascade_without_private_suffix(pkv, oracle_mod):
    """Every context equals the prefix (the decoded token is its last token)."""
    wl = dataclasses.replace(synth.WORKLOADS["shared"], num_seqs=3, shared_prefix=64,
                             num_blocks=64)
    case = synth.build_case(wl, "cuda", lengths=[0, 0, 0], seed=3)
    # with no suffix the decoded token is the prefix's last token, one shared slot:
    # only the first sequence writes it (a negative slot skips the row)
    case.slot_mapping[1:] = -1
    ref, _, _ = oracle_decode_case(oracle_mod, case)
    casc, _ = run_both(pkv, case, 64)
    check_attention(casc, ref)


def fused_cascade(pkv, case, prefix_len, partition_blocks=0):
    prefix_blocks = case.block_tables[0, :prefix_len // 16].contiguous()
    return pkv.paged_decode_cascade_append(case.q, case.k_pool, case.v_pool, case.k_new,
                                           case.v_new, prefix_blocks, prefix_len,
                                           case.block_tables, case.context_lens, case.scale,
                                           max_context=case.max_context,
                                           partition_blocks=partition_blocks)


@pytest.mark.parametrize("hq,prefix,suffixes,pb", [
    (32, 16, [1, 15, 16, 17, 100], 0),
    (32, 160, [1, 2, 300, 64, 1000], 2),
    (8, 64, [5, 33, 1, 200], 1),
])
def test_cascade_fused_append_matches_oracle_and_two_calls(pkv, oracle_mod, hq, prefix,
                                                           suffixes, pb):
    """pkv_paged_decode_cascade_append: the suffix decode stores and attends the newest
    tokens; same pools and output bits as kv_append followed by the cascade decode."""
    from tests.helpers import pool_equal
    wl = dataclasses.replace(synth.WORKLOADS["shared"], num_seqs=len(suffixes), num_q_heads=hq,
                             shared_prefix=prefix, num_blocks=1024)
    a = synth.build_case(wl, "cuda", lengths=suffixes, seed=prefix + hq + 1)
    b = synth.build_case(wl, "cuda", lengths=suffixes, seed=prefix + hq + 1)
    ref, kp, vp = oracle_decode_case(oracle_mod, a)
    out_f = fused_cascade(pkv, a, prefix, pb)
    torch.cuda.synchronize()
    assert pkv.read_device_status() == 0
    assert pool_equal(a.k_pool, kp) and pool_equal(a.v_pool, vp)
    check_attention(out_f, ref)
    out_s, _ = run_both(pkv, b, prefix, pb)
    assert torch.equal(out_f.view(torch.int16), out_s.view(torch.int16))
    assert torch.equal(a.k_pool.view(torch.int16), b.k_pool.view(torch.int16))


def test_cascade_fused_append_published_batch_full(pkv, published_decode_ref):
    """The published shared-prefix batch through the fused cascade call: every output
    against the oracle, and every new token stored at its slot."""
    ref = published_decode_ref("shared")
    case = synth.build_case("shared", "cuda")
    out = fused_cascade(pkv, case, 4096)
    torch.cuda.synchronize()
    assert pkv.read_device_status() == 0
    check_attention(out, ref, single_p=True)
    B = case.k_pool.shape[2]
    blk, off = case.slot_mapping // B, case.slot_mapping % B
    assert torch.equal(case.k_pool[blk, :, off], case.k_new)


def test_cascade_fused_append_token_inside_prefix_is_reported(pkv):
    """A sequence whose newest token lies in the shared prefix: nothing is stored into the
    shared blocks and the device status reads PKV_ERR_INVALID."""
    wl = dataclasses.replace(synth.WORKLOADS["shared"], num_seqs=3, shared_prefix=64,
                             num_blocks=256)
    case = synth.build_case(wl, "cuda", lengths=[0, 5, 0], seed=8)
    shared = case.block_tables[0, :4].long()
    k_before = case.k_pool[shared].clone()
    fused_cascade(pkv, case, 64)
    torch.cuda.synchronize()
    assert pkv.read_device_status() == 1
    assert pkv.read_device_status() == 0
    assert torch.equal(case.k_pool[shared].view(torch.int16), k_before.view(torch.int16))
    B = case.k_pool.shape[2]
    s1 = int(case.slot_mapping[1])
    assert torch.equal(case.k_pool[s1 // B, :, s1 % B], case.k_new[1])
