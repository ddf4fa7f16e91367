"""GPU parity of the shared-prefix cascade decode (C ABI) against the fp64 oracle
and against the plain paged decode."""
import dataclasses

import numpy as np
import pytest
import torch

import synth
from tests.helpers import check_attention, oracle_decode_case, to_f64

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


def test_shared_prefix_published_config_cascade(pkv, oracle_mod):
    case = synth.build_case("shared", "cuda")
    S, Hq = case.q.shape[:2]
    want = synth.sample_rows(S, Hq, 96, seed=11)
    ref, _, _ = oracle_decode_case(oracle_mod, case, want=want)
    casc, plain = run_both(pkv, case, 4096)
    check_attention(casc, ref, mask=want)
    check_attention(casc, to_f64(plain))     # every output against the plain decode


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
    check_attention(casc, ref)


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
