"""The allocation-free decode entry point against the workspace-taking one.

pkv_paged_decode_noalloc serves callers that cannot allocate device memory (a
fixed arena, a host process that owns every allocation, a loop that must not
call the allocator); its split-KV partials live in a scratch array built into
libpkv.  These tests call it through the C ABI, twice in a row, and check each
output bit for bit against pkv_paged_decode with a caller-allocated workspace
(the same kernels with the same partitions) and against the fp64 oracle; then
a call that fills much of the scratch array followed by a smaller one.  They sit
in their own file, collected last, and pass alone or after the other tests.
"""
import ctypes
import dataclasses

import pytest
import torch

import synth
from tests.helpers import check_attention, oracle_decode_case

pytestmark = pytest.mark.gpu


@pytest.fixture(scope="module")
def pkv():
    if not torch.cuda.is_available():
        pytest.skip("no CUDA device")
    from paged_kv_cache_58_gb300 import build
    build.build()
    import paged_kv_cache_58_gb300 as m
    lib = m.lib()
    vp, ci = ctypes.c_void_p, ctypes.c_int
    lib.pkv_paged_decode_noalloc.restype = ci
    lib.pkv_paged_decode_noalloc.argtypes = [ctypes.POINTER(m.PoolDesc), vp, vp, vp, vp, vp, ci,
                                             vp, ci, ci, ci, ctypes.c_float, ci, vp]
    return m


def call_noalloc(m, case, out, num_seqs=None, max_context=None):
    desc = m.pool_desc(case.k_pool)
    S, Hq, _ = case.q.shape
    return m.lib().pkv_paged_decode_noalloc(
        ctypes.byref(desc), out.data_ptr(), case.q.data_ptr(), case.k_pool.data_ptr(),
        case.v_pool.data_ptr(), case.block_tables.data_ptr(), case.block_tables.shape[1],
        case.context_lens.data_ptr(), max_context or case.max_context, num_seqs or S, Hq,
        case.scale, 0, torch.cuda.current_stream().cuda_stream)


def workspace_decode(m, case):
    out = m.paged_decode(case.q, case.k_pool, case.v_pool, case.block_tables,
                         case.context_lens, case.scale, max_context=case.max_context)
    torch.cuda.synchronize()
    assert m.read_device_status() == 0
    return out


def test_noalloc_decode_matches_workspace_decode(pkv, oracle_mod):
    """The 8B-shaped batch, twice in a row: the same kernels with the same partitions
    as the workspace call, so the same output bits, and within tolerance of the
    oracle."""
    case = synth.build_case("8b", "cuda")
    assert pkv.decode_workspace_bytes(*case.q.shape[:2], case.q.shape[2], case.max_context) > 0
    ref64, _, _ = oracle_decode_case(oracle_mod, case)
    pkv.kv_append(case.k_pool, case.v_pool, case.slot_mapping, case.k_new, case.v_new)
    ref = workspace_decode(pkv, case)
    for _ in range(2):
        out = torch.full_like(case.q, float("nan"))
        assert call_noalloc(pkv, case, out) == 0
        torch.cuda.synchronize()
        assert pkv.read_device_status() == 0
        assert torch.equal(out.view(torch.int16), ref.view(torch.int16))
        check_attention(out, ref64)


def test_noalloc_smaller_call_after_larger_one(pkv):
    """A call whose partials fill much of the scratch array (64 sequences of up to 32768
    tokens), then a smaller one: the smaller call reads only what it wrote itself."""
    big = synth.build_case(dataclasses.replace(synth.WORKLOADS["8b"], num_blocks=110000),
                           "cuda", lengths=[32768 - 250 * i for i in range(64)], seed=12)
    need = pkv.decode_workspace_bytes(*big.q.shape[:2], big.q.shape[2], big.max_context)
    assert 16 << 20 < need <= 64 << 20
    small = synth.build_case("8b", "cuda")
    for c in (big, small):
        pkv.kv_append(c.k_pool, c.v_pool, c.slot_mapping, c.k_new, c.v_new)
    ref_big, ref_small = workspace_decode(pkv, big), workspace_decode(pkv, small)
    for c, ref in ((big, ref_big), (small, ref_small)):
        out = torch.full_like(c.q, float("nan"))
        assert call_noalloc(pkv, c, out) == 0
        torch.cuda.synchronize()
        assert pkv.read_device_status() == 0
        assert torch.equal(out.view(torch.int16), ref.view(torch.int16))


def test_noalloc_rejects_requests_beyond_its_scratch(pkv):
    case = synth.build_case("tiny", "cuda")
    out = torch.empty_like(case.q)
    # 65535 sequences of up to 64 tokens with 1-block partitions need far more than
    # 64 MiB of partials; the call must refuse before launching anything.
    desc = pkv.pool_desc(case.k_pool)
    st = pkv.lib().pkv_paged_decode_noalloc(
        ctypes.byref(desc), out.data_ptr(), case.q.data_ptr(), case.k_pool.data_ptr(),
        case.v_pool.data_ptr(), case.block_tables.data_ptr(), case.block_tables.shape[1],
        case.context_lens.data_ptr(), 64, 65535, case.q.shape[1], case.scale, 1,
        torch.cuda.current_stream().cuda_stream)
    assert st == 6
