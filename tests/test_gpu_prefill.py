"""GPU parity of the tcgen05 prefix-chunk prefill against the fp64 oracle (C ABI)."""
import dataclasses

import numpy as np
import pytest
import torch

import synth
from tests.helpers import case_single_p, check_attention, oracle_prefill_case

pytestmark = pytest.mark.gpu


@pytest.fixture(scope="module")
def pkv():
    if not torch.cuda.is_available():
        pytest.skip("no CUDA device")
    import paged_kv_cache_58_gb300 as m
    from paged_kv_cache_58_gb300 import build
    build.build()
    return m


def run_prefill(pkv, case):
    pkv.kv_append(case.k_pool, case.v_pool, case.slot_mapping, case.k_new, case.v_new)
    out = pkv.paged_prefill(case.q, case.k_pool, case.v_pool, case.block_tables,
                            case.cached_lens, case.new_lens, case.q_offsets, case.scale,
                            max_new=int(case.new_lens.max()))
    torch.cuda.synchronize()
    assert pkv.read_device_status() == 0
    return out


def custom_case(hq, hkv, cached, new, seed, num_blocks=1024, **over):
    """Prefill case with per-request new lengths (the workload recipe fixes n); `over`
    replaces further recipe fields (head_dim, block_size)."""
    wl = dataclasses.replace(synth.WORKLOADS["prefill"], num_q_heads=hq, num_kv_heads=hkv,
                             new_tokens=max(new), num_blocks=num_blocks, **over)
    case = synth.build_case(wl, "cuda", lengths=cached, seed=seed)
    if all(x == max(new) for x in new):
        return case
    # keep the first new[r] tokens of each request: rebuild q / k_new / slots compactly
    n_max = max(new)
    keep = np.concatenate([np.arange(r * n_max, r * n_max + new[r]) for r in range(len(new))])
    keep_t = torch.as_tensor(keep, device="cuda")
    # drop the unused new tokens' pool slots back to NaN-free state is unnecessary: they
    # lie past each request's end and are never read as valid keys.
    case.q = case.q[keep_t].contiguous()
    case.k_new = case.k_new[keep_t].contiguous()
    case.v_new = case.v_new[keep_t].contiguous()
    case.slot_mapping = case.slot_mapping[keep_t].contiguous()
    case.new_lens = torch.tensor(new, dtype=torch.int32, device="cuda")
    case.q_offsets = torch.tensor(np.concatenate([[0], np.cumsum(new)]), dtype=torch.int32,
                                  device="cuda")
    case.context_lens = case.cached_lens + case.new_lens
    return case


@pytest.mark.parametrize("hq,hkv", [(32, 8), (8, 8), (16, 8), (64, 8)])
def test_prefill_small_mixed(pkv, oracle_mod, hq, hkv):
    cached = [0, 100, 1000, 16, 33]
    new = [37, 64, 300, 1, 128]
    case = custom_case(hq, hkv, cached, new, seed=hq)
    ref, _, _ = oracle_prefill_case(oracle_mod, case)
    check_attention(run_prefill(pkv, case), ref, single_p=case_single_p(case))


@pytest.mark.parametrize("cached,new", [([0], [1]), ([0], [128]), ([0], [129]), ([127], [1]),
                                        ([128], [128]), ([4095], [257]), ([1], [511])])
def test_prefill_edges(pkv, oracle_mod, cached, new):
    case = custom_case(32, 8, cached, new, seed=cached[0] + new[0])
    ref, _, _ = oracle_prefill_case(oracle_mod, case)
    check_attention(run_prefill(pkv, case), ref, single_p=case_single_p(case))


def test_prefill_p_modes_long_rows(pkv, oracle_mod, monkeypatch):
    """Query tiles whose rows all attend >= 1024 keys keep a single bf16 P by default;
    PKV_PREFILL_P=split forces the hi + lo split.  Both meet the tolerance on the same
    long-context case, and the split is closer to the oracle in RMS (its weights differ
    from the exact ones by 2^-14 instead of 2^-8)."""
    case = custom_case(32, 8, [1500, 3000], [200, 129], seed=11)
    ref, _, _ = oracle_prefill_case(oracle_mod, case)
    monkeypatch.delenv("PKV_PREFILL_P", raising=False)
    single = run_prefill(pkv, case)
    check_attention(single, ref, single_p=True)
    monkeypatch.setenv("PKV_PREFILL_P", "split")
    split = run_prefill(pkv, case)
    check_attention(split, ref)
    assert not torch.equal(single, split), "both runs took the same P path"
    rms = lambda t: float(np.sqrt(np.mean((t.double().cpu().numpy() - ref) ** 2)))
    assert rms(split) < rms(single)


def test_prefill_last_row_equals_decode(pkv, oracle_mod):
    """The last prefill row of a request equals a decode of that token (two kernels)."""
    case = custom_case(32, 8, [700], [40], seed=5)
    out = run_prefill(pkv, case)
    q_last = case.q[-1:].contiguous()
    dec = pkv.paged_decode(q_last, case.k_pool, case.v_pool, case.block_tables,
                           case.context_lens, case.scale, max_context=740)
    torch.cuda.synchronize()
    ref, _, _ = oracle_prefill_case(oracle_mod, case)
    check_attention(dec, ref[-1:])
    check_attention(out[-1:], ref[-1:], single_p=case_single_p(case))


def test_prefix_cached_prefill_published_config_full(pkv, oracle_mod):
    """Published prefill workload at full size (16 requests x 512 new tokens over cached
    prefixes of U[1024, 8192], 32 / 8 heads): every output against the oracle."""
    case = synth.build_case("prefill", "cuda")
    ref, _, _ = oracle_prefill_case(oracle_mod, case)
    out = run_prefill(pkv, case)
    assert ref.size == 8192 * 32 * 128
    check_attention(out, ref, single_p=True)


@pytest.mark.parametrize("dtype", [torch.bfloat16, torch.float32])
def test_prefill_out_of_range_block_id_raises_status(pkv, dtype):
    """A table entry past the pool inside a request's keys is not read (the tcgen05
    kernel stages block 0 in its place, the fp32 kernel zeros), and is reported."""
    case = custom_case(32, 8, [100, 40], [37, 64], seed=11, num_blocks=64, dtype=dtype)
    bt = case.block_tables.clone()
    bt[0, 2] = 64          # one past the last block: keys 32..47 of request 0
    pkv.paged_prefill(case.q, case.k_pool, case.v_pool, bt, case.cached_lens, case.new_lens,
                      case.q_offsets, case.scale, max_new=int(case.new_lens.max()))
    torch.cuda.synchronize()
    assert pkv.read_device_status() == 5
    assert pkv.read_device_status() == 0


@pytest.mark.parametrize("num_reqs", [128, 130])
def test_prefill_many_requests_both_schedules(pkv, oracle_mod, num_reqs):
    """128 requests run on persistent CTAs over the request-ranked item list, 130 on one
    CTA per query tile; ragged cached and new lengths, some requests without new tokens."""
    rng = np.random.default_rng(num_reqs)
    cached = [int(x) for x in rng.integers(0, 300, num_reqs)]
    new = [int(x) for x in rng.integers(0, 40, num_reqs)]
    new[0] = 40   # the recipe's n is max(new)
    case = custom_case(32, 8, cached, new, seed=num_reqs, num_blocks=4096)
    ref, _, _ = oracle_prefill_case(oracle_mod, case)
    check_attention(run_prefill(pkv, case), ref, single_p=case_single_p(case))


def host_prefill_step(pkv, case, mode):
    """pkv_paged_prefill_append_host over `case`, host buffers pinned, pageable or pinned
    but off a 16-byte boundary; returns the host output."""
    T, Hq, D = case.q.shape
    R = case.cached_lens.numel()
    mbs = case.block_tables.shape[1]
    lay = pkv.prefill_step_layout(case.k_pool, R, T, Hq, mbs)
    esz = case.q.element_size()
    if mode == "pinned_unaligned":
        host_in = torch.empty(lay.bytes + 16, dtype=torch.uint8).pin_memory()[8:8 + lay.bytes]
        raw = torch.empty((T * Hq * D + 16) * esz, dtype=torch.uint8).pin_memory()
        host_out = raw[esz:esz + T * Hq * D * esz].view(case.q.dtype).view(T, Hq, D)
    else:
        host_in = torch.empty(lay.bytes, dtype=torch.uint8)
        host_out = torch.empty((T, Hq, D), dtype=case.q.dtype)
        if mode == "pinned":
            host_in, host_out = host_in.pin_memory(), host_out.pin_memory()
    host_out.fill_(float("nan"))
    pkv.pack_prefill_step(host_in, lay, case.q.cpu(), case.block_tables.cpu(),
                          case.cached_lens.cpu(), case.new_lens.cpu(), case.q_offsets.cpu(),
                          case.k_new.cpu(), case.v_new.cpu(), case.slot_mapping.cpu())
    staging = torch.empty(pkv.prefill_host_staging_bytes(case.k_pool, R, T, Hq, mbs),
                          dtype=torch.uint8, device="cuda")
    pkv.paged_prefill_append_host(case.k_pool, case.v_pool, host_in, host_out, case.scale,
                                  num_reqs=R, total_new=T, max_new=int(case.new_lens.max()),
                                  num_q_heads=Hq, max_blocks_per_seq=mbs, staging=staging)
    torch.cuda.synchronize()
    assert pkv.read_device_status() == 0
    return host_out


@pytest.mark.parametrize("dtype", [torch.bfloat16, torch.float32], ids=["bf16", "fp32"])
@pytest.mark.parametrize("mode", ["pinned", "pageable", "pinned_unaligned"])
def test_prefill_host_step_matches_device_calls(pkv, mode, dtype):
    """pkv_paged_prefill_append_host (inputs copied in and the output copied back, in
    request chunks beside the kernels) gives the output bits and pools of kv_append +
    paged_prefill on device buffers, on bf16 (tensor cores) and fp32 (CUDA cores) pools,
    from pinned, pageable and misaligned pinned host buffers."""
    a = custom_case(32, 8, [0, 100, 1000, 16, 33], [37, 64, 300, 1, 128], seed=5, dtype=dtype)
    b = custom_case(32, 8, [0, 100, 1000, 16, 33], [37, 64, 300, 1, 128], seed=5, dtype=dtype)
    ref = run_prefill(pkv, b)
    out = host_prefill_step(pkv, a, mode)
    assert torch.equal(out.view(torch.uint8), ref.cpu().view(torch.uint8))
    assert torch.equal(a.k_pool.view(torch.uint8), b.k_pool.view(torch.uint8))
    assert torch.equal(a.v_pool.view(torch.uint8), b.v_pool.view(torch.uint8))


def test_prefill_host_step_published_batch(pkv):
    """The prefix-cached prefill batch (16 x 512 new tokens) through the host step with
    pinned buffers: the device calls' output bits."""
    a = synth.build_case("prefill", "cuda")
    b = synth.build_case("prefill", "cuda")
    ref = run_prefill(pkv, b)
    out = host_prefill_step(pkv, a, "pinned")
    assert torch.equal(out.view(torch.uint8), ref.cpu().view(torch.uint8))

