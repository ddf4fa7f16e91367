"""GPU parity of the fused append + decode (pkv_paged_decode_append) against the fp64
oracle and against kv_append followed by paged_decode.

Before the call the new token's slot holds NaN (every unowned slot does), so a kernel
that attended the pool row instead of k_new / v_new would poison its output."""
import dataclasses

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
    if request.param == "simt":
        monkeypatch.setenv("PKV_DECODE_KERNEL", "simt")
    else:
        monkeypatch.delenv("PKV_DECODE_KERNEL", raising=False)
    return request.param


def fused(pkv, case, partition_blocks=0):
    table_slots(case)
    out = pkv.paged_decode_append(case.q, case.k_pool, case.v_pool, case.k_new, case.v_new,
                                  case.block_tables, case.context_lens, case.scale,
                                  max_context=case.max_context,
                                  partition_blocks=partition_blocks)
    torch.cuda.synchronize()
    assert pkv.read_device_status() == 0
    return out


def separate(pkv, case, partition_blocks=0):
    pkv.kv_append(case.k_pool, case.v_pool, case.slot_mapping, case.k_new, case.v_new)
    out = pkv.paged_decode(case.q, case.k_pool, case.v_pool, case.block_tables,
                           case.context_lens, case.scale, max_context=case.max_context,
                           partition_blocks=partition_blocks)
    torch.cuda.synchronize()
    assert pkv.read_device_status() == 0
    return out


def table_slots(case):
    """The fused call stores token L-1 at the slot its table gives: check the case's
    slot_mapping (which the oracle's append uses) says the same."""
    bt = case.block_tables.cpu()
    lens = case.context_lens.cpu()
    B = case.k_pool.shape[2]
    want = [int(bt[s, (int(L) - 1) // B]) * B + (int(L) - 1) % B for s, L in enumerate(lens)]
    assert case.slot_mapping.cpu().tolist() == want


EDGE_LENS = [1, 2, 15, 16, 17, 31, 32, 33, 63, 64, 65, 127, 128, 129, 500, 1000]


@pytest.mark.parametrize("hq,hkv,d,bs", [(32, 8, 128, 16), (64, 8, 128, 16), (8, 8, 128, 16),
                                         (32, 8, 64, 16), (8, 1, 64, 16), (32, 8, 128, 32),
                                         (8, 2, 64, 32)])
@pytest.mark.parametrize("pb", [0, 1, 5])
def test_fused_matches_oracle_and_two_calls(pkv, oracle_mod, hq, hkv, d, bs, pb, kernel):
    wl = dataclasses.replace(synth.WORKLOADS["8b"], num_q_heads=hq, num_kv_heads=hkv,
                             head_dim=d, num_blocks=512, block_size=bs)
    seed = hq * 7 + d + pb + bs
    a = synth.build_case(wl, "cuda", lengths=EDGE_LENS, seed=seed)
    b = synth.build_case(wl, "cuda", lengths=EDGE_LENS, seed=seed)
    ref, kp, vp = oracle_decode_case(oracle_mod, a)
    out_f = fused(pkv, a, partition_blocks=pb)
    assert pool_equal(a.k_pool, kp) and pool_equal(a.v_pool, vp)
    check_attention(out_f, ref)
    out_s = separate(pkv, b, partition_blocks=pb)
    assert torch.equal(a.k_pool.view(torch.int16), b.k_pool.view(torch.int16))
    assert torch.equal(a.v_pool.view(torch.int16), b.v_pool.view(torch.int16))
    assert torch.equal(out_f.view(torch.int16), out_s.view(torch.int16))


@pytest.mark.parametrize("hq,hkv,d", [(4, 4, 64), (8, 2, 128), (32, 4, 128)])
def test_fused_fp32(pkv, oracle_mod, hq, hkv, d):
    wl = dataclasses.replace(synth.WORKLOADS["tiny"], num_q_heads=hq, num_kv_heads=hkv,
                             head_dim=d, num_blocks=256)
    case = synth.build_case(wl, "cuda", lengths=[1, 16, 17, 200, 333], seed=hq + d)
    ref, kp, vp = oracle_decode_case(oracle_mod, case)
    out = fused(pkv, case, partition_blocks=2)
    assert pool_equal(case.k_pool, kp) and pool_equal(case.v_pool, vp)
    check_attention(out, ref)


def test_fused_tiny_published_config(pkv, oracle_mod):
    case = synth.build_case("tiny", "cuda")
    ref, kp, vp = oracle_decode_case(oracle_mod, case)
    out = fused(pkv, case)
    assert pool_equal(case.k_pool, kp) and pool_equal(case.v_pool, vp)
    check_attention(out, ref)


def test_fused_llama3_8b_full(pkv, oracle_mod, kernel):
    """The Llama-3-8B-shaped batch at full size (the bench's launch configuration)."""
    case = synth.build_case("8b", "cuda")
    ref, kp, vp = oracle_decode_case(oracle_mod, case)
    out = fused(pkv, case)
    assert pool_equal(case.k_pool, kp) and pool_equal(case.v_pool, vp)
    check_attention(out, ref)


@pytest.mark.parametrize("wl_name", ["70b", "shared"])
def test_fused_full_size(pkv, published_decode_ref, wl_name):
    """The 70B long-context and shared-prefix batches at full size through the fused
    call (as the bench times them): every output against the oracle and every new slot
    stored."""
    ref = published_decode_ref(wl_name)
    case = synth.build_case(wl_name, "cuda")
    out = fused(pkv, case)
    check_attention(out, ref)
    B = case.k_pool.shape[2]
    blk, off = case.slot_mapping // B, case.slot_mapping % B
    assert torch.equal(case.k_pool[blk, :, off], case.k_new)
    assert torch.equal(case.v_pool[blk, :, off], case.v_new)


def test_fused_out_of_range_new_block_raises_status(pkv):
    """A table entry past the pool for the new token's block: no store, status OOB."""
    wl = dataclasses.replace(synth.WORKLOADS["8b"], num_seqs=2, num_blocks=64)
    case = synth.build_case(wl, "cuda", lengths=[40, 20], seed=9)
    bt = case.block_tables.clone()
    bt[0, 2] = 64          # block of token 39, one past the last block
    k_before = case.k_pool.clone()
    pkv.paged_decode_append(case.q, case.k_pool, case.v_pool, case.k_new, case.v_new, bt,
                            case.context_lens, case.scale, max_context=case.max_context)
    assert pkv.read_device_status() == 5
    assert pkv.read_device_status() == 0
    # only sequence 1's new slot changed
    diff = (case.k_pool.view(torch.int16) != k_before.view(torch.int16)).reshape(64, -1).any(1)
    s1 = int(case.slot_mapping[1]) // 16
    assert diff.nonzero().flatten().tolist() == [s1]


def test_fused_rejects_bad_new_rows(pkv):
    case = synth.build_case("tiny", "cuda")
    with pytest.raises(ValueError):
        pkv.paged_decode_append(case.q, case.k_pool, case.v_pool, case.k_new[:1],
                                case.v_new[:1], case.block_tables, case.context_lens,
                                case.scale, max_context=case.max_context)


@pytest.mark.parametrize("pinned", ["pinned", "pageable", "pinned_unaligned"])
@pytest.mark.parametrize("wl_name,lengths", [("8b", None), ("tiny", None),
                                             ("8b", [1, 16, 17, 4000, 33])])
def test_host_step_matches_device_call(pkv, wl_name, lengths, pinned):
    """pkv_paged_decode_append_host gives the device-buffer call's output bits and pools,
    with pinned host buffers (the kernels read the inputs and write the output in place),
    with pageable ones and with pinned ones off a 16-byte boundary (one copy each way
    through the staging buffer)."""
    kw = {} if lengths is None else {"lengths": lengths, "seed": 41}
    a = synth.build_case(wl_name, "cuda", **kw)
    b = synth.build_case(wl_name, "cuda", **kw)
    S, Hq, D = a.q.shape
    mbs = a.block_tables.shape[1]
    out_dev = fused(pkv, b)
    lay = pkv.decode_step_layout(a.k_pool, S, Hq, mbs)
    esz = a.q.element_size()
    if pinned == "pinned_unaligned":
        # views 8 bytes (input) and one element (output) past 16-byte aligned storage
        host_in = torch.empty(lay.bytes + 16, dtype=torch.uint8).pin_memory()[8:8 + lay.bytes]
        raw = torch.empty((S * Hq * D + 16) * esz, dtype=torch.uint8).pin_memory()
        host_out = raw[esz:esz + S * Hq * D * esz].view(a.q.dtype).view(S, Hq, D)
        host_out.fill_(float("nan"))
        assert host_in.data_ptr() % 16 == 8 and host_out.data_ptr() % 16 != 0
    else:
        host_in = torch.empty(lay.bytes, dtype=torch.uint8)
        host_out = torch.full((S, Hq, D), float("nan"), dtype=a.q.dtype)
        if pinned == "pinned":
            host_in, host_out = host_in.pin_memory(), host_out.pin_memory()
    assert host_in.is_pinned() == (pinned != "pageable")
    assert host_out.is_pinned() == (pinned != "pageable")
    pkv.pack_decode_step(host_in, lay, a.q.cpu(), a.k_new.cpu(), a.v_new.cpu(),
                         a.block_tables.cpu(), a.context_lens.cpu())
    staging = torch.empty(pkv.decode_host_staging_bytes(a.k_pool, S, Hq, mbs, a.max_context),
                          dtype=torch.uint8, device="cuda")
    pkv.paged_decode_append_host(a.k_pool, a.v_pool, host_in, host_out, a.scale, num_seqs=S,
                                 num_q_heads=Hq, max_blocks_per_seq=mbs,
                                 max_context=a.max_context, staging=staging)
    torch.cuda.synchronize()
    assert pkv.read_device_status() == 0
    assert torch.equal(host_out.view(torch.uint8), out_dev.cpu().view(torch.uint8))
    assert torch.equal(a.k_pool.view(torch.uint8), b.k_pool.view(torch.uint8))
    assert torch.equal(a.v_pool.view(torch.uint8), b.v_pool.view(torch.uint8))


def test_host_decode_step_plan_repeats_the_call(pkv):
    """HostDecodeStep (arguments bound once) gives the keyword call's output bits on
    every call, with the host buffer refilled in between."""
    a = synth.build_case("8b", "cuda")
    S, Hq, D = a.q.shape
    mbs = a.block_tables.shape[1]
    lay = pkv.decode_step_layout(a.k_pool, S, Hq, mbs)
    host_in = torch.empty(lay.bytes, dtype=torch.uint8).pin_memory()
    pkv.pack_decode_step(host_in, lay, a.q.cpu(), a.k_new.cpu(), a.v_new.cpu(),
                         a.block_tables.cpu(), a.context_lens.cpu())
    staging = torch.empty(pkv.decode_host_staging_bytes(a.k_pool, S, Hq, mbs, a.max_context),
                          dtype=torch.uint8, device="cuda")
    ref = torch.empty((S, Hq, D), dtype=a.q.dtype).pin_memory()
    kw = dict(num_seqs=S, num_q_heads=Hq, max_blocks_per_seq=mbs, max_context=a.max_context,
              staging=staging)
    pkv.paged_decode_append_host(a.k_pool, a.v_pool, host_in, ref, a.scale, **kw)
    torch.cuda.synchronize()
    out = torch.full((S, Hq, D), float("nan"), dtype=a.q.dtype).pin_memory()
    step = pkv.HostDecodeStep(a.k_pool, a.v_pool, host_in, out, a.scale, **kw)
    for i in range(3):
        out.fill_(float("nan"))
        q2 = a.q.cpu() * (1 + i)   # a different query each call, same new rows
        pkv.pack_decode_step(host_in, lay, q2, a.k_new.cpu(), a.v_new.cpu(),
                             a.block_tables.cpu(), a.context_lens.cpu())
        step()
        torch.cuda.synchronize()
        pkv.paged_decode_append_host(a.k_pool, a.v_pool, host_in, ref, a.scale, **kw)
        torch.cuda.synchronize()
        assert pkv.read_device_status() == 0
        assert torch.equal(out.view(torch.uint8), ref.view(torch.uint8))

