"""Stream capture: a decode step (kv_append + paged_decode, or the fused call), a
cascade decode and the host-buffer decode and prefill steps (pinned buffers) can be
recorded into a CUDA graph and replayed -- the calls allocate nothing and never
synchronise -- and a replay gives the same bits as the eager calls.
The forks onto the library's own streams (the cascade's prefix pass, the prefill
step's copies) become part of the graph."""
import dataclasses

import pytest
import torch

import synth

pytestmark = pytest.mark.gpu


@pytest.fixture(scope="module")
def pkv():
    if not torch.cuda.is_available():
        pytest.skip("no CUDA device")
    import paged_kv_cache_58_gb300 as m
    from paged_kv_cache_58_gb300 import build
    build.build()
    return m


def capture(fn):
    s = torch.cuda.Stream()
    s.wait_stream(torch.cuda.current_stream())
    g = torch.cuda.CUDAGraph()
    with torch.cuda.graph(g, stream=s):
        fn()
    torch.cuda.current_stream().wait_stream(s)
    return g


def test_decode_step_graph_replay(pkv):
    wl = dataclasses.replace(synth.WORKLOADS["8b"], num_seqs=16, num_blocks=4096)
    case = synth.build_case(wl, "cuda", seed=31)
    S, Hq, D = case.q.shape
    max_ctx = case.max_context   # host bound, read before capturing
    ws = torch.empty(max(pkv.decode_workspace_bytes(S, Hq, D, max_ctx), 16),
                     dtype=torch.uint8, device="cuda")
    out_eager = torch.empty_like(case.q)
    out_graph = torch.empty_like(case.q)

    def step(out):
        pkv.kv_append(case.k_pool, case.v_pool, case.slot_mapping, case.k_new, case.v_new)
        pkv.paged_decode(case.q, case.k_pool, case.v_pool, case.block_tables, case.context_lens,
                         case.scale, max_context=max_ctx, out=out, workspace=ws)

    step(out_eager)
    torch.cuda.synchronize()
    assert pkv.read_device_status() == 0
    g = capture(lambda: step(out_graph))
    g.replay()
    torch.cuda.synchronize()
    assert torch.equal(out_eager, out_graph)
    # a replay reads the inputs as they are at replay time
    case.q.mul_(-0.5)
    step(out_eager)
    g.replay()
    torch.cuda.synchronize()
    assert pkv.read_device_status() == 0
    assert torch.equal(out_eager, out_graph)


def test_fused_decode_step_graph_replay(pkv):
    """The fused append + decode call captured and replayed: same output bits and the
    same pool as the eager call, also after the new rows change."""
    wl = dataclasses.replace(synth.WORKLOADS["8b"], num_seqs=16, num_blocks=4096)
    case = synth.build_case(wl, "cuda", seed=35)
    S, Hq, D = case.q.shape
    max_ctx = case.max_context   # host bound, read before capturing
    ws = torch.empty(max(pkv.decode_workspace_bytes(S, Hq, D, max_ctx), 16),
                     dtype=torch.uint8, device="cuda")
    out_eager = torch.empty_like(case.q)
    out_graph = torch.empty_like(case.q)

    def step(out):
        pkv.paged_decode_append(case.q, case.k_pool, case.v_pool, case.k_new, case.v_new,
                                case.block_tables, case.context_lens, case.scale,
                                max_context=max_ctx, out=out, workspace=ws)

    step(out_eager)
    torch.cuda.synchronize()
    assert pkv.read_device_status() == 0
    g = capture(lambda: step(out_graph))
    g.replay()
    torch.cuda.synchronize()
    assert torch.equal(out_eager, out_graph)
    case.k_new.mul_(2.0)
    case.v_new.mul_(-1.0)
    step(out_eager)
    torch.cuda.synchronize()
    slots = case.slot_mapping
    B = case.k_pool.shape[2]
    blk, off = slots // B, slots % B
    case.k_pool[blk, :, off] = 0   # the replay must store the new rows again
    g.replay()
    torch.cuda.synchronize()
    assert pkv.read_device_status() == 0
    assert torch.equal(out_eager, out_graph)
    assert torch.equal(case.k_pool[blk, :, off], case.k_new)


def test_cascade_graph_replay(pkv):
    wl = dataclasses.replace(synth.WORKLOADS["shared"], num_seqs=32, shared_prefix=512,
                             num_blocks=4096)
    case = synth.build_case(wl, "cuda", seed=33)
    S, Hq, D = case.q.shape
    max_ctx = case.max_context   # host bound, read before capturing
    prefix_blocks = case.block_tables[0, :512 // 16].contiguous()
    ws = torch.empty(max(pkv.cascade_workspace_bytes(S, Hq, D, 512, max_ctx), 16),
                     dtype=torch.uint8, device="cuda")
    out_eager = torch.empty_like(case.q)
    out_graph = torch.empty_like(case.q)
    pkv.kv_append(case.k_pool, case.v_pool, case.slot_mapping, case.k_new, case.v_new)

    def call(out):
        pkv.paged_decode_cascade(case.q, case.k_pool, case.v_pool, prefix_blocks, 512,
                                 case.block_tables, case.context_lens, case.scale,
                                 max_context=max_ctx, out=out, workspace=ws)

    call(out_eager)
    torch.cuda.synchronize()
    assert pkv.read_device_status() == 0
    g = capture(lambda: call(out_graph))
    for _ in range(3):
        g.replay()
    torch.cuda.synchronize()
    assert pkv.read_device_status() == 0
    assert torch.equal(out_eager, out_graph)


def test_fused_cascade_graph_replay(pkv):
    """The cascade decode with the append fused in, captured and replayed."""
    wl = dataclasses.replace(synth.WORKLOADS["shared"], num_seqs=32, shared_prefix=512,
                             num_blocks=4096)
    case = synth.build_case(wl, "cuda", seed=37)
    S, Hq, D = case.q.shape
    max_ctx = case.max_context   # host bound, read before capturing
    prefix_blocks = case.block_tables[0, :512 // 16].contiguous()
    ws = torch.empty(max(pkv.cascade_workspace_bytes(S, Hq, D, 512, max_ctx), 16),
                     dtype=torch.uint8, device="cuda")
    out_eager = torch.empty_like(case.q)
    out_graph = torch.empty_like(case.q)

    def call(out):
        pkv.paged_decode_cascade_append(case.q, case.k_pool, case.v_pool, case.k_new,
                                        case.v_new, prefix_blocks, 512, case.block_tables,
                                        case.context_lens, case.scale, max_context=max_ctx,
                                        out=out, workspace=ws)

    call(out_eager)
    torch.cuda.synchronize()
    assert pkv.read_device_status() == 0
    g = capture(lambda: call(out_graph))
    for _ in range(3):
        g.replay()
    torch.cuda.synchronize()
    assert pkv.read_device_status() == 0
    assert torch.equal(out_eager, out_graph)


def test_cascade_error_after_fork_leaves_capture_joined(pkv, monkeypatch):
    """A cascade call that fails after forking its prefix pass onto the library's side
    stream (PKV_TEST_CASCADE_SUFFIX_FAIL=1: the suffix launch reports a failure) still
    makes the caller's stream wait for the side stream before returning: under stream
    capture the capture ends cleanly (an unjoined side stream would make ending it fail),
    and outside capture the next calls on the stream are correct."""
    wl = dataclasses.replace(synth.WORKLOADS["shared"], num_seqs=4, shared_prefix=64,
                             num_blocks=256)
    case = synth.build_case(wl, "cuda", lengths=[5, 33, 1, 70], seed=41)
    pkv.kv_append(case.k_pool, case.v_pool, case.slot_mapping, case.k_new, case.v_new)
    prefix_blocks = case.block_tables[0, :4].contiguous()
    max_ctx = case.max_context

    def casc():
        return pkv.paged_decode_cascade(case.q, case.k_pool, case.v_pool, prefix_blocks, 64,
                                        case.block_tables, case.context_lens, case.scale,
                                        max_context=max_ctx)

    ref = casc()   # outside capture first: status word and side stream exist
    torch.cuda.synchronize()
    assert pkv.read_device_status() == 0
    monkeypatch.setenv("PKV_TEST_CASCADE_SUFFIX_FAIL", "1")
    s = torch.cuda.Stream()
    s.wait_stream(torch.cuda.current_stream())
    g = torch.cuda.CUDAGraph()
    with pytest.raises(pkv.PkvError) as e:
        with torch.cuda.graph(g, stream=s):
            casc()
    assert e.value.status == 3
    torch.cuda.current_stream().wait_stream(s)
    with pytest.raises(pkv.PkvError):
        casc()   # eager: fails the same way, joined before it returns
    monkeypatch.delenv("PKV_TEST_CASCADE_SUFFIX_FAIL")
    out = casc()
    torch.cuda.synchronize()
    assert pkv.read_device_status() == 0
    assert torch.equal(out.view(torch.int16), ref.view(torch.int16))


def test_host_steps_graph_replay(pkv):
    """The host-buffer decode step (kernels reading and writing pinned memory in place)
    and the host-buffer prefill step (chunked copies on the library's copy streams,
    joined back) captured and replayed: the eager calls' host output bits."""
    # decode step
    a = synth.build_case(dataclasses.replace(synth.WORKLOADS["8b"], num_seqs=16,
                                             num_blocks=4096), "cuda", seed=33)
    S, Hq, D = a.q.shape
    mbs = a.block_tables.shape[1]
    lay = pkv.decode_step_layout(a.k_pool, S, Hq, mbs)
    hin = torch.empty(lay.bytes, dtype=torch.uint8).pin_memory()
    pkv.pack_decode_step(hin, lay, a.q.cpu(), a.k_new.cpu(), a.v_new.cpu(),
                         a.block_tables.cpu(), a.context_lens.cpu())
    stg = torch.empty(pkv.decode_host_staging_bytes(a.k_pool, S, Hq, mbs, a.max_context),
                      dtype=torch.uint8, device="cuda")
    ref = torch.empty((S, Hq, D), dtype=a.q.dtype).pin_memory()
    got = torch.full((S, Hq, D), float("nan"), dtype=a.q.dtype).pin_memory()
    kw = dict(num_seqs=S, num_q_heads=Hq, max_blocks_per_seq=mbs, max_context=a.max_context,
              staging=stg)
    pkv.paged_decode_append_host(a.k_pool, a.v_pool, hin, ref, a.scale, **kw)
    torch.cuda.synchronize()
    assert pkv.read_device_status() == 0
    g = capture(lambda: pkv.paged_decode_append_host(a.k_pool, a.v_pool, hin, got, a.scale,
                                                     **kw))
    g.replay()
    torch.cuda.synchronize()
    assert torch.equal(got.view(torch.uint8), ref.view(torch.uint8))
    # prefill step
    b = synth.build_case(dataclasses.replace(synth.WORKLOADS["prefill"], num_seqs=6,
                                             num_blocks=8192), "cuda", seed=35)
    T, Hq, D = b.q.shape
    R = b.cached_lens.numel()
    mbs = b.block_tables.shape[1]
    play = pkv.prefill_step_layout(b.k_pool, R, T, Hq, mbs)
    phin = torch.empty(play.bytes, dtype=torch.uint8).pin_memory()
    pkv.pack_prefill_step(phin, play, b.q.cpu(), b.block_tables.cpu(), b.cached_lens.cpu(),
                          b.new_lens.cpu(), b.q_offsets.cpu(), b.k_new.cpu(), b.v_new.cpu(),
                          b.slot_mapping.cpu())
    pstg = torch.empty(pkv.prefill_host_staging_bytes(b.k_pool, R, T, Hq, mbs),
                       dtype=torch.uint8, device="cuda")
    pref = torch.empty((T, Hq, D), dtype=b.q.dtype).pin_memory()
    pgot = torch.full((T, Hq, D), float("nan"), dtype=b.q.dtype).pin_memory()
    pkw = dict(num_reqs=R, total_new=T, max_new=int(b.new_lens.max()), num_q_heads=Hq,
               max_blocks_per_seq=mbs, staging=pstg)
    pkv.paged_prefill_append_host(b.k_pool, b.v_pool, phin, pref, b.scale, **pkw)
    torch.cuda.synchronize()
    assert pkv.read_device_status() == 0
    g2 = capture(lambda: pkv.paged_prefill_append_host(b.k_pool, b.v_pool, phin, pgot, b.scale,
                                                       **pkw))
    g2.replay()
    torch.cuda.synchronize()
    assert pkv.read_device_status() == 0
    assert torch.equal(pgot.view(torch.uint8), pref.view(torch.uint8))

