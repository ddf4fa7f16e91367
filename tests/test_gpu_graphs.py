"""Stream capture: a decode step (kv_append + paged_decode, or the fused call) and a
cascade decode can be recorded into a CUDA graph and replayed -- the calls allocate
nothing, read nothing back to the host and never synchronise -- and a replay gives the
same bits as the eager calls.
The cascade's fork onto the library's side stream becomes part of the graph."""
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
