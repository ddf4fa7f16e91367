"""The bounded pipeline wait on a GPU: a wait that runs out of time reports
PKV_ERR_TIMEOUT through the device status word and leaves the context usable.

The test hook PKV_TEST_DECODE_STALL=1 makes one warp of one CTA of the decode
kernel (tensor-core or CUDA-core) arm its first stage's barrier for 16 bytes more
than that stage's copies deliver.  All copies land; the barrier phase never completes, so that warp's wait
expires after its time budget (2 s), raises the status, drains its other stage and
finishes.  Nothing faults, traps or loops without a limit."""
import dataclasses

import pytest
import torch

import synth
from tests.helpers import check_attention, oracle_decode_case

pytestmark = pytest.mark.gpu

PKV_ERR_TIMEOUT = 4


@pytest.fixture(scope="module")
def pkv():
    if not torch.cuda.is_available():
        pytest.skip("no CUDA device")
    import paged_kv_cache_58_gb300 as m
    from paged_kv_cache_58_gb300 import build
    build.build()
    return m


@pytest.mark.parametrize("kernel", ["tc", "simt"])
def test_decode_wait_timeout_reports_status(pkv, oracle_mod, monkeypatch, kernel):
    """Both decode kernels: the tensor-core one (TMA boxes, converged-warp waits) and the
    CUDA-core one (bulk copies, per-lane waits)."""
    if kernel == "simt":
        monkeypatch.setenv("PKV_DECODE_KERNEL", "simt")
    else:
        monkeypatch.delenv("PKV_DECODE_KERNEL", raising=False)
    wl = dataclasses.replace(synth.WORKLOADS["8b"], num_blocks=256)
    case = synth.build_case(wl, "cuda", lengths=[100, 37, 300], seed=3)
    pkv.kv_append(case.k_pool, case.v_pool, case.slot_mapping, case.k_new, case.v_new)
    torch.cuda.synchronize()
    assert pkv.read_device_status() == 0

    def decode():
        return pkv.paged_decode(case.q, case.k_pool, case.v_pool, case.block_tables,
                                case.context_lens, case.scale, max_context=case.max_context)

    monkeypatch.setenv("PKV_TEST_DECODE_STALL", "1")
    decode()
    torch.cuda.synchronize()
    assert pkv.read_device_status() == PKV_ERR_TIMEOUT
    # reading the status cleared it; the context still runs kernels correctly
    monkeypatch.delenv("PKV_TEST_DECODE_STALL")
    out = decode()
    torch.cuda.synchronize()
    assert pkv.read_device_status() == 0
    ref, _, _ = oracle_decode_case(oracle_mod, case)
    check_attention(out, ref)


def test_prefill_wait_timeout_reports_status(pkv, oracle_mod, monkeypatch):
    """The same for the tcgen05 prefill: PKV_TEST_PREFILL_STALL=1 arms CTA 0's first Q
    barrier for 16 bytes more than the Q copy delivers.  The copy lands, the issuers'
    wait for the barrier expires and raises the status, the CTA's other roles see the
    abort and drain (bounded), and the next call, with the hook off, is correct."""
    from tests.helpers import oracle_prefill_case
    from tests.test_gpu_prefill import custom_case, run_prefill

    case = custom_case(32, 8, [100, 40], [37, 64], seed=5, num_blocks=64)
    pkv.kv_append(case.k_pool, case.v_pool, case.slot_mapping, case.k_new, case.v_new)
    torch.cuda.synchronize()
    assert pkv.read_device_status() == 0

    monkeypatch.setenv("PKV_TEST_PREFILL_STALL", "1")
    pkv.paged_prefill(case.q, case.k_pool, case.v_pool, case.block_tables, case.cached_lens,
                      case.new_lens, case.q_offsets, case.scale,
                      max_new=int(case.new_lens.max()))
    torch.cuda.synchronize()
    assert pkv.read_device_status() == PKV_ERR_TIMEOUT

    monkeypatch.delenv("PKV_TEST_PREFILL_STALL")
    ref, _, _ = oracle_prefill_case(oracle_mod, case)
    check_attention(run_prefill(pkv, case), ref)   # asserts a clean status; short rows
