"""CPU checks of the C ABI's argument errors: every device call validates its arguments
and returns a status before any CUDA call, so these run without a GPU.  The pointers are
fake (16-byte aligned or not, never dereferenced); a check that failed to fire would
reach the CUDA runtime and return PKV_ERR_CUDA instead of the status expected here."""
import ctypes

import pytest
import torch

# With a GPU present a check that failed to fire would launch a kernel on the fake
# pointers; these tests run only where no CUDA device exists.
pytestmark = pytest.mark.skipif(torch.cuda.is_available(),
                                reason="fake device pointers: host-only test")

OK, INVALID, UNSUPPORTED, NOMEM = 0, 1, 2, 6
A = 0x10000          # a 16-byte aligned fake device address
U = 0x10008          # a misaligned one


@pytest.fixture(scope="module")
def pkv():
    from paged_kv_cache_58_gb300 import build
    build.build()
    import paged_kv_cache_58_gb300 as m
    return m


def desc(pkv, nb=64, bs=16, hkv=8, d=128, dtype=1):
    return pkv.PoolDesc(nb, bs, hkv, d, dtype)


def decode(pkv, d, *, out=A, q=A, kp=A, vp=A, bt=A, mbs=8, cl=A, max_ctx=100, S=2, hq=32,
           scale=0.1, pb=0, ws=A, wsb=1 << 20):
    return pkv.lib().pkv_paged_decode(ctypes.byref(d), out, q, kp, vp, bt, mbs, cl, max_ctx, S,
                                      hq, scale, pb, ws, wsb, None)


def append_decode(pkv, d, *, kn=A, vn=A, S=2, max_ctx=100, hq=32, ws=A, wsb=1 << 20):
    mbs = max(8, -(-max_ctx // 16))
    return pkv.lib().pkv_paged_decode_append(ctypes.byref(d), A, A, A, A, kn, vn, A, mbs, A,
                                             max_ctx, S, hq, 0.1, 0, ws, wsb, None)


def test_pool_descriptor_checks(pkv):
    assert decode(pkv, desc(pkv, bs=8)) == UNSUPPORTED       # block size 16 or 32 only
    assert decode(pkv, desc(pkv, d=96)) == UNSUPPORTED       # head_dim 64 or 128 only
    assert decode(pkv, desc(pkv, dtype=7)) == UNSUPPORTED
    assert decode(pkv, desc(pkv, nb=0)) == INVALID
    assert decode(pkv, desc(pkv, hkv=0)) == INVALID


def test_decode_argument_checks(pkv):
    d = desc(pkv)
    assert decode(pkv, d, S=0) == OK                          # nothing to do, no launch
    assert decode(pkv, d, S=-1) == INVALID
    assert decode(pkv, d, q=None) == INVALID
    assert decode(pkv, d, bt=None) == INVALID
    assert decode(pkv, d, max_ctx=8 * 16 + 1) == INVALID      # beyond the table row
    assert decode(pkv, d, hq=20) == INVALID                   # not a multiple of Hkv
    assert decode(pkv, d, hq=24) == UNSUPPORTED               # GQA group 3
    assert decode(pkv, d, q=U) == INVALID                     # misaligned
    # 4096 tokens over 2 sequences: several partitions, so a workspace is needed
    assert decode(pkv, d, mbs=256, max_ctx=4096, wsb=16) == NOMEM     # too small
    assert decode(pkv, d, mbs=256, max_ctx=4096, ws=U) == NOMEM       # misaligned
    assert decode(pkv, d, mbs=256, max_ctx=4096, ws=None) == NOMEM    # missing
    assert decode(pkv, d, S=70000) == UNSUPPORTED


def test_fused_append_decode_argument_checks(pkv):
    d = desc(pkv)
    assert append_decode(pkv, d, S=0) == OK
    assert append_decode(pkv, d, kn=None) == INVALID
    assert append_decode(pkv, d, vn=None) == INVALID
    assert append_decode(pkv, d, kn=U) == INVALID
    assert append_decode(pkv, d, hq=24) == UNSUPPORTED
    assert append_decode(pkv, d, max_ctx=4096, wsb=16) == NOMEM


def test_kv_append_and_copy_blocks_checks(pkv):
    lib = pkv.lib()
    d = desc(pkv)
    assert lib.pkv_kv_append(ctypes.byref(d), A, A, A, A, A, 0, None) == OK
    assert lib.pkv_kv_append(ctypes.byref(d), A, A, A, A, A, -1, None) == INVALID
    assert lib.pkv_kv_append(ctypes.byref(d), A, A, None, A, A, 4, None) == INVALID
    assert lib.pkv_kv_append(ctypes.byref(d), A, A, A, U, A, 4, None) == INVALID
    assert lib.pkv_copy_blocks(ctypes.byref(d), A, A, A, 0, None) == OK


def test_prefill_and_cascade_checks(pkv):
    lib = pkv.lib()
    d = desc(pkv)
    pf = lib.pkv_paged_prefill
    assert pf(ctypes.byref(d), A, A, A, A, A, 8, A, A, A, 0, 0, 0, 32, 0.1, None) == OK
    assert pf(ctypes.byref(d), A, A, A, A, A, 8, A, A, A, 2, 10, 5, 32, 0.0, None) == INVALID
    assert pf(ctypes.byref(d), A, A, A, A, A, 8, A, None, A, 2, 10, 5, 32, 0.1, None) == INVALID
    assert pf(ctypes.byref(d), A, A, A, A, A, 8, A, A, A, 2, 10, 5, 24, 0.1, None) == UNSUPPORTED
    cas = lib.pkv_paged_decode_cascade
    args = dict(prefix=A, plen=64, mbs=8, max_ctx=100, S=2, hq=32, dt=d, ws=A, wsb=1 << 20)

    def c(**o):
        a = dict(args, **o)
        return cas(ctypes.byref(a["dt"]), A, A, A, A, a["prefix"], a["plen"], A, a["mbs"], A,
                   a["max_ctx"], a["S"], a["hq"], 0.1, 0, a["ws"], a["wsb"], None)

    ca = lib.pkv_paged_decode_cascade_append

    def cf(kn=A, vn=A, S=2):
        return ca(ctypes.byref(d), A, A, A, A, kn, vn, A, 64, A, 8, A, 100, S, 32, 0.1, 0, A,
                  1 << 20, None)

    assert cf(S=0) == OK
    assert cf(kn=None) == INVALID
    assert cf(vn=U) == INVALID
    assert c(S=0) == OK
    assert c(plen=40) == INVALID                              # not a multiple of the block
    assert c(plen=128, max_ctx=100) == INVALID                # prefix longer than the context
    assert c(prefix=None) == INVALID
    assert c(dt=desc(pkv, dtype=0)) == UNSUPPORTED            # bf16 only
    assert c(wsb=16) == NOMEM


def test_host_step_checks(pkv):
    lib = pkv.lib()
    d = desc(pkv)
    hs = lib.pkv_paged_decode_append_host

    def h(hin=A, hout=A, stg=0x100000, stgb=1 << 24, S=2):
        return hs(ctypes.byref(d), A, A, hin, hout, 8, 100, S, 32, 0.1, 0, stg, stgb, None)

    assert h(S=0) == OK
    assert h(hin=None) == INVALID
    assert h(hout=None) == INVALID
    assert h(stg=0x100010) == INVALID     # staging must be 256-byte aligned
    assert h(stgb=64) == NOMEM


def test_prefill_host_step_checks(pkv):
    """Argument errors of the host-buffer prefill step are returned before any CUDA call:
    sizes, null buffers, staging alignment and size, and q_offsets read from host_in that
    are not the prefix sum ending at total_new."""
    import numpy as np
    lib = pkv.lib()
    d = desc(pkv)
    R, T, Hq, mbs = 2, 10, 32, 4
    lay = pkv.PrefillLayout()
    assert lib.pkv_prefill_step_layout(ctypes.byref(d), R, T, Hq, mbs, ctypes.byref(lay)) == OK
    host = np.zeros(lay.bytes, dtype=np.uint8)
    qo = host[lay.q_offsets:lay.q_offsets + 4 * (R + 1)].view(np.int32)
    need = lib.pkv_paged_prefill_append_host_staging_bytes(ctypes.byref(d), R, T, Hq, mbs)
    ps = lib.pkv_paged_prefill_append_host

    def h(hin=None, hout=A, stg=0x100000, stgb=None, R=R, T=T):
        hin = host.ctypes.data if hin is None else hin
        return ps(ctypes.byref(d), A, A, hin, hout, R, T, 8, Hq, mbs, 0.1, stg,
                  need if stgb is None else stgb, None)

    qo[:] = [0, 4, 11]                     # ends past total_new
    assert h() == INVALID
    qo[:] = [0, 6, 4]                      # decreasing
    assert h() == INVALID
    qo[:] = [1, 4, 10]                     # does not start at 0
    assert h() == INVALID
    assert h(R=0) == OK and h(T=0) == OK
    assert h(hout=None) == INVALID
    assert h(stg=0x100010) == INVALID      # staging must be 256-byte aligned
    assert h(stgb=64) == NOMEM
    assert lib.pkv_prefill_step_layout(ctypes.byref(d), R, -1, Hq, mbs, ctypes.byref(lay)) == INVALID

