"""Python binding of libpkv (paged KV-cache attention on GB300 / sm_103a).

Argument marshalling only: every step of the path runs in libpkv's CUDA kernels
(see ``include/pkv.h`` for the contracts).  PyTorch provides device memory and
the current stream.  There is no fallback: if ``libpkv.so`` is missing or a
call fails, an exception is raised.
"""
from __future__ import annotations

import ctypes
import os

import numpy as np
import torch

_HERE = os.path.dirname(os.path.abspath(__file__))
LIB_PATH = os.path.join(_HERE, "libpkv.so")

PKV_F32 = 0
PKV_BF16 = 1
BLOCK_SIZE = 16

_STATUS = {0: "ok", 1: "invalid argument", 2: "unsupported configuration", 3: "CUDA error",
           4: "device pipeline wait timed out", 5: "slot or block id outside the pool",
           6: "out of blocks or workspace too small", 7: "unknown or duplicate sequence id"}


class PkvError(RuntimeError):
    def __init__(self, fn: str, status: int):
        super().__init__(f"{fn}: {_STATUS.get(status, 'unknown status')} ({status})")
        self.status = status


class PoolDesc(ctypes.Structure):
    _fields_ = [("num_blocks", ctypes.c_int64), ("block_size", ctypes.c_int32),
                ("num_kv_heads", ctypes.c_int32), ("head_dim", ctypes.c_int32),
                ("dtype", ctypes.c_int32)]


class PrefillLayout(ctypes.Structure):
    """Byte offsets of one prefill step's inputs in a packed host buffer: the part copied
    to the device (q and the control arrays, `copied_bytes`), then the new rows."""
    _fields_ = [("q", ctypes.c_uint64), ("block_tables", ctypes.c_uint64),
                ("cached_lens", ctypes.c_uint64), ("new_lens", ctypes.c_uint64),
                ("q_offsets", ctypes.c_uint64), ("copied_bytes", ctypes.c_uint64),
                ("k_new", ctypes.c_uint64), ("v_new", ctypes.c_uint64),
                ("slot_mapping", ctypes.c_uint64), ("bytes", ctypes.c_uint64)]


class StepLayout(ctypes.Structure):
    """Byte offsets of one decode step's inputs in a packed host buffer (and its size)."""
    _fields_ = [("q", ctypes.c_uint64), ("k_new", ctypes.c_uint64), ("v_new", ctypes.c_uint64),
                ("block_tables", ctypes.c_uint64), ("context_lens", ctypes.c_uint64),
                ("bytes", ctypes.c_uint64)]


_lib = None


def _load():
    global _lib
    if _lib is not None:
        return _lib
    if not os.path.exists(LIB_PATH):
        raise ImportError(f"libpkv.so is not built ({LIB_PATH}); run "
                          "paged_kv_cache_58_gb300.build.build() first")
    lib = ctypes.CDLL(LIB_PATH)
    vp, i32, i64, f32, sz = ctypes.c_void_p, ctypes.c_int32, ctypes.c_int64, ctypes.c_float, \
        ctypes.c_size_t
    P = ctypes.POINTER
    lib.pkv_status_string.restype = ctypes.c_char_p
    lib.pkv_status_string.argtypes = [ctypes.c_int]
    lib.pkv_version.restype = ctypes.c_int
    lib.pkv_pool_bytes.restype = ctypes.c_uint64
    lib.pkv_pool_bytes.argtypes = [P(PoolDesc)]
    lib.pkv_kv_append.restype = ctypes.c_int
    lib.pkv_kv_append.argtypes = [P(PoolDesc), vp, vp, vp, vp, vp, i64, vp]
    lib.pkv_paged_decode_workspace_bytes.restype = sz
    lib.pkv_paged_decode_workspace_bytes.argtypes = [ctypes.c_int] * 6
    lib.pkv_paged_decode_auto_partition.restype = ctypes.c_int
    lib.pkv_paged_decode_auto_partition.argtypes = [ctypes.c_int] * 4
    lib.pkv_paged_decode.restype = ctypes.c_int
    lib.pkv_paged_decode.argtypes = [P(PoolDesc), vp, vp, vp, vp, vp, ctypes.c_int, vp,
                                     ctypes.c_int, ctypes.c_int, ctypes.c_int, f32, ctypes.c_int,
                                     vp, sz, vp]
    lib.pkv_paged_decode_append.restype = ctypes.c_int
    lib.pkv_paged_decode_append.argtypes = [P(PoolDesc), vp, vp, vp, vp, vp, vp, vp,
                                            ctypes.c_int, vp, ctypes.c_int, ctypes.c_int,
                                            ctypes.c_int, f32, ctypes.c_int, vp, sz, vp]
    lib.pkv_paged_decode_cascade_append.restype = ctypes.c_int
    lib.pkv_paged_decode_cascade_append.argtypes = [P(PoolDesc), vp, vp, vp, vp, vp, vp, vp,
                                                    ctypes.c_int, vp, ctypes.c_int, vp,
                                                    ctypes.c_int, ctypes.c_int, ctypes.c_int,
                                                    f32, ctypes.c_int, vp, sz, vp]
    lib.pkv_decode_step_layout.restype = ctypes.c_int
    lib.pkv_decode_step_layout.argtypes = [P(PoolDesc), ctypes.c_int, ctypes.c_int, ctypes.c_int,
                                           P(StepLayout)]
    lib.pkv_paged_decode_append_host_staging_bytes.restype = sz
    lib.pkv_paged_decode_append_host_staging_bytes.argtypes = [P(PoolDesc)] + [ctypes.c_int] * 5
    lib.pkv_prefill_step_layout.restype = ctypes.c_int
    lib.pkv_prefill_step_layout.argtypes = [P(PoolDesc)] + [ctypes.c_int] * 4 + [P(PrefillLayout)]
    lib.pkv_paged_prefill_append_host_staging_bytes.restype = sz
    lib.pkv_paged_prefill_append_host_staging_bytes.argtypes = [P(PoolDesc)] + [ctypes.c_int] * 4
    lib.pkv_paged_prefill_append_host.restype = ctypes.c_int
    lib.pkv_paged_prefill_append_host.argtypes = [P(PoolDesc), vp, vp, vp, vp] + \
        [ctypes.c_int] * 5 + [f32, vp, sz, vp]
    lib.pkv_paged_decode_append_host.restype = ctypes.c_int
    lib.pkv_paged_decode_append_host.argtypes = [P(PoolDesc), vp, vp, vp, vp, ctypes.c_int,
                                                 ctypes.c_int, ctypes.c_int, ctypes.c_int, f32,
                                                 ctypes.c_int, vp, sz, vp]
    lib.pkv_paged_prefill.restype = ctypes.c_int
    lib.pkv_paged_prefill.argtypes = [P(PoolDesc), vp, vp, vp, vp, vp, ctypes.c_int, vp, vp, vp,
                                      ctypes.c_int, ctypes.c_int, ctypes.c_int, ctypes.c_int, f32,
                                      vp]
    lib.pkv_copy_blocks.restype = ctypes.c_int
    lib.pkv_copy_blocks.argtypes = [P(PoolDesc), vp, vp, vp, ctypes.c_int, vp]
    lib.pkv_read_device_status.restype = ctypes.c_int
    lib.pkv_read_device_status.argtypes = [P(ctypes.c_int), vp]
    lib.pkv_alloc_create.restype = vp
    lib.pkv_alloc_create.argtypes = [i64, ctypes.c_int, ctypes.c_uint64]
    lib.pkv_alloc_destroy.restype = None
    lib.pkv_alloc_destroy.argtypes = [vp]
    lib.pkv_alloc_add_seq.restype = ctypes.c_int
    lib.pkv_alloc_add_seq.argtypes = [vp, i64, i64]
    lib.pkv_alloc_fork.restype = ctypes.c_int
    lib.pkv_alloc_fork.argtypes = [vp, i64, i64]
    lib.pkv_alloc_append.restype = ctypes.c_int
    lib.pkv_alloc_append.argtypes = [vp, i64, i64, P(i64), P(i32), P(ctypes.c_int)]
    lib.pkv_alloc_free_seq.restype = ctypes.c_int
    lib.pkv_alloc_free_seq.argtypes = [vp, i64]
    lib.pkv_alloc_block_table.restype = ctypes.c_int
    lib.pkv_alloc_block_table.argtypes = [vp, P(i64), ctypes.c_int, P(i32), ctypes.c_int]
    lib.pkv_alloc_num_free.restype = i64
    lib.pkv_alloc_num_free.argtypes = [vp]
    lib.pkv_alloc_refcount.restype = ctypes.c_int
    lib.pkv_alloc_refcount.argtypes = [vp, i64]
    lib.pkv_alloc_seq_len.restype = i64
    lib.pkv_alloc_seq_len.argtypes = [vp, i64]
    lib.pkv_alloc_seq_num_blocks.restype = i64
    lib.pkv_alloc_seq_num_blocks.argtypes = [vp, i64]
    lib.pkv_alloc_add_seq_shared.restype = ctypes.c_int
    lib.pkv_alloc_add_seq_shared.argtypes = [vp, i64, P(i32), ctypes.c_int, i64]
    lib.pkv_paged_decode_cascade_workspace_bytes.restype = sz
    lib.pkv_paged_decode_cascade_workspace_bytes.argtypes = [ctypes.c_int] * 7
    lib.pkv_paged_decode_cascade.restype = ctypes.c_int
    lib.pkv_paged_decode_cascade.argtypes = [P(PoolDesc), vp, vp, vp, vp, vp, ctypes.c_int, vp,
                                             ctypes.c_int, vp, ctypes.c_int, ctypes.c_int,
                                             ctypes.c_int, f32, ctypes.c_int, vp, sz, vp]
    u64 = ctypes.c_uint64
    lib.pkv_block_hash.restype = u64
    lib.pkv_block_hash.argtypes = [u64, u64, P(i32), ctypes.c_int, u64]
    lib.pkv_pcache_create.restype = vp
    lib.pkv_pcache_create.argtypes = [vp]
    lib.pkv_pcache_destroy.restype = None
    lib.pkv_pcache_destroy.argtypes = [vp]
    lib.pkv_pcache_match.restype = ctypes.c_int
    lib.pkv_pcache_match.argtypes = [vp, P(i32), i64, u64, P(i32), ctypes.c_int]
    lib.pkv_pcache_insert.restype = ctypes.c_int
    lib.pkv_pcache_insert.argtypes = [vp, i64, P(i32), i64, u64]
    lib.pkv_pcache_evict.restype = i64
    lib.pkv_pcache_evict.argtypes = [vp, i64]
    lib.pkv_pcache_size.restype = i64
    lib.pkv_pcache_size.argtypes = [vp]
    lib.pkv_radix_create.restype = vp
    lib.pkv_radix_create.argtypes = [vp]
    lib.pkv_radix_destroy.restype = None
    lib.pkv_radix_destroy.argtypes = [vp]
    lib.pkv_radix_match.restype = i64
    lib.pkv_radix_match.argtypes = [vp, P(i32), i64, P(i32), ctypes.c_int]
    lib.pkv_radix_insert.restype = ctypes.c_int
    lib.pkv_radix_insert.argtypes = [vp, i64, P(i32), i64]
    lib.pkv_radix_lock.restype = ctypes.c_int
    lib.pkv_radix_lock.argtypes = [vp, P(i32), i64, ctypes.c_int]
    lib.pkv_radix_evict.restype = i64
    lib.pkv_radix_evict.argtypes = [vp, i64]
    lib.pkv_radix_num_nodes.restype = i64
    lib.pkv_radix_num_nodes.argtypes = [vp]
    lib.pkv_radix_cached_tokens.restype = i64
    lib.pkv_radix_cached_tokens.argtypes = [vp]
    _lib = lib
    return lib


def lib():
    """The loaded libpkv handle (ctypes.CDLL)."""
    return _load()


def _check(fn: str, st: int) -> None:
    if st != 0:
        raise PkvError(fn, st)


def _dtype_code(t: torch.Tensor) -> int:
    if t.dtype == torch.bfloat16:
        return PKV_BF16
    if t.dtype == torch.float32:
        return PKV_F32
    raise TypeError(f"unsupported dtype {t.dtype}")


_POOL_DESCS: dict = {}


def pool_desc(k_pool: torch.Tensor) -> PoolDesc:
    """The pool descriptor of a [num_blocks, Hkv, B, D] pool (cached per shape and dtype:
    it holds sizes only)."""
    key = (tuple(k_pool.shape), k_pool.dtype)
    d = _POOL_DESCS.get(key)
    if d is None:
        nb, hkv, bs, dim = key[0]
        d = PoolDesc(nb, bs, hkv, dim, _dtype_code(k_pool))
        if len(_POOL_DESCS) > 64:
            _POOL_DESCS.clear()
        _POOL_DESCS[key] = d
    return d


def _dev(t: torch.Tensor, name: str, dtype=None) -> int:
    if not t.is_cuda:
        raise ValueError(f"{name} must be a CUDA tensor")
    if not t.is_contiguous():
        raise ValueError(f"{name} must be contiguous")
    if dtype is not None and t.dtype != dtype:
        raise TypeError(f"{name} must be {dtype}, got {t.dtype}")
    return t.data_ptr()


def _stream(stream) -> int:
    if stream is None:
        return torch.cuda.current_stream().cuda_stream
    if isinstance(stream, torch.cuda.Stream):
        return stream.cuda_stream
    return int(stream)


def pool_bytes(num_blocks: int, num_kv_heads: int, head_dim: int, dtype=torch.bfloat16,
               block_size: int = BLOCK_SIZE) -> int:
    """Bytes of one (K or V) pool of this shape, as computed by libpkv."""
    d = PoolDesc(num_blocks, block_size, num_kv_heads, head_dim, _dtype_code(torch.empty(0,
                                                                                       dtype=dtype)))
    return int(_load().pkv_pool_bytes(ctypes.byref(d)))


def kv_append(k_pool, v_pool, slot_mapping, k, v, stream=None) -> None:
    """Scatter k/v [T, Hkv, D] into their pool slots (slot < 0 = skip)."""
    d = pool_desc(k_pool)
    T = k.shape[0]
    st = _load().pkv_kv_append(ctypes.byref(d), _dev(k_pool, "k_pool"),
                               _dev(v_pool, "v_pool", k_pool.dtype),
                               _dev(slot_mapping, "slot_mapping", torch.int64),
                               _dev(k, "k", k_pool.dtype), _dev(v, "v", k_pool.dtype), T,
                               _stream(stream))
    _check("pkv_kv_append", st)


def decode_workspace_bytes(num_seqs, num_q_heads, head_dim, max_context, partition_blocks=0,
                           block_size=BLOCK_SIZE):
    return int(_load().pkv_paged_decode_workspace_bytes(num_seqs, num_q_heads, head_dim,
                                                        max_context, block_size,
                                                        partition_blocks))


def auto_partition(num_seqs, num_q_heads, max_context, block_size=BLOCK_SIZE) -> int:
    """Partition size (in pool blocks) paged_decode picks when partition_blocks == 0."""
    return int(_load().pkv_paged_decode_auto_partition(num_seqs, num_q_heads, max_context,
                                                       block_size))


def paged_decode(q, k_pool, v_pool, block_tables, context_lens, scale, *, max_context,
                 out=None, partition_blocks=0, workspace=None, stream=None):
    """Decode attention: q [S, Hq, D] over the paged pools; returns out [S, Hq, D].

    `max_context` is the host-side upper bound of context_lens (no device sync).
    `workspace` (uint8 CUDA tensor) is allocated here when not given.
    """
    d = pool_desc(k_pool)
    S, Hq, D = q.shape
    if out is None:
        out = torch.empty_like(q)
    if workspace is None:   # the library checks a given workspace's size itself
        need = decode_workspace_bytes(S, Hq, D, max_context, partition_blocks, d.block_size)
        if need > 0:
            workspace = torch.empty(need, dtype=torch.uint8, device=q.device)
    wptr = workspace.data_ptr() if workspace is not None else None
    wbytes = workspace.numel() * workspace.element_size() if workspace is not None else 0
    st = _load().pkv_paged_decode(ctypes.byref(d), _dev(out, "out", q.dtype),
                                  _dev(q, "q", k_pool.dtype), _dev(k_pool, "k_pool"),
                                  _dev(v_pool, "v_pool", k_pool.dtype),
                                  _dev(block_tables, "block_tables", torch.int32),
                                  block_tables.shape[1],
                                  _dev(context_lens, "context_lens", torch.int32),
                                  int(max_context), S, Hq, float(scale), int(partition_blocks),
                                  wptr, wbytes, _stream(stream))
    _check("pkv_paged_decode", st)
    return out


def paged_decode_append(q, k_pool, v_pool, k_new, v_new, block_tables, context_lens, scale, *,
                        max_context, out=None, partition_blocks=0, workspace=None, stream=None):
    """kv_append + paged_decode in one pass: k_new / v_new [S, Hkv, D] are the K / V of
    each sequence's token context_lens[s] - 1, stored into the slot the block table gives
    for that position and attended; returns out [S, Hq, D]."""
    d = pool_desc(k_pool)
    S, Hq, D = q.shape
    if out is None:
        out = torch.empty_like(q)
    if workspace is None:   # the library checks a given workspace's size itself
        need = decode_workspace_bytes(S, Hq, D, max_context, partition_blocks, d.block_size)
        if need > 0:
            workspace = torch.empty(need, dtype=torch.uint8, device=q.device)
    wptr = workspace.data_ptr() if workspace is not None else None
    wbytes = workspace.numel() * workspace.element_size() if workspace is not None else 0
    if tuple(k_new.shape) != (S, d.num_kv_heads, D) or tuple(v_new.shape) != tuple(k_new.shape):
        raise ValueError("k_new / v_new must be [num_seqs, num_kv_heads, head_dim]")
    st = _load().pkv_paged_decode_append(
        ctypes.byref(d), _dev(out, "out", q.dtype), _dev(q, "q", k_pool.dtype),
        _dev(k_pool, "k_pool"), _dev(v_pool, "v_pool", k_pool.dtype),
        _dev(k_new, "k_new", k_pool.dtype), _dev(v_new, "v_new", k_pool.dtype),
        _dev(block_tables, "block_tables", torch.int32), block_tables.shape[1],
        _dev(context_lens, "context_lens", torch.int32), int(max_context), S, Hq, float(scale),
        int(partition_blocks), wptr, wbytes, _stream(stream))
    _check("pkv_paged_decode_append", st)
    return out


def decode_step_layout(k_pool, num_seqs, num_q_heads, max_blocks_per_seq) -> StepLayout:
    """Packed host-buffer layout of one decode step's inputs (pkv_decode_step_layout)."""
    lay = StepLayout()
    _check("pkv_decode_step_layout",
           _load().pkv_decode_step_layout(ctypes.byref(pool_desc(k_pool)), num_seqs, num_q_heads,
                                          max_blocks_per_seq, ctypes.byref(lay)))
    return lay


def pack_decode_step(host_in, layout, q, k_new, v_new, block_tables, context_lens):
    """Write one step's inputs (CPU tensors) into the packed host buffer `host_in` (uint8)."""
    for off, t in ((layout.q, q), (layout.k_new, k_new), (layout.v_new, v_new),
                   (layout.block_tables, block_tables), (layout.context_lens, context_lens)):
        b = t.contiguous().view(torch.uint8).reshape(-1)
        host_in[off:off + b.numel()].copy_(b)


def decode_host_staging_bytes(k_pool, num_seqs, num_q_heads, max_blocks_per_seq, max_context,
                              partition_blocks=0):
    return int(_load().pkv_paged_decode_append_host_staging_bytes(
        ctypes.byref(pool_desc(k_pool)), num_seqs, num_q_heads, max_blocks_per_seq, max_context,
        partition_blocks))


def paged_decode_append_host(k_pool, v_pool, host_in, host_out, scale, *, num_seqs, num_q_heads,
                             max_blocks_per_seq, max_context, staging, partition_blocks=0,
                             stream=None):
    """One decode step from host memory: host_in (uint8, packed as decode_step_layout)
    -> fused append + decode -> host_out ([S, Hq, D]).  Pinned buffers are read and
    written by the kernels in place; pageable ones go through `staging` with one copy
    each way.  Queued on the stream; host_out is complete after a synchronise."""
    if host_in.is_cuda or host_out.is_cuda:
        raise ValueError("host_in and host_out must be host tensors")
    st = _load().pkv_paged_decode_append_host(
        ctypes.byref(pool_desc(k_pool)), _dev(k_pool, "k_pool"), _dev(v_pool, "v_pool",
                                                                       k_pool.dtype),
        host_in.data_ptr(), host_out.data_ptr(), int(max_blocks_per_seq), int(max_context),
        int(num_seqs), int(num_q_heads), float(scale), int(partition_blocks),
        _dev(staging, "staging"), staging.numel() * staging.element_size(), _stream(stream))
    _check("pkv_paged_decode_append_host", st)
    return host_out


class HostDecodeStep:
    """paged_decode_append_host with every argument bound once, for a loop that runs
    the same step shape over the same buffers (refilling host_in between calls): each
    call is then one ctypes call on pre-converted arguments, about 3 us less host time
    than the keyword form.  The stream is bound too (stream=None: the current stream
    at construction).  The tensors are held for the object's lifetime."""

    def __init__(self, k_pool, v_pool, host_in, host_out, scale, *, num_seqs, num_q_heads,
                 max_blocks_per_seq, max_context, staging, partition_blocks=0, stream=None):
        if host_in.is_cuda or host_out.is_cuda:
            raise ValueError("host_in and host_out must be host tensors")
        self._keep = (k_pool, v_pool, host_in, host_out, staging)
        self._desc = pool_desc(k_pool)
        vp = ctypes.c_void_p
        self._fn = _load().pkv_paged_decode_append_host
        self._args = (ctypes.byref(self._desc), vp(_dev(k_pool, "k_pool")),
                      vp(_dev(v_pool, "v_pool", k_pool.dtype)), vp(host_in.data_ptr()),
                      vp(host_out.data_ptr()), ctypes.c_int(int(max_blocks_per_seq)),
                      ctypes.c_int(int(max_context)), ctypes.c_int(int(num_seqs)),
                      ctypes.c_int(int(num_q_heads)), ctypes.c_float(float(scale)),
                      ctypes.c_int(int(partition_blocks)), vp(_dev(staging, "staging")),
                      ctypes.c_size_t(staging.numel() * staging.element_size()),
                      vp(_stream(stream)))
        self.host_out = host_out

    def __call__(self):
        st = self._fn(*self._args)
        if st != 0:
            raise PkvError("pkv_paged_decode_append_host", st)
        return self.host_out


def prefill_step_layout(k_pool, num_reqs, total_new, num_q_heads,
                        max_blocks_per_seq) -> PrefillLayout:
    """Packed host-buffer layout of one prefill step's inputs (pkv_prefill_step_layout)."""
    lay = PrefillLayout()
    _check("pkv_prefill_step_layout",
           _load().pkv_prefill_step_layout(ctypes.byref(pool_desc(k_pool)), num_reqs, total_new,
                                           num_q_heads, max_blocks_per_seq, ctypes.byref(lay)))
    return lay


def pack_prefill_step(host_in, layout, q, block_tables, cached_lens, new_lens, q_offsets,
                      k_new, v_new, slot_mapping):
    """Write one prefill step's inputs (CPU tensors) into the packed host buffer
    `host_in` (uint8)."""
    for off, t in ((layout.q, q), (layout.block_tables, block_tables),
                   (layout.cached_lens, cached_lens), (layout.new_lens, new_lens),
                   (layout.q_offsets, q_offsets), (layout.k_new, k_new),
                   (layout.v_new, v_new), (layout.slot_mapping, slot_mapping)):
        b = t.contiguous().view(torch.uint8).reshape(-1)
        host_in[off:off + b.numel()].copy_(b)


def prefill_host_staging_bytes(k_pool, num_reqs, total_new, num_q_heads, max_blocks_per_seq):
    return int(_load().pkv_paged_prefill_append_host_staging_bytes(
        ctypes.byref(pool_desc(k_pool)), num_reqs, total_new, num_q_heads, max_blocks_per_seq))


def paged_prefill_append_host(k_pool, v_pool, host_in, host_out, scale, *, num_reqs, total_new,
                              max_new, num_q_heads, max_blocks_per_seq, staging, stream=None):
    """One prefill step from host memory: host_in (uint8, packed as prefill_step_layout)
    -> kv_append of the new rows + paged_prefill -> host_out ([total_new, Hq, D]),
    through `staging`, with the copies pipelined against the kernels over request chunks.
    Queued on the stream; host_out is complete after a synchronise."""
    if host_in.is_cuda or host_out.is_cuda:
        raise ValueError("host_in and host_out must be host tensors")
    st = _load().pkv_paged_prefill_append_host(
        ctypes.byref(pool_desc(k_pool)), _dev(k_pool, "k_pool"),
        _dev(v_pool, "v_pool", k_pool.dtype), host_in.data_ptr(), host_out.data_ptr(),
        int(num_reqs), int(total_new), int(max_new), int(num_q_heads), int(max_blocks_per_seq),
        float(scale), _dev(staging, "staging"), staging.numel() * staging.element_size(),
        _stream(stream))
    _check("pkv_paged_prefill_append_host", st)
    return host_out


def cascade_workspace_bytes(num_seqs, num_q_heads, head_dim, prefix_len, max_context,
                            partition_blocks=0, block_size=BLOCK_SIZE):
    return int(_load().pkv_paged_decode_cascade_workspace_bytes(
        num_seqs, num_q_heads, head_dim, prefix_len, max_context, block_size, partition_blocks))


def paged_decode_cascade(q, k_pool, v_pool, prefix_blocks, prefix_len, block_tables,
                         context_lens, scale, *, max_context, out=None, partition_blocks=0,
                         workspace=None, stream=None):
    """Decode of sequences sharing their first `prefix_len` tokens in `prefix_blocks`
    (int32 [prefix_len / block_size] CUDA tensor); same result as paged_decode."""
    d = pool_desc(k_pool)
    S, Hq, D = q.shape
    if out is None:
        out = torch.empty_like(q)
    need = cascade_workspace_bytes(S, Hq, D, prefix_len, max_context, partition_blocks,
                                   d.block_size)
    if workspace is None:
        workspace = torch.empty(max(need, 16), dtype=torch.uint8, device=q.device)
    st = _load().pkv_paged_decode_cascade(
        ctypes.byref(d), _dev(out, "out", q.dtype), _dev(q, "q", k_pool.dtype),
        _dev(k_pool, "k_pool"), _dev(v_pool, "v_pool", k_pool.dtype),
        _dev(prefix_blocks, "prefix_blocks", torch.int32), int(prefix_len),
        _dev(block_tables, "block_tables", torch.int32), block_tables.shape[1],
        _dev(context_lens, "context_lens", torch.int32), int(max_context), S, Hq, float(scale),
        int(partition_blocks), workspace.data_ptr(), workspace.numel(), _stream(stream))
    _check("pkv_paged_decode_cascade", st)
    return out


def paged_decode_cascade_append(q, k_pool, v_pool, k_new, v_new, prefix_blocks, prefix_len,
                                block_tables, context_lens, scale, *, max_context, out=None,
                                partition_blocks=0, workspace=None, stream=None):
    """Cascade decode with the append fused in: k_new / v_new [S, Hkv, D] are the K / V
    of each sequence's token context_lens[s] - 1 (in its private suffix)."""
    d = pool_desc(k_pool)
    S, Hq, D = q.shape
    if out is None:
        out = torch.empty_like(q)
    if workspace is None:
        need = cascade_workspace_bytes(S, Hq, D, prefix_len, max_context, partition_blocks,
                                       d.block_size)
        workspace = torch.empty(max(need, 16), dtype=torch.uint8, device=q.device)
    if tuple(k_new.shape) != (S, d.num_kv_heads, D) or tuple(v_new.shape) != tuple(k_new.shape):
        raise ValueError("k_new / v_new must be [num_seqs, num_kv_heads, head_dim]")
    st = _load().pkv_paged_decode_cascade_append(
        ctypes.byref(d), _dev(out, "out", q.dtype), _dev(q, "q", k_pool.dtype),
        _dev(k_pool, "k_pool"), _dev(v_pool, "v_pool", k_pool.dtype),
        _dev(k_new, "k_new", k_pool.dtype), _dev(v_new, "v_new", k_pool.dtype),
        _dev(prefix_blocks, "prefix_blocks", torch.int32), int(prefix_len),
        _dev(block_tables, "block_tables", torch.int32), block_tables.shape[1],
        _dev(context_lens, "context_lens", torch.int32), int(max_context), S, Hq, float(scale),
        int(partition_blocks), workspace.data_ptr(), workspace.numel(), _stream(stream))
    _check("pkv_paged_decode_cascade_append", st)
    return out


def paged_prefill(q, k_pool, v_pool, block_tables, cached_lens, new_lens, q_offsets, scale, *,
                  max_new, out=None, stream=None):
    """Causal prefill of q [N, Hq, D] over cached prefix + new tokens; returns out."""
    d = pool_desc(k_pool)
    N, Hq, D = q.shape
    if out is None:
        out = torch.empty_like(q)
    R = cached_lens.shape[0]
    st = _load().pkv_paged_prefill(ctypes.byref(d), _dev(out, "out", q.dtype),
                                   _dev(q, "q", k_pool.dtype), _dev(k_pool, "k_pool"),
                                   _dev(v_pool, "v_pool", k_pool.dtype),
                                   _dev(block_tables, "block_tables", torch.int32),
                                   block_tables.shape[1],
                                   _dev(cached_lens, "cached_lens", torch.int32),
                                   _dev(new_lens, "new_lens", torch.int32),
                                   _dev(q_offsets, "q_offsets", torch.int32), R, N, int(max_new),
                                   Hq, float(scale), _stream(stream))
    _check("pkv_paged_prefill", st)
    return out


def copy_blocks(k_pool, v_pool, pairs, stream=None) -> None:
    """pool[dst] = pool[src] for each row (src, dst) of int32 pairs [P, 2]."""
    d = pool_desc(k_pool)
    st = _load().pkv_copy_blocks(ctypes.byref(d), _dev(k_pool, "k_pool"),
                                 _dev(v_pool, "v_pool", k_pool.dtype),
                                 _dev(pairs, "pairs", torch.int32), pairs.shape[0],
                                 _stream(stream))
    _check("pkv_copy_blocks", st)


def read_device_status(stream=None) -> int:
    """Synchronise and return (and clear) the library's device status word."""
    v = ctypes.c_int(0)
    _check("pkv_read_device_status", _load().pkv_read_device_status(ctypes.byref(v),
                                                                    _stream(stream)))
    return v.value


class BlockAllocator:
    """Host block allocator (libpkv's C++ pkv_alloc): slots, tables, refcounts, CoW."""

    def __init__(self, num_blocks: int, block_size: int = BLOCK_SIZE, seed: int = 0):
        self._lib = _load()
        self._h = self._lib.pkv_alloc_create(num_blocks, block_size, seed)
        if not self._h:
            raise ValueError("pkv_alloc_create: invalid arguments")
        self.num_blocks = num_blocks
        self.block_size = block_size

    def close(self):
        if self._h:
            self._lib.pkv_alloc_destroy(self._h)
            self._h = None

    def __del__(self):
        try:
            self.close()
        except Exception:
            pass

    def add_seq(self, seq_id: int, num_tokens: int) -> None:
        _check("pkv_alloc_add_seq", self._lib.pkv_alloc_add_seq(self._h, seq_id, num_tokens))

    def add_seq_shared(self, seq_id: int, shared_blocks, num_tokens: int) -> None:
        """New sequence whose first blocks are existing (shared) blocks."""
        arr = (ctypes.c_int32 * max(len(shared_blocks), 1))(*shared_blocks)
        _check("pkv_alloc_add_seq_shared", self._lib.pkv_alloc_add_seq_shared(
            self._h, seq_id, arr, len(shared_blocks), num_tokens))

    def fork(self, parent: int, child: int) -> None:
        _check("pkv_alloc_fork", self._lib.pkv_alloc_fork(self._h, parent, child))

    def append(self, seq_id: int, n: int = 1):
        """Reserve n slots; returns (slots list, cow pair (old, new) or None)."""
        slots = (ctypes.c_int64 * max(n, 1))()
        pairs = (ctypes.c_int32 * 2)()
        ncow = ctypes.c_int(0)
        _check("pkv_alloc_append", self._lib.pkv_alloc_append(self._h, seq_id, n, slots, pairs,
                                                              ctypes.byref(ncow)))
        return list(slots[:n]), ((pairs[0], pairs[1]) if ncow.value else None)

    def free_seq(self, seq_id: int) -> None:
        _check("pkv_alloc_free_seq", self._lib.pkv_alloc_free_seq(self._h, seq_id))

    def block_table(self, seq_ids, max_blocks: int) -> torch.Tensor:
        ids = (ctypes.c_int64 * len(seq_ids))(*seq_ids)
        out = torch.empty((len(seq_ids), max_blocks), dtype=torch.int32)
        _check("pkv_alloc_block_table", self._lib.pkv_alloc_block_table(
            self._h, ids, len(seq_ids),
            ctypes.cast(out.data_ptr(), ctypes.POINTER(ctypes.c_int32)), max_blocks))
        return out

    @property
    def num_free(self) -> int:
        return int(self._lib.pkv_alloc_num_free(self._h))

    def refcount(self, block: int) -> int:
        return int(self._lib.pkv_alloc_refcount(self._h, block))

    def seq_len(self, seq_id: int) -> int:
        return int(self._lib.pkv_alloc_seq_len(self._h, seq_id))

    def seq_num_blocks(self, seq_id: int) -> int:
        return int(self._lib.pkv_alloc_seq_num_blocks(self._h, seq_id))


def _i32(values):
    """Token ids as a contiguous int32 buffer for the C ABI: (pointer, count).  A numpy
    conversion, not an element-by-element ctypes array (the pointer keeps its buffer
    alive for the call)."""
    a = np.ascontiguousarray(values, dtype=np.int32).reshape(-1)
    n = int(a.size)
    if n == 0:
        a = np.zeros(1, dtype=np.int32)
    return a.ctypes.data_as(ctypes.POINTER(ctypes.c_int32)), n


def block_hash(parent_hash: int, salt: int, tokens, extra: int = 0) -> int:
    arr, n = _i32(tokens)
    return int(_load().pkv_block_hash(parent_hash, salt, arr, n, extra))


class PrefixCache:
    """Chained block-hash prefix cache (libpkv pkv_pcache) over a BlockAllocator."""

    def __init__(self, alloc: BlockAllocator):
        self._lib = _load()
        self.alloc = alloc
        self._h = self._lib.pkv_pcache_create(alloc._h)

    def close(self):
        if self._h:
            self._lib.pkv_pcache_destroy(self._h)
            self._h = None

    def match(self, tokens, salt: int = 0) -> list:
        arr, n = _i32(tokens)
        out = (ctypes.c_int32 * max(n // self.alloc.block_size, 1))()
        k = self._lib.pkv_pcache_match(self._h, arr, n, salt, out, n // self.alloc.block_size)
        if k < 0:
            raise ValueError("pkv_pcache_match: bad arguments")
        return list(out[:k])

    def insert(self, seq_id: int, tokens, salt: int = 0) -> int:
        arr, n = _i32(tokens)
        k = self._lib.pkv_pcache_insert(self._h, seq_id, arr, n, salt)
        if k < 0:
            raise ValueError("pkv_pcache_insert: unknown sequence or too few tokens")
        return k

    def evict(self, min_free: int) -> int:
        return int(self._lib.pkv_pcache_evict(self._h, min_free))

    def __len__(self):
        return int(self._lib.pkv_pcache_size(self._h))


class RadixTree:
    """Radix tree of token sequences (libpkv pkv_radix) over a BlockAllocator."""

    def __init__(self, alloc: BlockAllocator):
        self._lib = _load()
        self.alloc = alloc
        self._h = self._lib.pkv_radix_create(alloc._h)

    def close(self):
        if self._h:
            self._lib.pkv_radix_destroy(self._h)
            self._h = None

    def match(self, tokens):
        """(matched token count, blocks of the matched positions)."""
        arr, n = _i32(tokens)
        nb = -(-n // self.alloc.block_size)
        out = (ctypes.c_int32 * max(nb, 1))()
        m = int(self._lib.pkv_radix_match(self._h, arr, n, out, nb))
        if m < 0:
            raise ValueError("pkv_radix_match: bad arguments")
        return m, list(out[:-(-m // self.alloc.block_size)])

    def insert(self, seq_id: int, tokens) -> None:
        arr, n = _i32(tokens)
        _check("pkv_radix_insert", self._lib.pkv_radix_insert(self._h, seq_id, arr, n))

    def lock(self, tokens, delta: int = 1) -> None:
        arr, n = _i32(tokens)
        _check("pkv_radix_lock", self._lib.pkv_radix_lock(self._h, arr, n, delta))

    def evict(self, min_free: int) -> int:
        return int(self._lib.pkv_radix_evict(self._h, min_free))

    @property
    def num_nodes(self) -> int:
        return int(self._lib.pkv_radix_num_nodes(self._h))

    @property
    def cached_tokens(self) -> int:
        return int(self._lib.pkv_radix_cached_tokens(self._h))
