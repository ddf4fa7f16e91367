"""fp64 CPU oracle for paged-KV attention -- TEST INFRASTRUCTURE ONLY.

Only ``tests/``, ``__graft_entry__.smoke()`` and the CPU-baseline leg of
``bench.py`` may import this package.  The product library
(``paged_kv_cache_58_gb300``) never imports it and shares no code with it.

The arithmetic lives in ``oracle.cpp`` (plain C++17, fp64); this module only
compiles it with g++ and marshals numpy arrays through ctypes.  See the
header of ``oracle.cpp`` for the passages of the pages each function follows
and the readings taken where the pages are silent.

Parity status: every function here is pinned by ``tests/test_oracle_pins.py``
(brute force on tiny inputs, closed forms, invariants the pages fix).
"""
from __future__ import annotations

import ctypes
import os
import subprocess
import threading

import numpy as np

_HERE = os.path.dirname(os.path.abspath(__file__))
_SRC = os.path.join(_HERE, "oracle.cpp")
_LIB = os.path.join(_HERE, "liboracle.so")
_lock = threading.Lock()
_lib = None

F32 = 0
BF16 = 1


def build(force: bool = False) -> str:
    """Compile ``oracle.cpp`` into ``liboracle.so`` (g++, -O2, no -march)."""
    with _lock:
        if force or not os.path.exists(_LIB) or os.path.getmtime(_LIB) < os.path.getmtime(_SRC):
            tmp = _LIB + f".tmp{os.getpid()}"
            cmd = ["g++", "-std=c++17", "-O2", "-fPIC", "-shared", "-pthread", _SRC, "-o", tmp]
            subprocess.run(cmd, check=True)
            os.replace(tmp, _LIB)
    return _LIB


def _load():
    global _lib
    if _lib is None:
        build()
        lib = ctypes.CDLL(_LIB)
        vp, i32p, i64p, f64p, u8p = (ctypes.c_void_p, ctypes.POINTER(ctypes.c_int32),
                                     ctypes.POINTER(ctypes.c_int64),
                                     ctypes.POINTER(ctypes.c_double), ctypes.POINTER(ctypes.c_uint8))
        ci, cl, cd = ctypes.c_int, ctypes.c_int64, ctypes.c_double
        lib.oracle_kv_append.restype = cl
        lib.oracle_kv_append.argtypes = [ci, cl, ci, ci, ci, i64p, cl, vp, vp, vp, vp]
        lib.oracle_copy_blocks.restype = ci
        lib.oracle_copy_blocks.argtypes = [ci, cl, ci, ci, ci, i32p, cl, vp, vp]
        lib.oracle_gather.restype = ci
        lib.oracle_gather.argtypes = [ci, vp, vp, cl, ci, ci, ci, i32p, cl, ci, f64p, f64p]
        lib.oracle_paged_decode.restype = ci
        lib.oracle_paged_decode.argtypes = [ci, vp, vp, vp, cl, ci, ci, ci, i32p, ci, i32p, ci,
                                            ci, cd, u8p, f64p, ci]
        lib.oracle_paged_prefill.restype = ci
        lib.oracle_paged_prefill.argtypes = [ci, vp, vp, vp, cl, ci, ci, ci, i32p, ci, i32p, i32p,
                                             i32p, ci, ci, cd, u8p, f64p, ci]
        lib.oracle_attend_partial.restype = ci
        lib.oracle_attend_partial.argtypes = [f64p, f64p, f64p, cl, cl, ci, cd, f64p, f64p, f64p]
        lib.oracle_lse_merge.restype = ci
        lib.oracle_lse_merge.argtypes = [ci, ci, f64p, f64p, f64p, f64p]
        _lib = lib
    return _lib


def _ptr(a: np.ndarray, ctype=None):
    if ctype is None:
        return ctypes.c_void_p(a.ctypes.data)
    return a.ctypes.data_as(ctypes.POINTER(ctype))


def _dtype_code(a: np.ndarray) -> int:
    """Pool/query element type: float32 arrays are fp32, uint16 arrays hold bf16 bits."""
    if a.dtype == np.float32:
        return F32
    if a.dtype == np.uint16:
        return BF16
    raise TypeError(f"oracle takes float32 or uint16 (bf16 bits) arrays, got {a.dtype}")


def _c(a, dtype=None):
    return np.ascontiguousarray(a if dtype is None else np.asarray(a, dtype=dtype))


def kv_append(slot_mapping, k, v, k_pool, v_pool):
    """In-place scatter of k/v [T, Hkv, D] rows into pools [NB, Hkv, B, D]."""
    assert k_pool.flags.c_contiguous and v_pool.flags.c_contiguous
    code = _dtype_code(k_pool)
    nb, hkv, bs, d = k_pool.shape
    slots = _c(slot_mapping, np.int64)
    k = _c(k).astype(k_pool.dtype, copy=False)
    v = _c(v).astype(v_pool.dtype, copy=False)
    n = _load().oracle_kv_append(code, nb, bs, hkv, d, _ptr(slots, ctypes.c_int64), slots.size,
                                 _ptr(k), _ptr(v), _ptr(k_pool), _ptr(v_pool))
    if n < 0:
        raise ValueError("slot out of range")
    return n


def copy_blocks(pairs, k_pool, v_pool):
    """In-place pool[dst] = pool[src] for each (src, dst) pair, in order."""
    code = _dtype_code(k_pool)
    nb, hkv, bs, d = k_pool.shape
    pr = _c(pairs, np.int32).reshape(-1, 2)
    rc = _load().oracle_copy_blocks(code, nb, bs, hkv, d, _ptr(pr, ctypes.c_int32), pr.shape[0],
                                    _ptr(k_pool), _ptr(v_pool))
    if rc != 0:
        raise ValueError("block id out of range")


def gather(k_pool, v_pool, table_row, length: int, kvh: int):
    """Contiguous fp64 K, V [length, D] of one (sequence, kv head)."""
    code = _dtype_code(k_pool)
    nb, hkv, bs, d = k_pool.shape
    row = _c(table_row, np.int32)
    K = np.zeros((length, d), np.float64)
    V = np.zeros((length, d), np.float64)
    rc = _load().oracle_gather(code, _ptr(k_pool), _ptr(v_pool), nb, bs, hkv, d,
                               _ptr(row, ctypes.c_int32), length, kvh, _ptr(K, ctypes.c_double),
                               _ptr(V, ctypes.c_double))
    if rc != 0:
        raise ValueError("block table points outside the pool")
    return K, V


def paged_decode(q, k_pool, v_pool, block_tables, context_lens, scale, want=None, nthreads=0):
    """fp64 decode output [S, Hq, D]; rows not in `want` ([S, Hq] bool) stay NaN."""
    code = _dtype_code(k_pool)
    assert _dtype_code(q) == code
    nb, hkv, bs, d = k_pool.shape
    s, hq, dq = q.shape
    assert dq == d
    q = _c(q)
    bt = _c(block_tables, np.int32)
    cl = _c(context_lens, np.int32)
    out = np.full((s, hq, d), np.nan, np.float64)
    wp = None
    if want is not None:
        w = _c(want, np.uint8)
        wp = _ptr(w, ctypes.c_uint8)
    rc = _load().oracle_paged_decode(code, _ptr(q), _ptr(_c(k_pool)), _ptr(_c(v_pool)), nb, bs,
                                     hkv, d, _ptr(bt, ctypes.c_int32), bt.shape[1],
                                     _ptr(cl, ctypes.c_int32), s, hq, float(scale), wp,
                                     _ptr(out, ctypes.c_double), int(nthreads))
    if rc != 0:
        raise ValueError(f"oracle_paged_decode failed ({rc})")
    return out


def paged_prefill(q, k_pool, v_pool, block_tables, cached_lens, new_lens, q_offsets, scale,
                  want=None, nthreads=0):
    """fp64 prefill output [N, Hq, D]; rows not in `want` ([N, Hq] bool) stay NaN."""
    code = _dtype_code(k_pool)
    assert _dtype_code(q) == code
    nb, hkv, bs, d = k_pool.shape
    n, hq, dq = q.shape
    assert dq == d
    q = _c(q)
    bt = _c(block_tables, np.int32)
    c = _c(cached_lens, np.int32)
    nl = _c(new_lens, np.int32)
    qo = _c(q_offsets, np.int32)
    out = np.full((n, hq, d), np.nan, np.float64)
    wp = None
    if want is not None:
        w = _c(want, np.uint8)
        wp = _ptr(w, ctypes.c_uint8)
    rc = _load().oracle_paged_prefill(code, _ptr(q), _ptr(_c(k_pool)), _ptr(_c(v_pool)), nb, bs,
                                      hkv, d, _ptr(bt, ctypes.c_int32), bt.shape[1],
                                      _ptr(c, ctypes.c_int32), _ptr(nl, ctypes.c_int32),
                                      _ptr(qo, ctypes.c_int32), c.size, hq, float(scale), wp,
                                      _ptr(out, ctypes.c_double), int(nthreads))
    if rc != 0:
        raise ValueError(f"oracle_paged_prefill failed ({rc})")
    return out


def attend_partial(q, K, V, lo: int, hi: int, scale: float):
    """(o_part[D], m, l) of fp64 query q over contiguous keys [lo, hi)."""
    q = _c(q, np.float64)
    K = _c(K, np.float64)
    V = _c(V, np.float64)
    d = q.size
    o = np.zeros(d, np.float64)
    m = ctypes.c_double()
    l = ctypes.c_double()
    rc = _load().oracle_attend_partial(_ptr(q, ctypes.c_double), _ptr(K, ctypes.c_double),
                                       _ptr(V, ctypes.c_double), lo, hi, d, float(scale),
                                       _ptr(o, ctypes.c_double), ctypes.byref(m), ctypes.byref(l))
    if rc != 0:
        raise ValueError("empty key range")
    return o, m.value, l.value


def lse_merge(o_parts, m_parts, l_parts):
    """Log-sum-exp merge of P partials o_parts [P, D], m_parts [P], l_parts [P]."""
    o = _c(o_parts, np.float64)
    m = _c(m_parts, np.float64)
    l = _c(l_parts, np.float64)
    p, d = o.shape
    out = np.zeros(d, np.float64)
    rc = _load().oracle_lse_merge(p, d, _ptr(o, ctypes.c_double), _ptr(m, ctypes.c_double),
                                  _ptr(l, ctypes.c_double), _ptr(out, ctypes.c_double))
    if rc != 0:
        raise ValueError("no partials")
    return out
