"""Shared test helpers: oracle runs on seeded cases and the tolerance check."""
from __future__ import annotations

import numpy as np
import torch

import synth

# Attention outputs (bf16 or fp32 in, fp32 accumulate): pass iff the largest
# absolute error is <= 2e-3 AND the largest error relative to max(|ref|, 1e-3)
# is <= 1e-2.  The 1e-3 floor makes the relative test meaningful for outputs
# near zero.
ATOL = 2e-3
RTOL = 1e-2
REL_FLOOR = 1e-3


def to_f64(t: torch.Tensor) -> np.ndarray:
    return t.detach().float().cpu().numpy().astype(np.float64)


def check_attention(got: torch.Tensor, ref: np.ndarray, mask: np.ndarray | None = None):
    """Compare kernel output with the fp64 oracle; returns (max_abs, max_rel)."""
    g = to_f64(got)
    if mask is not None:
        g = g[mask]
        ref = ref[mask]
    assert np.all(np.isfinite(ref)), "oracle rows requested but not computed"
    assert np.all(np.isfinite(g)), "kernel produced non-finite values"
    err = np.abs(g - ref)
    max_abs = float(err.max()) if err.size else 0.0
    max_rel = float((err / np.maximum(np.abs(ref), REL_FLOOR)).max()) if err.size else 0.0
    assert max_abs <= ATOL, f"max abs error {max_abs:.3e} > {ATOL}"
    assert max_rel <= RTOL, f"max rel error {max_rel:.3e} > {RTOL}"
    return max_abs, max_rel


def oracle_decode_case(oracle, case: synth.Case, want=None, nthreads=0):
    """Oracle view of a decode case: append on host copies, then fp64 decode."""
    kp = synth.host_bits(case.k_pool)
    vp = synth.host_bits(case.v_pool)
    oracle.kv_append(synth.host_bits(case.slot_mapping), synth.host_bits(case.k_new),
                     synth.host_bits(case.v_new), kp, vp)
    ref = oracle.paged_decode(synth.host_bits(case.q), kp, vp, synth.host_bits(case.block_tables),
                              synth.host_bits(case.context_lens), case.scale, want=want,
                              nthreads=nthreads)
    return ref, kp, vp


def oracle_prefill_case(oracle, case: synth.Case, want=None, nthreads=0):
    kp = synth.host_bits(case.k_pool)
    vp = synth.host_bits(case.v_pool)
    oracle.kv_append(synth.host_bits(case.slot_mapping), synth.host_bits(case.k_new),
                     synth.host_bits(case.v_new), kp, vp)
    ref = oracle.paged_prefill(synth.host_bits(case.q), kp, vp, synth.host_bits(case.block_tables),
                               synth.host_bits(case.cached_lens), synth.host_bits(case.new_lens),
                               synth.host_bits(case.q_offsets), case.scale, want=want,
                               nthreads=nthreads)
    return ref, kp, vp


def pool_equal(gpu_pool: torch.Tensor, host_pool: np.ndarray) -> bool:
    """Bit equality of a device pool with a host pool of bits."""
    if gpu_pool.dtype == torch.bfloat16:
        return torch.equal(gpu_pool.view(torch.int16).cpu(),
                           torch.from_numpy(host_pool.view(np.int16)))
    return torch.equal(gpu_pool.view(torch.int32).cpu(), torch.from_numpy(host_pool.view(np.int32)))
