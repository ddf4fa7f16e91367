"""Shared test helpers: oracle runs on seeded cases and the tolerance check."""
from __future__ import annotations

import json
import os

import numpy as np
import torch

import synth

# Attention outputs (bf16 or fp32 in, fp32 accumulate) against the fp64 oracle.
# Reading of "max-abs 2e-3 and max-rel 1e-2": each element must be within the
# absolute bound OR within the relative bound.  Requiring both of every element is
# impossible for a bf16 output: rounding alone moves a value in [1, 2) by up to
# 2^-8 = 3.9e-3 > 2e-3, while its relative error stays below 2^-9 < 1e-2; and near
# zero only the absolute bound is meaningful.
ATOL = 2e-3
RTOL = 1e-2


def to_f64(t: torch.Tensor) -> np.ndarray:
    return t.detach().float().cpu().numpy().astype(np.float64)


def check_attention(got: torch.Tensor, ref: np.ndarray, mask: np.ndarray | None = None):
    """Compare kernel output with the fp64 oracle; returns (max_abs, max_rel_excess).

    max_rel_excess is the largest err / max(ATOL / RTOL, |ref|): <= RTOL iff every
    element meets one of the two bounds."""
    g = to_f64(got)
    if mask is not None:
        g = g[mask]
        ref = ref[mask]
    assert np.all(np.isfinite(ref)), "oracle rows requested but not computed"
    assert np.all(np.isfinite(g)), "kernel produced non-finite values"
    err = np.abs(g - ref)
    if err.size == 0:
        return 0.0, 0.0
    bad = (err > ATOL) & (err > RTOL * np.abs(ref))
    max_abs = float(err.max())
    score = float((err / np.maximum(np.abs(ref), ATOL / RTOL)).max())
    log = os.environ.get("PKV_PARITY_LOG")
    if log:   # optional record of the errors, for reports
        with open(log, "a") as f:
            f.write(json.dumps({"test": os.environ.get("PYTEST_CURRENT_TEST", "?"),
                                "elements": int(err.size), "max_abs": max_abs,
                                "max_rel_floored": score,
                                "max_rel": float((err / np.maximum(np.abs(ref), 1e-30)).max()),
                                "outside": int(bad.sum())}) + "\n")
    if bad.any():
        i = np.unravel_index(np.argmax(np.where(bad, err, 0)), err.shape)
        raise AssertionError(f"{int(bad.sum())} of {err.size} elements outside both bounds; "
                             f"worst at {i}: got {g[i]:.6g} ref {ref[i]:.6g} "
                             f"(max abs {max_abs:.3e})")
    return max_abs, score


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
