"""Benchmark of the paged-KV decode hot path on GB300.

A step is one pass of the hot path over one batch of the Llama-3-8B-shaped
decode layer: kv_append of the batch's 64 new tokens and paged_decode of the
64 queries over their paged contexts (split-KV partitions + LSE combine).  By
default both run as one call, pkv_paged_decode_append (the decode kernel stores
and attends the new tokens); --separate-append times kv_append followed by
paged_decode instead.
Inputs are seeded synthetic tensors already resident in HBM.  Prints ONE JSON
line (rank 0).  Beside the step, the line carries measurements of the other
published workloads on the same GPU, each with its roofline and the fp64 oracle
timed on the host cores: the prefix-cached prefill (its kv_append alone, the
prefill alone, and the two as one step), the Llama-3.1-70B-shaped long-context
decode, and the shared-prefix batch through the cascade decode.

  python bench.py [--gpus N] [--steps K] [--warmup W] [--impl ours|reference]

--impl reference times the fp64 CPU oracle (the only baseline that exists for
this path) on the host cores, on a bounded sample of the same workload.
--gpus N runs N independent replicas, one process per GPU (re-launched through
torch.distributed.run unless already under it); the decode batch exchanges no
data, so the only cross-rank traffic is the barriers around the timed region
and the max of its time over ranks (weak scaling).
"""
from __future__ import annotations

import argparse
import json
import math
import os
import statistics
import subprocess
import sys
import time

ROOT = os.path.dirname(os.path.abspath(__file__))
if ROOT not in sys.path:
    sys.path.insert(0, ROOT)

METRIC = "paged decode HBM GB/s (% of ~8 TB/s peak) and decode tokens/s per layer"
NOMINAL_HBM_GBS = 8000.0
FALLBACK_HBM_GBS = 6800.0
FP32_ALU_TFLOPS = 152 * 128 * 2 * 2.07e9 / 1e12   # 80.5
DECODE_WORKLOADS = ("8b", "70b", "shared", "tiny")


def parse():
    p = argparse.ArgumentParser()
    p.add_argument("--gpus", type=int, default=1)
    p.add_argument("--steps", type=int, default=200)
    p.add_argument("--warmup", type=int, default=20)
    p.add_argument("--impl", choices=["ours", "reference"], default="ours")
    p.add_argument("--no-cpu-baseline", action="store_true")
    p.add_argument("--no-e2e", action="store_true")
    p.add_argument("--workload", choices=DECODE_WORKLOADS, default="8b",
                   help="decode workload of the step (default: the Llama-3-8B-shaped batch)")
    p.add_argument("--partition-blocks", type=int, default=0,
                   help="split-KV partition size in blocks (0: the library's policy)")
    p.add_argument("--cascade", action="store_true",
                   help="shared workload: decode with the shared-prefix cascade")
    p.add_argument("--separate-append", action="store_true",
                   help="time kv_append + paged_decode as two calls instead of the fused "
                        "pkv_paged_decode_append")
    p.add_argument("--block-size", type=int, choices=[16, 32], default=0,
                   help="tokens per pool block for the decode and prefill workloads "
                        "(default: the recipe's 16; the pools keep their byte size)")
    p.add_argument("--prefill-head-dim", type=int, choices=[64, 128], default=128)
    p.add_argument("--prefill-dtype", choices=["bf16", "fp32"], default="bf16")
    p.add_argument("--no-prefill", action="store_true")
    p.add_argument("--no-prefix-cache", action="store_true",
                   help="skip the host prefix-reuse measurement")
    p.add_argument("--prefill-steps", type=int, default=20)
    p.add_argument("--no-long-decode", action="store_true",
                   help="skip the Llama-3.1-70B-shaped long-context decode sub-line")
    p.add_argument("--no-cascade-line", action="store_true",
                   help="skip the shared-prefix cascade decode sub-line")
    p.add_argument("--sub-steps", type=int, default=20,
                   help="timed calls of each decode sub-line")
    p.add_argument("--min-warm-seconds", type=float, default=1.0,
                   help="warm-up also runs at least this long (clock sampling under load)")
    return p.parse_args()


def dist_env():
    ws = int(os.environ.get("WORLD_SIZE", "1"))
    rank = int(os.environ.get("RANK", "0"))
    local = int(os.environ.get("LOCAL_RANK", "0"))
    return ws, rank, local


def _free_port() -> int:
    import socket
    with socket.socket() as sk:
        sk.bind(("127.0.0.1", 0))
        return sk.getsockname()[1]


def launch_replicas(n: int, argv, script: str | None = None, stdout=None):
    """Runs `script` (this file by default) as n processes on this node through
    torch.distributed.run, one per GPU, rendezvous on 127.0.0.1; returns the
    CompletedProcess.  Rank 0 prints the JSON line (passed through, or captured when
    stdout is subprocess.PIPE)."""
    cmd = [sys.executable, "-m", "torch.distributed.run", "--nnodes=1",
           f"--nproc-per-node={n}", "--master-addr=127.0.0.1", f"--master-port={_free_port()}",
           script or os.path.abspath(__file__), *argv]
    return subprocess.run(cmd, stdout=stdout, text=True)


class Ranks:
    """The replica processes of one run (RANK, LOCAL_RANK, WORLD_SIZE and MASTER_* from
    the environment, as torch.distributed.run sets them).  Replicas are independent: the
    only collectives are the barriers around a timed region and the max of its time."""

    def __init__(self, backend: str, device=None):
        import torch.distributed as dist
        self.dist = dist
        self.ws, self.rank, self.local = dist_env()
        self.device = device
        if self.ws > 1:
            dist.init_process_group(backend)

    def barrier(self):
        if self.ws > 1:
            self.dist.barrier()

    def max(self, x: float) -> float:
        if self.ws == 1:
            return x
        import torch
        t = torch.tensor([x], dtype=torch.float64, device=self.device)
        self.dist.all_reduce(t, op=self.dist.ReduceOp.MAX)
        return float(t.item())

    def close(self):
        if self.ws > 1:
            self.dist.destroy_process_group()


class EventClock:
    """Seconds between two CUDA events on the launching stream (synchronised)."""

    def __init__(self, stream):
        import torch
        self.torch, self.stream = torch, stream

    def sync(self):
        self.torch.cuda.synchronize()

    def begin(self):
        self.a = self.torch.cuda.Event(enable_timing=True)
        self.b = self.torch.cuda.Event(enable_timing=True)
        self.a.record(self.stream)

    def end(self) -> float:
        self.b.record(self.stream)
        self.torch.cuda.synchronize()
        return self.a.elapsed_time(self.b) * 1e-3


class WallClock:
    """Host seconds around work that synchronises itself (the end-to-end steps)."""

    def sync(self):
        pass

    def begin(self):
        self.t0 = time.perf_counter()

    def end(self) -> float:
        return time.perf_counter() - self.t0


def replica_rate(ranks: Ranks, step, K: int, units_per_step: float, clock):
    """K steps back to back, with a barrier and a synchronisation on both sides; returns
    (whole-job units per second, max over ranks of the elapsed seconds): the work of all
    ranks over the slowest rank's time."""
    ranks.barrier()
    clock.sync()
    clock.begin()
    for _ in range(K):
        step()
    el = clock.end()
    ranks.barrier()
    return aggregate(el, units_per_step * K, ranks.ws, ranks.max)


FALLBACK_BF16_TFLOPS = 1900.0


def peaks():
    """(hbm GB/s, bf16 burst TFLOP/s, kind) from MEASURED_PEAKS.json, else the fallback."""
    path = os.path.join(ROOT, "MEASURED_PEAKS.json")
    try:
        d = json.load(open(path))
        return float(d["hbm_gbs"]), float(d["bf16_tflops"]), "measured"
    except Exception:
        return FALLBACK_HBM_GBS, FALLBACK_BF16_TFLOPS, "fallback"


def prefill_flops(case):
    """Algorithmic flops of one prefill call: QK^T and PV over causal pairs only,
    4 * D * Hq per (query token, key it attends)."""
    D = case.q.shape[2]
    Hq = case.q.shape[1]
    total = 0
    for c, n in zip(case.cached_lens.tolist(), case.new_lens.tolist()):
        total += n * c + n * (n + 1) // 2     # sum over i < n of (c + i + 1)
    return 4 * D * Hq * total


class L2Flush:
    """Writes a buffer of twice the L2 size, evicting what earlier calls left in L2, for
    timed calls whose bytes would otherwise fit in it."""

    def __init__(self, dev):
        import torch
        l2 = torch.cuda.get_device_properties(dev).L2_cache_size or (129 << 20)
        self.buf = torch.empty(2 * l2, dtype=torch.uint8, device=dev)

    def __call__(self):
        self.buf.fill_(1)


def time_calls(call, steps, stream, before=None):
    """Mean seconds of `call` over `steps` launches, CUDA events around each on the
    launching stream; `before` (an L2 flush) runs ahead of each start event."""
    import torch
    evs = [(torch.cuda.Event(enable_timing=True), torch.cuda.Event(enable_timing=True))
           for _ in range(steps)]
    for a, b in evs:
        if before is not None:
            before()
        a.record(stream)
        call()
        b.record(stream)
    torch.cuda.synchronize()
    return statistics.mean(a.elapsed_time(b) for a, b in evs) * 1e-3


def append_bytes_of(k_new, slot_mapping):
    """Algorithmic bytes of one kv_append: the new K and V rows read, the same bytes
    written into the pools, and the slot mapping read."""
    return 2 * 2 * k_new.numel() * k_new.element_size() + \
        slot_mapping.numel() * slot_mapping.element_size()


def bench_prefill(pkv, dev, steps, stream, block_size=0, head_dim=128, dtype="bf16",
                  peaks_=None, cpu=True, e2e=True):
    """Prefix-cached chunked prefill (16 requests x 512 new tokens over cached
    prefixes of U[1024, 8192]) measured three ways: the kv_append of the 8192 new rows
    alone (L2 flushed before each call: its 67 MB fit in L2), the prefill call alone
    (K/V of 335 MB per call > L2), and the workload's step, append then prefill, K
    times back to back.  block_size, head_dim and dtype vary the recipe (the pool keeps
    its byte size).  With `e2e` the step is also timed end to end from pinned host
    buffers; with `cpu` the oracle prefill is timed on the host cores over the first
    requests of the batch."""
    import dataclasses
    import torch
    import synth
    hbm, tpeak, kind = peaks_ or peaks()
    wl = synth.WORKLOADS["prefill"]
    over = {}
    if block_size and block_size != wl.block_size:
        over.update(block_size=block_size,
                    num_blocks=wl.num_blocks * wl.block_size // block_size)
    if head_dim != wl.head_dim:
        over.update(head_dim=head_dim)
    if dtype == "fp32":
        over.update(dtype=torch.float32)
    if over:
        wl = dataclasses.replace(wl, name=wl.name + "".join(
            f"_{k}{v}" for k, v in (("B", over.get("block_size")), ("D", over.get("head_dim")),
                                    ("", "f32" if dtype == "fp32" else None)) if v), **over)
    case = synth.build_case(wl, dev)
    out = torch.empty_like(case.q)
    max_new = int(case.new_lens.max())

    def append():
        pkv.kv_append(case.k_pool, case.v_pool, case.slot_mapping, case.k_new, case.v_new,
                      stream=stream)

    def call():
        pkv.paged_prefill(case.q, case.k_pool, case.v_pool, case.block_tables,
                          case.cached_lens, case.new_lens, case.q_offsets, case.scale,
                          max_new=max_new, out=out, stream=stream)

    def step():
        append()
        call()

    for _ in range(3):
        step()
    torch.cuda.synchronize()
    assert pkv.read_device_status() == 0
    ms = time_calls(call, steps, stream) * 1e3
    flush = L2Flush(dev)
    append_s = time_calls(append, steps, stream, before=flush)
    sustained_s, eager_s = append_sustained(pkv, case, steps, stream)
    clock = EventClock(stream)
    clock.sync()
    clock.begin()
    for _ in range(steps):
        step()
    step_s = clock.end() / steps
    assert pkv.read_device_status() == 0
    del flush
    flops = prefill_flops(case)
    esz = case.q.element_size()
    kv_bytes = int((case.context_lens.to(torch.int64)).sum()) * case.k_pool.shape[1] * \
        case.q.shape[2] * esz * 2
    ab = append_bytes_of(case.k_new, case.slot_mapping)
    res = {"workload": case.wl.name, "ms": ms, "tflops": flops / (ms * 1e-3) / 1e12,
           "flops_per_call": flops, "kv_bytes_per_call": kv_bytes, "launches": steps,
           "block_size": case.k_pool.shape[2], "head_dim": case.q.shape[2],
           "dtype": "f32" if esz == 4 else "bf16",
           "step": {"calls": "kv_append (8192 new rows) + paged_prefill, back to back",
                    "ms": step_s * 1e3, "tflops": flops / step_s / 1e12, "steps": steps,
                    "gpu_launches": 2 * steps},
           "append": {"kernel": "kv_append_kernel", "rows": int(case.k_new.shape[0]),
                      "bytes_per_call": ab, "ms": sustained_s * 1e3,
                      "timing": ("calls back to back over 4 rotating sets of new rows and "
                                 "slots (268 MB, larger than L2), replayed from a CUDA graph, "
                                 "CUDA events around all"),
                      "ms_eager_back_to_back": eager_s * 1e3,
                      "ms_single_call_l2_flushed": append_s * 1e3,
                      "roofline": {"bound": "hbm", "achieved": ab / sustained_s / 1e9,
                                   "peak": hbm, "unit": "GB/s",
                                   "frac": ab / sustained_s / 1e9 / hbm,
                                   "peak_kind": f"{kind} hbm_gbs",
                                   "frac_of_8tbs": ab / sustained_s / 1e9 / NOMINAL_HBM_GBS,
                                   "traffic": None}}}
    if e2e:
        res["e2e"] = prefill_e2e(pkv, case, out, max_new, steps, stream, flops)
    if cpu:
        res["cpu_baseline"] = prefill_cpu_baseline(case, flops)
    del case, out
    torch.cuda.empty_cache()
    return res


def prefill_e2e(pkv, case, out, max_new, steps, stream, flops):
    """The prefill step end to end from pinned host memory through
    pkv_paged_prefill_append_host, per step: the step's packed inputs (q, the block
    tables, the requests' cached and new lengths and q offsets, the new K/V rows and
    their slots) copied in, the output copied back, and a synchronise.  Host seconds
    over `steps` steps."""
    import torch
    T, Hq, D = case.q.shape
    R = case.cached_lens.numel()
    mbs = case.block_tables.shape[1]
    lay = pkv.prefill_step_layout(case.k_pool, R, T, Hq, mbs)
    host_in = torch.empty(lay.bytes, dtype=torch.uint8).pin_memory()
    pkv.pack_prefill_step(host_in, lay, case.q.cpu(), case.block_tables.cpu(),
                          case.cached_lens.cpu(), case.new_lens.cpu(), case.q_offsets.cpu(),
                          case.k_new.cpu(), case.v_new.cpu(), case.slot_mapping.cpu())
    out_h = torch.empty(out.shape, dtype=out.dtype).pin_memory()
    staging = torch.empty(pkv.prefill_host_staging_bytes(case.k_pool, R, T, Hq, mbs),
                          dtype=torch.uint8, device=case.q.device)

    def step():
        pkv.paged_prefill_append_host(case.k_pool, case.v_pool, host_in, out_h, case.scale,
                                      num_reqs=R, total_new=T, max_new=max_new, num_q_heads=Hq,
                                      max_blocks_per_seq=mbs, staging=staging, stream=stream)
        stream.synchronize()

    for _ in range(3):
        step()
    assert pkv.read_device_status() == 0
    assert torch.equal(out_h.view(torch.uint8), out.cpu().view(torch.uint8))
    clock = WallClock()
    clock.begin()
    for _ in range(steps):
        step()
    sec = clock.end() / steps
    moved = {"h2d_bytes_per_step": lay.bytes, "d2h_bytes_per_step": out_h.numel() * out_h.element_size()}
    return {"value": flops / sec / 1e12, "unit": "TFLOP/s", "ms_per_step": sec * 1e3,
            "api": ("pkv_paged_prefill_append_host (pinned buffers; copies in and out "
                    "pipelined with the kernels over 4 request chunks)"),
            **moved, "steps": steps}


def append_sustained(pkv, case, steps, stream, sets=4):
    """Seconds per kv_append of the workload's shape (8192 rows of K and V) with calls
    back to back: `sets` different sets of new rows, each with its own slots in pool
    blocks no block table references, used in turn, so that what a call reads and
    writes was last touched sets - 1 calls earlier (268 MB in between at 4 sets, more
    than L2 holds).  The workload's own pool contents are left as they are.  Returns
    (seconds per call replayed from a CUDA graph, seconds per call launched eagerly)."""
    import torch
    nb, _, B, _ = case.k_pool.shape
    T = case.k_new.shape[0]
    used = torch.zeros(nb, dtype=torch.bool, device=case.k_pool.device)
    bt = case.block_tables
    used[bt[bt >= 0].long()] = True
    free = torch.nonzero(~used).flatten()
    per = -(-T // B)
    if free.numel() < sets * per:
        return float("nan"), float("nan")
    g = torch.Generator(device=case.k_pool.device).manual_seed(77)
    data = []
    for i in range(sets):
        blocks = free[i * per:(i + 1) * per]
        slots = (blocks[:, None] * B + torch.arange(B, device=blocks.device)[None, :]).flatten()
        slots = slots[torch.randperm(slots.numel(), generator=g, device=slots.device)[:T]]
        kn = torch.randn(case.k_new.shape, generator=g, device=case.k_new.device).to(
            case.k_new.dtype)
        vn = torch.randn(case.v_new.shape, generator=g, device=case.v_new.device).to(
            case.v_new.dtype)
        data.append((slots.contiguous(), kn, vn))
    for i in range(2 * sets):
        sl, kn, vn = data[i % sets]
        pkv.kv_append(case.k_pool, case.v_pool, sl, kn, vn, stream=stream)
    n = max(steps, 2 * sets)
    clock = EventClock(stream)
    clock.sync()
    clock.begin()
    for i in range(n):
        sl, kn, vn = data[i % sets]
        pkv.kv_append(case.k_pool, case.v_pool, sl, kn, vn, stream=stream)
    eager = clock.end() / n
    # The same n calls captured once in a CUDA graph and replayed: back to back on the
    # GPU without the Python call between launches (a ~10 us kernel is shorter than
    # the host side of one call).
    gs = torch.cuda.Stream(device=case.k_pool.device)
    gs.wait_stream(stream)
    graph = torch.cuda.CUDAGraph()
    with torch.cuda.graph(graph, stream=gs):
        for i in range(n):
            sl, kn, vn = data[i % sets]
            pkv.kv_append(case.k_pool, case.v_pool, sl, kn, vn, stream=gs)
    with torch.cuda.stream(gs):   # replay() launches on the current stream
        graph.replay()
        gclock = EventClock(gs)
        gclock.sync()
        gclock.begin()
        graph.replay()
        sec = gclock.end() / n
    assert pkv.read_device_status() == 0
    del graph
    return sec, eager


def prefill_cpu_baseline(case, flops_all, budget_s=10.0):
    """The oracle prefill on the host cores over the batch's first requests (the number
    sized so that the repeated passes take about `budget_s`), in TFLOP/s of the same
    algorithmic flops the GPU figure counts."""
    import numpy as np
    import oracle
    import synth
    oracle.build()
    kp, vp = synth.host_bits(case.k_pool), synth.host_bits(case.v_pool)
    q, bt = synth.host_bits(case.q), synth.host_bits(case.block_tables)
    cl, nl = synth.host_bits(case.cached_lens), synth.host_bits(case.new_lens)
    qo = synth.host_bits(case.q_offsets)
    D, Hq = q.shape[2], q.shape[1]

    def run(nr):
        rows = int(qo[nr])
        t0 = time.perf_counter()
        oracle.paged_prefill(q[:rows], kp, vp, bt[:nr], cl[:nr], nl[:nr], qo[:nr + 1],
                             case.scale)
        return time.perf_counter() - t0

    t1 = run(1)
    nr = int(max(1, min(len(cl), budget_s / 2 / max(t1, 1e-9))))
    reps, el = 0, 0.0
    while el < budget_s / 2 or reps < 1:
        el += run(nr)
        reps += 1
    sub = 4 * D * Hq * sum(int(n) * int(c) + int(n) * (int(n) + 1) // 2
                           for c, n in zip(cl[:nr], nl[:nr]))
    return {"value": sub * reps / el / 1e12, "unit": "TFLOP/s", "cores": os.cpu_count(),
            "kind": "oracle",
            "sample": f"first {nr} of {len(cl)} requests ({sub / 1e9:.1f} of "
                      f"{flops_all / 1e9:.0f} GFLOP), {reps} passes in {el:.1f} s; fp64, "
                      "std::thread over (request, kv head)"}


def decode_cpu_baseline(case, bytes_all, tokens_all, budget_s=8.0):
    """The oracle decode on the host cores over the batch's first sequences (sized so the
    repeated passes take about `budget_s`), in GB/s of the same algorithmic bytes the GPU
    figure counts, scaled by the sample's share of the attended tokens."""
    import numpy as np
    import oracle
    import synth
    oracle.build()
    kp, vp = synth.host_bits(case.k_pool), synth.host_bits(case.v_pool)
    oracle.kv_append(synth.host_bits(case.slot_mapping), synth.host_bits(case.k_new),
                     synth.host_bits(case.v_new), kp, vp)
    q, bt = synth.host_bits(case.q), synth.host_bits(case.block_tables)
    cl = synth.host_bits(case.context_lens)

    def run(n):
        t0 = time.perf_counter()
        oracle.paged_decode(q[:n], kp, vp, bt[:n], cl[:n], case.scale)
        return time.perf_counter() - t0

    t1 = run(1)
    n = int(max(1, min(len(cl), budget_s / 2 / max(t1, 1e-9))))
    reps, el = 0, 0.0
    while el < budget_s / 2 or reps < 1:
        el += run(n)
        reps += 1
    tok = int(cl[:n].astype(np.int64).sum())
    sub_bytes = bytes_all * tok / max(tokens_all, 1)
    return {"value": sub_bytes * reps / el / 1e9, "unit": "GB/s", "cores": os.cpu_count(),
            "kind": "oracle", "tokens_per_s_per_layer": n * reps / el,
            "sample": f"first {n} of {len(cl)} sequences ({tok} of {tokens_all} tokens, all "
                      f"heads), {reps} passes in {el:.1f} s; fp64, std::thread over "
                      "(sequence, kv head)"}


def with_block_size(wl, block_size):
    """The workload recipe with `block_size`-token pool blocks (the pool keeps its byte
    size); unchanged for 0 or the recipe's own size."""
    import dataclasses
    if not block_size or block_size == wl.block_size:
        return wl
    return dataclasses.replace(wl, name=f"{wl.name}_B{block_size}", block_size=block_size,
                               num_blocks=wl.num_blocks * wl.block_size // block_size)


def bench_decode_line(pkv, dev, name, steps, stream, peaks_, cascade=False, cpu=True,
                      block_size=0):
    """One published decode workload through its fused call (append + decode, or the
    cascade decode with the append for the shared-prefix batch), timed per call with
    CUDA events; its GB/s on the unique bytes against the HBM roofline, the logical rate,
    tokens/s, and the oracle on the host cores."""
    import torch
    import synth
    hbm, _, kind = peaks_
    case = synth.build_case(with_block_size(synth.WORKLOADS[name], block_size), dev)
    S, Hq, D = case.q.shape
    B = case.k_pool.shape[2]
    decode_bytes, append_bytes, tokens, unique = workload_bytes(case)
    append_bytes -= case.slot_mapping.numel() * case.slot_mapping.element_size()  # fused
    max_ctx = case.max_context
    out = torch.empty_like(case.q)
    if cascade:
        plen = case.wl.shared_prefix
        prefix_blocks = case.block_tables[0, :plen // B].contiguous()
        ws = torch.empty(max(16, pkv.cascade_workspace_bytes(S, Hq, D, plen, max_ctx,
                                                             block_size=B)),
                         dtype=torch.uint8, device=dev)

        def call():
            pkv.paged_decode_cascade_append(case.q, case.k_pool, case.v_pool, case.k_new,
                                            case.v_new, prefix_blocks, plen,
                                            case.block_tables, case.context_lens, case.scale,
                                            max_context=max_ctx, out=out, workspace=ws,
                                            stream=stream)
        kernel = ("paged_decode_cascade_append (tcgen05 prefix pass on a side stream + suffix "
                  "split-KV decode with the append + combine)")
        launches = 3
    else:
        pb = pkv.auto_partition(S, Hq, max_ctx, block_size=B)
        ws = torch.empty(max(16, pkv.decode_workspace_bytes(S, Hq, D, max_ctx, pb,
                                                            block_size=B)),
                         dtype=torch.uint8, device=dev)

        def call():
            pkv.paged_decode_append(case.q, case.k_pool, case.v_pool, case.k_new, case.v_new,
                                    case.block_tables, case.context_lens, case.scale,
                                    max_context=max_ctx, out=out, partition_blocks=pb,
                                    workspace=ws, stream=stream)
        kernel = "paged_decode_append (decode_tc split-KV with the append + combine)"
        launches = 2
    for _ in range(3):
        call()
    torch.cuda.synchronize()
    assert pkv.read_device_status() == 0
    sec = time_calls(call, steps, stream)
    assert pkv.read_device_status() == 0
    call_bytes = unique + append_bytes
    achieved = call_bytes / sec / 1e9
    res = {"workload": case.wl.name, "num_seqs": S, "q_heads": Hq,
           "kv_heads": case.k_pool.shape[1], "head_dim": D, "block_size": B,
           "mean_context": tokens / S, "max_context": max_ctx, "ms": sec * 1e3,
           "calls": steps, "gpu_launches": launches * steps,
           "tokens_per_s_per_layer": S / sec,
           "logical_gbs": (decode_bytes + append_bytes) / sec / 1e9,
           "kv_bytes_per_call": decode_bytes, "unique_kv_bytes_per_call": unique,
           "l2": ("K/V per call larger than L2" if unique > 2 * 129e6
                  else "K/V per call fits in L2: warm-cache figure"),
           "roofline": {"bound": "hbm", "kernel": kernel, "achieved": achieved, "peak": hbm,
                        "unit": "GB/s", "frac": achieved / hbm,
                        "peak_kind": f"{kind} hbm_gbs", "bytes_per_launch": call_bytes,
                        "frac_of_8tbs": achieved / NOMINAL_HBM_GBS, "traffic": None}}
    if cpu:
        res["cpu_baseline"] = decode_cpu_baseline(case, decode_bytes + append_bytes, tokens)
    del case, out, ws
    torch.cuda.empty_cache()
    return res


def bench_prefix_cache(pkv, convs=32, turns=8, system=1024, per_turn=160, tail=64, reps=3):
    """Host prefix reuse on a multi-turn agent workload (seeded): `convs` conversations
    behind one shared `system`-token prompt; turn t's prompt is the system prompt plus
    the conversation's first t * per_turn + tail tokens.  Each admission is the serving
    flow through the binding: match, admit with the matched blocks shared, append the
    rest, insert, free.  Reports admissions/s and the share of prompt tokens reused,
    for the radix tree and for the chained block-hash cache."""
    import random
    rng = random.Random(58)
    sys_prompt = [rng.randrange(32000) for _ in range(system)]
    conv = [[rng.randrange(32000) for _ in range(turns * per_turn + tail)]
            for _ in range(convs)]
    order = [(t, c) for t in range(turns) for c in range(convs)]   # turns interleaved
    res = {}
    for kind in ("radix", "block_hash"):
        best = None
        for _ in range(reps):
            alloc = pkv.BlockAllocator(16384)
            cache = pkv.RadixTree(alloc) if kind == "radix" else pkv.PrefixCache(alloc)
            reused = total = 0
            t0 = time.perf_counter()
            for sid, (t, c) in enumerate(order):
                prompt = sys_prompt + conv[c][:t * per_turn + tail]
                if kind == "radix":
                    m, blocks = cache.match(prompt)
                else:
                    blocks = cache.match(prompt)
                    m = len(blocks) * alloc.block_size
                alloc.add_seq_shared(sid, blocks, m)
                alloc.append(sid, len(prompt) - m)
                cache.insert(sid, prompt)
                alloc.free_seq(sid)
                reused += m
                total += len(prompt)
            el = time.perf_counter() - t0
            cache.close()
            alloc.close()
            if best is None or el < best:
                best = el
        res[kind] = {"admissions_per_s": len(order) / best, "reused_fraction": reused / total,
                     "prompt_tokens": total}
    res["workload"] = (f"{convs} conversations x {turns} turns, {system}-token shared system "
                       f"prompt, +{per_turn} tokens a turn; one host thread through the "
                       "Python binding")
    return res


class ClockSampler:
    """nvidia-smi sampling of SM clock and throttle reasons while the GPU works."""
    Q = ("index,clocks.sm,clocks.max.sm,power.draw,clocks_event_reasons.active,"
         "clocks_event_reasons.hw_slowdown,clocks_event_reasons.hw_thermal_slowdown,"
         "clocks_event_reasons.sw_thermal_slowdown,clocks_event_reasons.sw_power_cap")

    def __init__(self, gpu_index: int):
        self.gpu = gpu_index
        self.proc = None
        self.lines = []

    def start(self):
        try:
            self.proc = subprocess.Popen(
                ["nvidia-smi", f"--id={self.gpu}", f"--query-gpu={self.Q}",
                 "--format=csv,noheader,nounits", "-lms", "100"],
                stdout=subprocess.PIPE, stderr=subprocess.DEVNULL, text=True)
        except Exception:
            self.proc = None

    def stop(self):
        if not self.proc:
            return {"sm_mhz": None, "sm_max_mhz": None, "reasons": ["nvidia-smi unavailable"]}
        self.proc.terminate()
        try:
            out, _ = self.proc.communicate(timeout=5)
        except Exception:
            self.proc.kill()
            out, _ = self.proc.communicate()
        sm, smax, reasons = [], [], set()
        names = ["hw_slowdown", "hw_thermal_slowdown", "sw_thermal_slowdown", "sw_power_cap"]
        for line in out.strip().splitlines():
            f = [x.strip() for x in line.split(",")]
            if len(f) < 9:
                continue
            try:
                sm.append(float(f[1]))
                smax.append(float(f[2]))
            except ValueError:
                continue
            for n, v in zip(names, f[5:9]):
                if v.lower() == "active":
                    reasons.add(n)
        return {"sm_mhz": statistics.median(sm) if sm else None,
                "sm_max_mhz": max(smax) if smax else None,
                "samples": len(sm), "reasons": sorted(reasons)}


def aggregate(elapsed: float, units_per_rank: float, ws: int, all_reduce_max=None):
    """Whole-job rate over `ws` independent replicas: the time is the slowest rank's
    (max over ranks), the work the sum over ranks.  `all_reduce_max` maps a local float
    to the max over ranks (None: one rank)."""
    t = all_reduce_max(elapsed) if all_reduce_max and ws > 1 else elapsed
    return ws * units_per_rank / t, t


def workload_bytes(case):
    """Algorithmic bytes of one step: decode reads every attended K/V row once, q,
    block-table entries and context lengths once, writes out once; kv_append reads
    the new rows and writes them into the pool.  Also the unique decode bytes: each
    distinct pool slot counted once however many sequences share it (what has to
    come from HBM at least; equal to the logical bytes when nothing is shared)."""
    import torch
    S, Hq, D = case.q.shape
    Hkv = case.k_pool.shape[1]
    esz = case.q.element_size()
    B = case.k_pool.shape[2]   # tokens per pool block
    lens = case.context_lens.cpu().to(torch.int64)
    tokens = int(lens.sum())
    kv = tokens * Hkv * D * esz * 2
    nblk = int(((lens + B - 1) // B).sum())
    small = 2 * S * Hq * D * esz + nblk * 4 + S * 4
    decode = kv + small
    T = case.k_new.shape[0]
    append = 2 * 2 * T * Hkv * D * esz + T * 8
    # distinct (block, row) slots: per physical block the most rows any sequence uses
    bt = case.block_tables.cpu().to(torch.int64)
    j = torch.arange(bt.shape[1])
    nb = (lens + B - 1) // B
    used = j[None, :] < nb[:, None]
    rows = (lens[:, None] - B * j[None, :]).clamp(0, B)
    per_block = torch.zeros(case.k_pool.shape[0], dtype=torch.int64)
    per_block.scatter_reduce_(0, bt[used], rows[used], reduce="amax")
    unique_tokens = int(per_block.sum())
    unique = unique_tokens * Hkv * D * esz * 2 + small
    return decode, append, tokens, unique


def run_reference(args, ws, rank):
    """fp64 CPU oracle on the host cores: each step is a bounded sample of the batch."""
    if rank != 0:
        return
    import numpy as np
    import oracle
    import synth
    oracle.build()
    case = synth.build_case(args.workload, "cpu")
    decode_bytes, append_bytes, tokens, _ = workload_bytes(case)
    kp, vp = synth.host_bits(case.k_pool), synth.host_bits(case.v_pool)
    q, bt = synth.host_bits(case.q), synth.host_bits(case.block_tables)
    cl = synth.host_bits(case.context_lens)
    slots, kn, vn = (synth.host_bits(case.slot_mapping), synth.host_bits(case.k_new),
                     synth.host_bits(case.v_new))
    oracle.kv_append(slots, kn, vn, kp, vp)
    S = q.shape[0]
    # calibrate one full pass, then size each step's sample so the run stays bounded
    t0 = time.perf_counter()
    oracle.paged_decode(q, kp, vp, bt, cl, case.scale)
    t_full = time.perf_counter() - t0
    budget = 150.0
    n = max(1, min(S, int(S * budget / max(1e-9, (args.steps + args.warmup) * t_full))))
    idx = np.arange(n)
    sub_bytes = decode_bytes * float(cl[idx].astype(np.int64).sum()) / tokens
    for _ in range(args.warmup):
        oracle.paged_decode(q[idx], kp, vp, bt[idx], cl[idx], case.scale)
    t0 = time.perf_counter()
    for _ in range(args.steps):
        oracle.paged_decode(q[idx], kp, vp, bt[idx], cl[idx], case.scale)
    dt = (time.perf_counter() - t0) / args.steps
    value = sub_bytes / dt / 1e9
    cores = os.cpu_count()
    line = {
        "impl": "reference", "metric": METRIC, "value": value, "unit": "GB/s", "n_gpus": ws,
        "steps": args.steps, "warmup": args.warmup, "ms_per_step": dt * 1e3,
        "higher_is_better": True, "scaling": "weak", "vs_baseline": None, "dtype": "f64",
        "data": "synthetic", "tokens_per_s_per_layer": n / dt,
        "config": {"workload": case.wl.name, "num_seqs": S, "sample_seqs": n},
        "cpu_baseline": {"value": value, "unit": "GB/s", "cores": cores, "kind": "oracle",
                         "sample": f"first {n} of {S} sequences per step (all heads), "
                                   f"full pass {t_full:.3f} s"},
        "e2e": {"value": value, "unit": "GB/s", "h2d_bytes_per_step": 0,
                "d2h_bytes_per_step": 0},
    }
    print(json.dumps(line), flush=True)


def cpu_baseline(case, decode_bytes, tokens):
    """The oracle as it stands, on the host cores, over repeated full passes (~5 s)."""
    import numpy as np
    import oracle
    import synth
    oracle.build()
    kp, vp = synth.host_bits(case.k_pool), synth.host_bits(case.v_pool)
    oracle.kv_append(synth.host_bits(case.slot_mapping), synth.host_bits(case.k_new),
                     synth.host_bits(case.v_new), kp, vp)
    q, bt = synth.host_bits(case.q), synth.host_bits(case.block_tables)
    cl = synth.host_bits(case.context_lens)
    reps = 0
    t0 = time.perf_counter()
    while True:
        oracle.paged_decode(q, kp, vp, bt, cl, case.scale)
        reps += 1
        el = time.perf_counter() - t0
        if el > 5.0 or reps >= 200:
            break
    dt = el / reps
    # The same oracle on one thread, over the first sequences of the batch (~2 s).
    n1 = min(4, q.shape[0])
    q1, bt1, cl1 = q[:n1].copy(), bt[:n1].copy(), cl[:n1].copy()
    tok1 = int(cl1.astype(np.int64).sum())
    bytes1 = decode_bytes * tok1 / max(tokens, 1)   # the sample's share of the K/V bytes
    reps1 = 0
    t1 = time.perf_counter()
    while True:
        oracle.paged_decode(q1, kp, vp, bt1, cl1, case.scale, nthreads=1)
        reps1 += 1
        el1 = time.perf_counter() - t1
        if el1 > 2.0 or reps1 >= 200:
            break
    return {"value": decode_bytes / dt / 1e9, "unit": "GB/s", "cores": os.cpu_count(),
            "kind": "oracle",
            "sample": f"whole batch ({q.shape[0]} seqs, {tokens} tokens), {reps} passes in "
                      f"{el:.1f} s; decode only (fp64, std::thread over (seq, kv head))",
            "tokens_per_s_per_layer": q.shape[0] / dt,
            "value_1core": bytes1 / (el1 / reps1) / 1e9,
            "sample_1core": f"first {n1} seqs ({tok1} tokens), {reps1} passes in {el1:.1f} s "
                            f"on one thread"}


def main():
    args = parse()
    ws, rank, local = dist_env()
    if args.impl == "reference":
        run_reference(args, ws, rank)
        return
    if args.gpus > 1 and "WORLD_SIZE" not in os.environ:
        # N replicas, one process per GPU, through torch.distributed.run
        sys.exit(launch_replicas(args.gpus, sys.argv[1:]).returncode)

    import torch
    torch.cuda.set_device(local)
    dev = torch.device("cuda", local)
    ranks = Ranks("nccl", dev)

    import synth
    import paged_kv_cache_58_gb300 as pkv
    from paged_kv_cache_58_gb300 import build as pkv_build
    if rank == 0 or ws == 1:
        pkv_build.build()
    ranks.barrier()

    case = synth.build_case(with_block_size(synth.WORKLOADS[args.workload], args.block_size),
                            dev)
    S, Hq, D = case.q.shape
    B = case.k_pool.shape[2]
    decode_bytes, append_bytes, tokens, unique_bytes = workload_bytes(case)
    max_ctx = case.max_context
    pb = args.partition_blocks or pkv.auto_partition(S, Hq, max_ctx, block_size=B)
    wsz = pkv.decode_workspace_bytes(S, Hq, D, max_ctx, pb, block_size=B)
    workspace = torch.empty(max(wsz, 16), dtype=torch.uint8, device=dev)
    out = torch.empty_like(case.q)
    stream = torch.cuda.current_stream(dev)
    max_parts = math.ceil(math.ceil(max_ctx / B) / pb)
    launches_per_step = 2 + (1 if max_parts > 1 else 0)

    cascade = args.cascade and case.wl.shared_prefix > 0
    fused = not args.separate_append
    if cascade:
        plen = case.wl.shared_prefix
        prefix_blocks = case.block_tables[0, :plen // B].contiguous()
        wsz = pkv.cascade_workspace_bytes(S, Hq, D, plen, max_ctx, block_size=B)
        workspace = torch.empty(max(wsz, 16), dtype=torch.uint8, device=dev)
        launches_per_step = 4
    if fused:
        launches_per_step -= 1   # the append runs inside the (suffix) decode kernel
        # The fused call reads no slot mapping: the table gives each new token's slot.
        append_bytes -= case.slot_mapping.numel() * case.slot_mapping.element_size()

    def append(slots, kn, vn):
        if not fused:
            pkv.kv_append(case.k_pool, case.v_pool, slots, kn, vn, stream=stream)

    def decode(q, bt, cl, kn=None, vn=None):
        if fused and cascade:
            pkv.paged_decode_cascade_append(q, case.k_pool, case.v_pool, kn, vn, prefix_blocks,
                                            plen, bt, cl, case.scale, max_context=max_ctx,
                                            out=out, workspace=workspace, stream=stream)
        elif fused:
            pkv.paged_decode_append(q, case.k_pool, case.v_pool, kn, vn, bt, cl, case.scale,
                                    max_context=max_ctx, out=out, partition_blocks=pb,
                                    workspace=workspace, stream=stream)
        elif cascade:
            pkv.paged_decode_cascade(q, case.k_pool, case.v_pool, prefix_blocks, plen, bt, cl,
                                     case.scale, max_context=max_ctx, out=out,
                                     workspace=workspace, stream=stream)
        else:
            pkv.paged_decode(q, case.k_pool, case.v_pool, bt, cl, case.scale,
                             max_context=max_ctx, out=out, partition_blocks=pb,
                             workspace=workspace, stream=stream)

    def step():
        append(case.slot_mapping, case.k_new, case.v_new)
        decode(case.q, case.block_tables, case.context_lens, case.k_new, case.v_new)

    clocks = ClockSampler(local)
    clocks.start()
    for _ in range(max(3, args.warmup)):
        step()
    torch.cuda.synchronize()
    t0 = time.perf_counter()
    while time.perf_counter() - t0 < args.min_warm_seconds:
        for _ in range(50):
            step()
        torch.cuda.synchronize()
    assert pkv.read_device_status() == 0

    K = args.steps
    step_bytes = decode_bytes + append_bytes
    # K steps back to back for the step time (an event between two steps would hold the
    # next step's launch behind the previous one), then K more with events around each
    # decode call for the kernel's own duration (the roofline).
    rate, total_s = replica_rate(ranks, step, K, step_bytes, EventClock(stream))
    ev = [(torch.cuda.Event(enable_timing=True), torch.cuda.Event(enable_timing=True))
          for _ in range(K)]
    for i in range(K):
        append(case.slot_mapping, case.k_new, case.v_new)
        ev[i][0].record(stream)
        decode(case.q, case.block_tables, case.context_lens, case.k_new, case.v_new)
        ev[i][1].record(stream)
    torch.cuda.synchronize()
    ranks.barrier()
    clk = clocks.stop()
    decode_ms = statistics.mean(a.elapsed_time(b) for a, b in ev)
    assert pkv.read_device_status() == 0
    value = rate / 1e9
    ms_step = total_s * 1e3 / K
    tok_s = ws * S * K / total_s

    # end to end through the public API with host buffers: H2D of the step's inputs
    # from pinned memory, the two calls, D2H of the output, synchronised per step.
    e2e = None
    if not args.no_e2e:
        # The step's inputs staged in one pinned host buffer (256-byte aligned pieces) and
        # moved by one host-to-device copy; the kernels read device views of it.
        names = ("q", "k_new", "v_new", "block_tables", "context_lens")
        if not fused:
            names += ("slot_mapping",)
        srcs = [getattr(case, n).contiguous() for n in names]
        offs, total = [], 0
        for t in srcs:
            total = (total + 255) // 256 * 256
            offs.append(total)
            total += t.numel() * t.element_size()
        host_buf = torch.empty(total, dtype=torch.uint8).pin_memory()
        dev_buf = torch.empty(total, dtype=torch.uint8, device=dev)
        devb = {}
        for n, t, o in zip(names, srcs, offs):
            nbytes = t.numel() * t.element_size()
            host_buf[o:o + nbytes].copy_(t.cpu().view(torch.uint8).reshape(-1))
            devb[n] = dev_buf[o:o + nbytes].view(t.dtype).view(t.shape)
        out_h = torch.empty(out.shape, dtype=out.dtype).pin_memory()
        h2d = total
        d2h = out_h.numel() * out_h.element_size()

        e2e_api = "torch H2D copy + " + ("paged_decode_cascade_append" if cascade and fused
                                         else "kv_append + paged_decode_cascade" if cascade
                                         else "kv_append + paged_decode") + " + torch D2H copy"

        def e2e_step():
            dev_buf.copy_(host_buf, non_blocking=True)
            append(devb.get("slot_mapping"), devb["k_new"], devb["v_new"])
            decode(devb["q"], devb["block_tables"], devb["context_lens"], devb["k_new"],
                   devb["v_new"])
            out_h.copy_(out, non_blocking=True)
            stream.synchronize()

        if fused and not cascade:
            # The C ABI's host-buffer step: one packed pinned input buffer, one copy each way.
            mbs = case.block_tables.shape[1]
            lay = pkv.decode_step_layout(case.k_pool, S, Hq, mbs)
            host_in = torch.empty(lay.bytes, dtype=torch.uint8).pin_memory()
            pkv.pack_decode_step(host_in, lay, case.q.cpu(), case.k_new.cpu(), case.v_new.cpu(),
                                 case.block_tables.cpu(), case.context_lens.cpu())
            staging = torch.empty(pkv.decode_host_staging_bytes(case.k_pool, S, Hq, mbs, max_ctx,
                                                                pb),
                                  dtype=torch.uint8, device=dev)
            h2d = lay.bytes
            e2e_api = ("pkv_paged_decode_append_host through HostDecodeStep (pinned buffers: "
                       "the kernels read the packed inputs from host memory and write the "
                       "output there in place)")

            host_step = pkv.HostDecodeStep(case.k_pool, case.v_pool, host_in, out_h,
                                           case.scale, num_seqs=S, num_q_heads=Hq,
                                           max_blocks_per_seq=mbs, max_context=max_ctx,
                                           staging=staging, partition_blocks=pb,
                                           stream=stream)

            def e2e_step():
                host_step()
                stream.synchronize()

        for _ in range(max(3, args.warmup)):
            e2e_step()
        e2e_rate, el = replica_rate(ranks, e2e_step, K, step_bytes, WallClock())
        e2e = {"value": e2e_rate / 1e9, "unit": "GB/s", "api": e2e_api,
               "h2d_bytes_per_step": h2d, "d2h_bytes_per_step": d2h,
               "ms_per_step": el / K * 1e3, "tokens_per_s_per_layer": ws * S * K / el}

    if rank != 0:
        ranks.close()
        return

    pk = peaks()
    peak, tpeak, peak_kind = pk
    # Roofline on the unique bytes: a shared prefix is read from HBM once per step and
    # from L2 by every other sequence, so the logical rate can exceed HBM bandwidth.  The
    # fused call also moves the new rows (read from the input, stored into the pool).
    call_bytes = unique_bytes + (append_bytes if fused else 0)
    achieved = call_bytes / (decode_ms * 1e-3) / 1e9
    del workspace, out
    # The sub-lines and the oracle timings are single-GPU figures: with N replicas they
    # would repeat the N = 1 line while every GPU is held, so they run at N = 1 only.
    single = ws == 1
    cpu_on = single and not args.no_cpu_baseline
    prefill = None
    if single and not args.no_prefill:
        prefill = bench_prefill(pkv, dev, args.prefill_steps, stream, args.block_size,
                                args.prefill_head_dim, args.prefill_dtype, pk,
                                cpu=cpu_on, e2e=not args.no_e2e)
        if prefill["dtype"] == "f32":
            # fp32 pools run on the CUDA cores: fp32 FMA peak from the unit counts and the
            # maximum SM clock (152 SMs x 128 FMA a clock x 2 flop x 2.07 GHz).
            apeak = FP32_ALU_TFLOPS
            prefill.update({"bound": "alu", "peak": apeak, "unit": "TFLOP/s",
                            "frac": prefill["tflops"] / apeak,
                            "peak_kind": "derived fp32 FMA peak (152 SMs x 128 x 2 x 2.07 GHz)"})
        else:
            prefill.update({"bound": "tensor", "peak": tpeak, "unit": "TFLOP/s",
                            "frac": prefill["tflops"] / tpeak,
                            "peak_kind": f"{peak_kind} bf16_tflops (burst; kernel timed alone)"})
    long_decode = cascade_line = None
    if single and not args.no_long_decode and args.workload != "70b":
        long_decode = bench_decode_line(pkv, dev, "70b", args.sub_steps, stream, pk,
                                        cpu=cpu_on, block_size=args.block_size)
    if single and not args.no_cascade_line and not (args.workload == "shared" and cascade):
        cascade_line = bench_decode_line(pkv, dev, "shared", args.sub_steps, stream, pk,
                                         cascade=True, cpu=cpu_on, block_size=args.block_size)
    dtype = {torch.bfloat16: "bf16", torch.float32: "f32"}[case.q.dtype]
    line = {
        "metric": METRIC, "value": value, "unit": "GB/s", "n_gpus": ws, "steps": K,
        "warmup": args.warmup, "ms_per_step": ms_step, "higher_is_better": True,
        "scaling": "weak", "vs_baseline": None, "dtype": dtype, "data": "synthetic",
        "pct_of_8tbs": 100.0 * value / ws / NOMINAL_HBM_GBS,
        "tokens_per_s_per_layer": tok_s,
        "config": {"workload": case.wl.name, "num_seqs": S, "q_heads": Hq,
                   "kv_heads": case.k_pool.shape[1], "head_dim": D, "block_size": B,
                   "pool_blocks": case.k_pool.shape[0], "mean_context": tokens / S,
                   "max_context": max_ctx, "partition_blocks": pb,
                   "kv_bytes_per_step": decode_bytes, "append_bytes_per_step": append_bytes,
                   "unique_kv_bytes_per_step": unique_bytes,
                   "l2": ("inputs larger than L2 (K/V read per step > 129 MB L2)"
                          if decode_bytes > 2 * 129e6 else
                          "K/V per step smaller than L2: warm-cache figure"),
                   "parallelism": f"replicas x{ws}", "cascade": cascade,
                   "step": (("paged_decode_cascade_append" if cascade else
                             "paged_decode_append") + " (append fused into the decode)" if fused
                            else "kv_append + " + ("paged_decode_cascade" if cascade
                                                   else "paged_decode"))},
        "roofline": {"bound": "hbm",
                     "kernel": ("paged_decode_cascade (prefix pass + suffix split-KV + combine"
                                + (", append fused)" if fused else ")")
                                if cascade else
                                "paged_decode_append (decode_tc split-KV with the append "
                                "+ combine)" if fused else
                                "paged_decode (decode_tc split-KV + combine)"),
                     "achieved": achieved, "peak": peak, "unit": "GB/s",
                     "bytes_per_launch": call_bytes,
                     "logical_gbs": (decode_bytes + (append_bytes if fused else 0)) /
                                    (decode_ms * 1e-3) / 1e9,
                     "frac": achieved / peak, "peak_kind": f"{peak_kind} hbm_gbs",
                     "frac_of_8tbs": achieved / NOMINAL_HBM_GBS,
                     "decode_ms": decode_ms, "traffic": None},
        "e2e": e2e,
        "prefill": prefill,
        "long_decode": long_decode,
        "shared_prefix_cascade": cascade_line,
        "prefix_cache": None if (args.no_prefix_cache or not single) else bench_prefix_cache(pkv),
        "gpu_launches": launches_per_step * K,
        "clocks": clk,
    }
    if cpu_on:
        line["cpu_baseline"] = cpu_baseline(case, decode_bytes, tokens)
    print(json.dumps(line), flush=True)
    ranks.close()


if __name__ == "__main__":
    main()
