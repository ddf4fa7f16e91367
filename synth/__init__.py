"""Seeded synthetic inputs for paged-KV attention (shared by tests, bench, oracle).

This module only draws inputs: random block placements, context lengths and
N(0, 1) query/key/value values, laid out as the pool contract requires.  It
holds none of the attention arithmetic; both the CUDA path and the fp64 oracle
consume what it returns.

Pool contract: ``k_pool``/``v_pool`` are ``[num_blocks, Hkv, B, D]``; token j
of a sequence lives in block ``block_tables[s, j // B]`` at offset ``j % B``;
unused table entries are -1.  Every pool slot that no sequence owns -- whole
unreferenced blocks and the tail of each sequence's last block -- holds NaN,
so a kernel that reads outside a sequence poisons its output.

Decode reading (applied to every decode workload): a drawn context length L
counts the token being decoded.  Tokens 0..L-2 are pre-filled in the pool; the
K/V of token L-1 arrive as ``k_new``/``v_new`` with ``slot_mapping`` and must
be written by kv_append before attention.  Prefill reading: a request with c
cached and n new tokens has tokens 0..c-1 pre-filled and the n new rows in
``k_new``/``v_new``/``slot_mapping``.

Values are drawn with ``torch.Generator`` on the device the case is built on;
the same bits reach the oracle through host copies.
"""
from __future__ import annotations

import math
from dataclasses import dataclass, field

import numpy as np
import torch

BLOCK = 16


@dataclass
class Workload:
    """Shape recipe of one workload (sizes follow the published configs)."""
    name: str
    kind: str                 # "decode" or "prefill"
    num_seqs: int
    num_q_heads: int
    num_kv_heads: int
    head_dim: int
    dtype: torch.dtype
    num_blocks: int
    seed: int
    ctx_fixed: tuple = ()     # explicit context lengths (decode) / cached lens (prefill)
    ctx_lo: int = 0           # uniform integer range [lo, hi] otherwise
    ctx_hi: int = 0
    shared_prefix: int = 0    # tokens of a prefix shared by all sequences (multiple of B)
    new_tokens: int = 0       # prefill: new tokens per request
    block_size: int = BLOCK   # tokens per pool block (16, or 32)


WORKLOADS = {
    # 4 sequences, contexts {17, 33, 5, 64}, 4 q = 4 kv heads, D 64, fp32, 64-block pool.
    "tiny": Workload("tiny_decode_s4_d64_f32", "decode", 4, 4, 4, 64, torch.float32, 64, 1,
                     ctx_fixed=(17, 33, 5, 64)),
    # Llama-3-8B-shaped decode layer: 64 seqs, 32/8 heads, D 128, ctx U[512, 4096].
    "8b": Workload("llama3_8b_decode_s64_ctx512-4096", "decode", 64, 32, 8, 128, torch.bfloat16,
                   32768, 2, ctx_lo=512, ctx_hi=4096),
    # Llama-3.1-70B-shaped long decode: 16 seqs, 64/8 heads, ctx U[16384, 131072].
    "70b": Workload("llama31_70b_decode_s16_ctx16k-128k", "decode", 16, 64, 8, 128,
                    torch.bfloat16, 163840, 3, ctx_lo=16384, ctx_hi=131072),
    # Shared 4096-token prefix (256 blocks, refcount 256) + private suffix U[64, 1024].
    "shared": Workload("shared_prefix4096_decode_s256", "decode", 256, 32, 8, 128,
                       torch.bfloat16, 32768, 4, ctx_lo=64, ctx_hi=1024, shared_prefix=4096),
    # Prefix-cached chunked prefill: 16 requests, cached U[1024, 8192], 512 new tokens.
    "prefill": Workload("prefix_cached_prefill_r16_c1k-8k_n512", "prefill", 16, 32, 8, 128,
                        torch.bfloat16, 32768, 5, ctx_lo=1024, ctx_hi=8192, new_tokens=512),
}


@dataclass
class Case:
    """Device tensors of one drawn workload plus the host-side recipe."""
    wl: Workload
    q: torch.Tensor              # decode [S, Hq, D]; prefill [N, Hq, D]
    k_pool: torch.Tensor         # [NB, Hkv, B, D], pre-append contents
    v_pool: torch.Tensor
    block_tables: torch.Tensor   # int32 [S, max_blocks], -1 padded
    context_lens: torch.Tensor   # int32 [S] (decode: L incl. new token; prefill: c + n)
    slot_mapping: torch.Tensor   # int64 [T] slots of the rows in k_new / v_new
    k_new: torch.Tensor          # [T, Hkv, D]
    v_new: torch.Tensor
    scale: float
    cached_lens: torch.Tensor | None = None   # prefill only, int32 [R]
    new_lens: torch.Tensor | None = None      # prefill only, int32 [R]
    q_offsets: torch.Tensor | None = None     # prefill only, int32 [R + 1]
    extra: dict = field(default_factory=dict)

    @property
    def max_context(self) -> int:
        return int(self.context_lens.max().item())


def _gen(seed: int, device) -> torch.Generator:
    g = torch.Generator(device=device)
    g.manual_seed(seed)
    return g


def _randn(shape, g, device, dtype) -> torch.Tensor:
    return torch.randn(shape, generator=g, device=device, dtype=torch.float32).to(dtype)


def _fill_blocks(pool: torch.Tensor, blocks: torch.Tensor, g, chunk: int = 4096) -> None:
    """pool[blocks] = N(0,1), drawn in chunks to bound the fp32 staging memory."""
    for i in range(0, blocks.numel(), chunk):
        b = blocks[i:i + chunk]
        pool[b] = _randn((b.numel(),) + tuple(pool.shape[1:]), g, pool.device, pool.dtype)


def draw_lengths(wl: Workload, g_cpu: torch.Generator) -> list[int]:
    if wl.ctx_fixed:
        return [int(x) for x in wl.ctx_fixed]
    return torch.randint(wl.ctx_lo, wl.ctx_hi + 1, (wl.num_seqs,), generator=g_cpu).tolist()


def build_case(wl: Workload | str, device="cuda", *, lengths=None, seed=None,
               num_blocks=None) -> Case:
    """Draw one workload on `device`.

    `lengths` overrides the drawn context lengths (decode: L; prefill: cached c);
    `seed`/`num_blocks` override the recipe's (used for small parity cases).
    """
    if isinstance(wl, str):
        wl = WORKLOADS[wl]
    seed = wl.seed if seed is None else seed
    nb = wl.num_blocks if num_blocks is None else num_blocks
    g_cpu = _gen(seed, "cpu")
    g_dev = _gen(seed + 1000, device)
    lens = list(lengths) if lengths is not None else draw_lengths(wl, g_cpu)
    S, Hq, Hkv, D = len(lens), wl.num_q_heads, wl.num_kv_heads, wl.head_dim
    B = wl.block_size

    if wl.kind == "decode":
        if wl.shared_prefix:
            totals = [wl.shared_prefix + x for x in lens]   # prefix + private suffix
        else:
            totals = lens
        prefill_valid = [L - 1 for L in totals]  # last token comes through kv_append
    else:
        totals = [c + wl.new_tokens for c in lens]
        prefill_valid = lens

    nblk = [math.ceil(L / B) for L in totals]
    shared_blocks = wl.shared_prefix // B
    private_needed = sum(n - shared_blocks for n in nblk)
    need = shared_blocks + private_needed
    if need > nb:
        raise ValueError(f"pool of {nb} blocks cannot hold {need} blocks")
    perm = torch.randperm(nb, generator=g_cpu)[:need]
    max_blocks = max(nblk)
    bt = torch.full((S, max_blocks), -1, dtype=torch.int32)
    shared_ids = perm[:shared_blocks]
    pos = shared_blocks
    for s in range(S):
        bt[s, :shared_blocks] = shared_ids.to(torch.int32)
        k = nblk[s] - shared_blocks
        bt[s, shared_blocks:nblk[s]] = perm[pos:pos + k].to(torch.int32)
        pos += k

    dtype = wl.dtype
    k_pool = torch.full((nb, Hkv, B, D), float("nan"), dtype=dtype, device=device)
    v_pool = torch.full((nb, Hkv, B, D), float("nan"), dtype=dtype, device=device)
    used = perm.to(device)
    _fill_blocks(k_pool, used, g_dev)
    _fill_blocks(v_pool, used, g_dev)
    # Slots past the pre-filled prefix of each sequence hold NaN until written.
    tail_blk, tail_off = [], []
    for s in range(S):
        j = torch.arange(prefill_valid[s], nblk[s] * B)
        tail_blk.append(bt[s, j // B].long())
        tail_off.append(j % B)
    tail_blk = torch.cat(tail_blk).to(device)
    tail_off = torch.cat(tail_off).to(device)
    k_pool[tail_blk, :, tail_off, :] = float("nan")
    v_pool[tail_blk, :, tail_off, :] = float("nan")

    if wl.kind == "decode":
        T = S
        slots = [int(bt[s, (totals[s] - 1) // B]) * B + (totals[s] - 1) % B for s in range(S)]
        q = _randn((S, Hq, D), g_dev, device, dtype)
    else:
        n = wl.new_tokens
        T = S * n
        slots = []
        for s in range(S):
            for i in range(n):
                p = lens[s] + i
                slots.append(int(bt[s, p // B]) * B + p % B)
        q = _randn((T, Hq, D), g_dev, device, dtype)
    k_new = _randn((T, Hkv, D), g_dev, device, dtype)
    v_new = _randn((T, Hkv, D), g_dev, device, dtype)

    case = Case(
        wl=wl, q=q, k_pool=k_pool, v_pool=v_pool,
        block_tables=bt.to(device), context_lens=torch.tensor(totals, dtype=torch.int32,
                                                              device=device),
        slot_mapping=torch.tensor(slots, dtype=torch.int64, device=device),
        k_new=k_new, v_new=v_new, scale=1.0 / math.sqrt(D))
    if wl.kind == "prefill":
        case.cached_lens = torch.tensor(lens, dtype=torch.int32, device=device)
        case.new_lens = torch.full((S,), wl.new_tokens, dtype=torch.int32, device=device)
        case.q_offsets = torch.arange(0, (S + 1) * wl.new_tokens, wl.new_tokens,
                                      dtype=torch.int32, device=device)
    case.extra["num_used_blocks"] = need
    return case


def host_bits(t: torch.Tensor) -> np.ndarray:
    """Host numpy copy with exact bits: fp32 -> float32, bf16 -> uint16."""
    t = t.detach().contiguous().cpu()
    if t.dtype == torch.bfloat16:
        return t.view(torch.int16).numpy().view(np.uint16).copy()
    if t.dtype == torch.float32:
        return t.numpy().copy()
    return t.numpy().copy()


def sample_rows(num_rows: int, num_heads: int, count: int, seed: int) -> np.ndarray:
    """Boolean [rows, heads] mask with `count` seeded (row, head) picks, first/last rows kept."""
    rng = np.random.default_rng(seed)
    want = np.zeros((num_rows, num_heads), dtype=bool)
    idx = rng.choice(num_rows * num_heads, size=min(count, num_rows * num_heads), replace=False)
    want.flat[idx] = True
    want[0, :] = True
    want[-1, :] = True
    return want
