"""The prefix-reuse serving flow on the GPU, through the radix tree and through the
chained block-hash cache, against the fp64 oracle.

A prompt A is prefilled and registered in the index.  Two later prompts share a prefix
with it: B its first 1300 tokens (not a block boundary), C its first 37.  For each, the
index returns the blocks holding the matched positions; the sequence is admitted with
those blocks shared (pkv_alloc_add_seq_shared); its first append copies a partly filled
shared block first (the copy-on-write pair pkv_alloc_append returns, run through
pkv_copy_blocks); kv_append writes the unmatched suffix; one batched pkv_paged_prefill
computes only the new rows of B and C over their reused prefixes; then one decode step.
Only the unseen suffix is computed while the cached prefix is reused (aitalk.it
"RadixAttention: A Tree That Does Not Forget", "Two Layers, Not Two Rivals"; aifetchly
guide, "Prefill Bypass"); sharing is a pointer change and mutation after it copies
(Triptych "Paged Attention for Efficient Memory Management").

Checks: the pools equal, bit for bit, an oracle replay of the same copies and appends;
the prefill and decode outputs match the oracle run on the shared tables, and the
oracle on the shared tables equals the oracle on a private, contiguous copy of each
prompt's K/V (so the reuse changed nothing); A's own K/V are unchanged afterwards.
"""
import numpy as np
import pytest
import torch

import synth
from tests.helpers import check_attention, pool_equal

pytestmark = pytest.mark.gpu

HKV, HQ, D, B = 8, 32, 128, 16
NB = 1024
LA, SHARE_B, LB, SHARE_C, LC = 2000, 1300, 1800, 37, 420


@pytest.fixture(scope="module")
def pkv():
    if not torch.cuda.is_available():
        pytest.skip("no CUDA device")
    import paged_kv_cache_58_gb300 as m
    from paged_kv_cache_58_gb300 import build
    build.build()
    return m


class Replay:
    """The device pools and a host copy that the oracle updates with the same ops."""

    def __init__(self, pkv, oracle):
        self.pkv, self.oracle = pkv, oracle
        self.kp = torch.full((NB, HKV, B, D), float("nan"), dtype=torch.bfloat16, device="cuda")
        self.vp = torch.full_like(self.kp, float("nan"))
        self.hk, self.hv = synth.host_bits(self.kp), synth.host_bits(self.vp)

    def append(self, slots, k, v):
        st = torch.tensor(slots, dtype=torch.int64)
        self.pkv.kv_append(self.kp, self.vp, st.cuda(), k, v)
        self.oracle.kv_append(st.numpy(), synth.host_bits(k), synth.host_bits(v), self.hk,
                              self.hv)

    def copy(self, pair):
        pr = torch.tensor([pair], dtype=torch.int32)
        self.pkv.copy_blocks(self.kp, self.vp, pr.cuda())
        self.oracle.copy_blocks(pr.numpy(), self.hk, self.hv)

    def check_pools(self):
        torch.cuda.synchronize()
        assert self.pkv.read_device_status() == 0
        assert pool_equal(self.kp, self.hk) and pool_equal(self.vp, self.hv)


def contiguous_pool(rows_k, rows_v):
    """Host bf16-bit pools holding each prompt's K/V in private consecutive blocks, and
    their table: the layout with no sharing at all."""
    nblk = [-(-r.shape[0] // B) for r in rows_k]
    kp = np.full((sum(nblk), HKV, B, D), 0x7fc0, np.uint16)   # NaN bits
    vp = kp.copy()
    bt = np.full((len(rows_k), max(nblk)), -1, np.int32)
    base = 0
    for s, (rk, rv) in enumerate(zip(rows_k, rows_v)):
        for j in range(rk.shape[0]):
            kp[base + j // B, :, j % B] = rk[j]
            vp[base + j // B, :, j % B] = rv[j]
        bt[s, :nblk[s]] = np.arange(base, base + nblk[s])
        base += nblk[s]
    return kp, vp, bt


@pytest.mark.parametrize("index", ["radix", "block_hash"])
def test_prefix_reuse_flow_matches_oracle(pkv, oracle_mod, index):
    g = torch.Generator(device="cuda").manual_seed(58 if index == "radix" else 59)
    rng = np.random.default_rng(7)
    tok_a = rng.integers(0, 32000, LA).tolist()
    tok_b = tok_a[:SHARE_B] + rng.integers(0, 32000, LB - SHARE_B).tolist()
    tok_c = tok_a[:SHARE_C] + rng.integers(0, 32000, LC - SHARE_C).tolist()
    tok_b[SHARE_B] = (tok_a[SHARE_B] + 1) % 32000   # the prompts diverge exactly there
    tok_c[SHARE_C] = (tok_a[SHARE_C] + 1) % 32000

    def rows(n):
        return (torch.randn((n, HKV, D), generator=g, device="cuda").to(torch.bfloat16),
                torch.randn((n, HKV, D), generator=g, device="cuda").to(torch.bfloat16))

    # K/V of a position depend on the tokens up to it, so a prompt that shares A's first
    # p tokens has A's rows at positions < p and its own after.
    ka, va = rows(LA)
    kb_own, vb_own = rows(LB - SHARE_B)
    kc_own, vc_own = rows(LC - SHARE_C)
    kb, vb = torch.cat([ka[:SHARE_B], kb_own]), torch.cat([va[:SHARE_B], vb_own])
    kc, vc = torch.cat([ka[:SHARE_C], kc_own]), torch.cat([va[:SHARE_C], vc_own])

    rp = Replay(pkv, oracle_mod)
    alloc = pkv.BlockAllocator(NB, B, seed=11)
    cache = pkv.RadixTree(alloc) if index == "radix" else pkv.PrefixCache(alloc)

    # Prompt A: nothing cached yet; admitted, written, registered in the index.
    alloc.add_seq(0, 0)
    slots, cow = alloc.append(0, LA)
    assert cow is None
    rp.append(slots, ka, va)
    cache.insert(0, tok_a)
    rp.check_pools()

    # B and C: match, admit with the matched blocks shared, copy-on-write, append.
    matched = {}
    for sid, toks, kx, vx in ((1, tok_b, kb, vb), (2, tok_c, kc, vc)):
        if index == "radix":
            m, blocks = cache.match(toks)
        else:
            blocks = cache.match(toks)
            m = len(blocks) * B
        share = SHARE_B if sid == 1 else SHARE_C
        assert m == (share if index == "radix" else share // B * B)
        alloc.add_seq_shared(sid, blocks, m)
        for j, blk in enumerate(blocks):
            assert alloc.refcount(blk) >= 2   # A (and the index) hold it too
        slots, cow = alloc.append(sid, len(toks) - m)
        # a partly filled shared last block is copied before the first write into it
        assert (cow is not None) == (m % B != 0)
        if cow is not None:
            assert cow[0] == blocks[-1]
            rp.copy(cow)
        rp.append(slots, kx[m:], vx[m:])
        matched[sid] = m
    rp.check_pools()

    # One batched prefill of the new rows of B and C over their reused prefixes.
    cached = [matched[1], matched[2]]
    new = [LB - matched[1], LC - matched[2]]
    q = torch.randn((sum(new), HQ, D), generator=g, device="cuda").to(torch.bfloat16)
    qo = torch.tensor([0, new[0], new[0] + new[1]], dtype=torch.int32)
    mbs = -(-(LB + 1) // B)
    bt = alloc.block_table([1, 2], mbs)
    scale = D ** -0.5
    out = pkv.paged_prefill(q, rp.kp, rp.vp, bt.cuda(), torch.tensor(cached, dtype=torch.int32,
                                                                       device="cuda"),
                            torch.tensor(new, dtype=torch.int32, device="cuda"), qo.cuda(),
                            scale, max_new=max(new))
    torch.cuda.synchronize()
    assert pkv.read_device_status() == 0
    qh = synth.host_bits(q)
    ref = oracle_mod.paged_prefill(qh, rp.hk, rp.hv, bt.numpy(), np.array(cached, np.int32),
                                   np.array(new, np.int32), qo.numpy(), scale)
    # the same prompts with private, contiguous K/V: identical fp64 result
    ck, cv, cbt = contiguous_pool([synth.host_bits(kb), synth.host_bits(kc)],
                                  [synth.host_bits(vb), synth.host_bits(vc)])
    ref_private = oracle_mod.paged_prefill(qh, ck, cv, cbt, np.array(cached, np.int32),
                                           np.array(new, np.int32), qo.numpy(), scale)
    np.testing.assert_array_equal(ref, ref_private)
    check_attention(out, ref, single_p=True)

    # One decode step of B and C: append one token each (their last blocks are private).
    dslots = []
    for sid in (1, 2):
        s, cow = alloc.append(sid, 1)
        assert cow is None
        dslots += s
    kd, vd = rows(2)
    rp.append(dslots, kd, vd)
    lens = torch.tensor([LB + 1, LC + 1], dtype=torch.int32)
    bt = alloc.block_table([1, 2], mbs)
    qd = torch.randn((2, HQ, D), generator=g, device="cuda").to(torch.bfloat16)
    outd = pkv.paged_decode(qd, rp.kp, rp.vp, bt.cuda(), lens.cuda(), scale,
                            max_context=LB + 1)
    rp.check_pools()
    refd = oracle_mod.paged_decode(synth.host_bits(qd), rp.hk, rp.hv, bt.numpy(), lens.numpy(),
                                   scale)
    check_attention(outd, refd)

    # A's own K/V are untouched by B's and C's writes.
    bta = alloc.block_table([0], -(-LA // B)).numpy()[0]
    for kvh in (0, HKV - 1):
        K, V = oracle_mod.gather(rp.hk, rp.hv, bta, LA, kvh)
        np.testing.assert_array_equal(K, ka[:, kvh].double().cpu().numpy())
        np.testing.assert_array_equal(V, va[:, kvh].double().cpu().numpy())
    cache.close()
    alloc.close()
